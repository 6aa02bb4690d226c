// The correction / bonus sampling, touching only the one row (or row pair)
// per request that the accept/reject walk selected.
//
// "Speculative Decoding and EAGLE-3" lesson, "Invariant: Leviathan rejection
// sampling" and "Build it" step 2: after a rejection at position j the token
// comes from the residual r_t = (q_j(t) - p_j(t))_+ normalised by its sum
// (from q_j itself if that sum is 0); after a full acceptance it comes from
// q_{N+1}.
//
// The draw is a grouped inverse CDF with one uniform per level: the
// vocabulary is split into level-1 blocks of 8192 consecutive tokens, a block
// into 32 blocks of 256, those into 16 blocks of 16, and those into tokens;
// at each level the sub-block is the smallest index whose running mass
// exceeds u_level times the level's total (the last one with mass if
// rounding leaves none).  The law is exactly r / sum(r), and every decision
// compares a uniform against at most a few dozen float32 edges.
//
// Grid: one CTA per request and group of blocks_per_cta() level-1 blocks
// (one block per CTA when the batch is small enough that the grid would
// leave SMs idle), request-major, launched with programmatic dependent launch: it becomes
// resident once every row-statistics CTA has started, while that grid
// drains, and never waits for the grid as a whole.  The walk polls the tags
// of its own request's partials instead, so the requests whose rows were
// reduced first are sampled while later rows still stream.  Every CTA runs the request's
// accept/reject walk itself from the row-statistics partials (one L2 round
// trip; CTA 0 of the request writes the walk's outputs).  For a sampled
// request each CTA then stages its blocks' row pair in shared memory
// (cp.async, all of it in flight at once), evaluates r over each block
// (thread t takes tokens [32t, 32t + 32): two level-3 masses per thread, a
// level-2 mass per eight threads, the level-1 mass per CTA) and picks the
// block's candidate token at levels 2-4 with u_2..u_4, as if level 1 had
// chosen this block.  It stores (level-1 mass, candidate) and counts itself
// in the request's arrival word with one atomic add; the CTA that arrives
// last picks level 1 over the blocks' masses with u_1, writes the chosen
// block's candidate and clears the word for the next call.  No CTA waits
// for another.  If the residual has no mass anywhere, that last CTA redoes
// every block with q alone.  A CTA whose wait for the row statistics ran
// out evaluates nothing but still counts in, marking the word; the last CTA
// then fails the whole request (SV_ERRBIT_WAIT), so a request is either
// sampled from every block or failed.  A CTA whose walk found the request's
// inputs bad (a token out of range, a logit that is NaN or +inf) evaluates
// nothing either and counts in unmarked: the walk has already failed the
// request, and every CTA of it counts in, so the word is clear after every
// call.
//
// r_t = max(q_t - p_t, 0) with q_t = 2^(z_t k - c_q) / s_q and likewise p_t,
// evaluated two tokens at a time with the paired float instructions.  Its
// rounding (a few float32 ulps of q_t per token) moves the level edges by
// ~1e-7 of the level mass, well inside the 1e-5 near-threshold window.

#include <climits>
#include <cuda_bf16.h>

#include "sv_device.cuh"
#include "sv_pick.cuh"
#include "sv_walk.cuh"

namespace sv {
namespace {

// Level-1 blocks one CTA takes: their row pair is staged in shared memory
// (64 KB for two bf16 blocks or one fp32 block), all of it requested at
// once.  Build-time override: -DSV_SAMPLE_BF16_BLOCKS=1 (one bf16 block per
// CTA, twice the CTAs per request, 32 KB each).
#ifndef SV_SAMPLE_BF16_BLOCKS
#define SV_SAMPLE_BF16_BLOCKS 2
#endif
template <typename T>
constexpr int blocks_per_cta() {
  return sizeof(T) == 2 ? SV_SAMPLE_BF16_BLOCKS : 1;
}
template <typename T, int kB>
constexpr int stage_bytes() {
  return 2 * kB * kLevel1 * static_cast<int>(sizeof(T));
}
// A batch whose sampler grid at blocks_per_cta() blocks per CTA would leave
// most SMs idle takes one block per CTA instead (twice the CTAs, half the
// staging and arithmetic each): when the one-block grid has at most
// SV_SAMPLE_SMALL_PER_SM CTAs per SM (mixture-bf16, B 16 at V 163840: 23-25
// against 27.2 us per call; batch64-bf16 keeps two blocks per CTA).
// Build-time override -DSV_SAMPLE_SMALL_PER_SM=<n> (0: never).
#ifndef SV_SAMPLE_SMALL_PER_SM
#define SV_SAMPLE_SMALL_PER_SM 3
#endif

// Arrival counting of a request's sampler CTAs: each adds 1 to the
// request's word (plus kLateUnit when its wait for the row statistics ran
// out) with one atomic, and the CTA whose arrival brings the count to the
// request's CTA total is the last; it clears the word for the next call.
// Every CTA of a sampled request counts in exactly once (a CTA that gave up
// waiting counts in as late, one whose walk failed the request as failed),
// so the last one always does, and a call never meets a count left by an
// earlier one.  Returns the word after this CTA's
// arrival: the count in the low half, the late arrivals in the high half.
constexpr unsigned long long kLateUnit = 1ull << 32;
__device__ __forceinline__ unsigned long long count_in(unsigned long long* word, bool late) {
  const unsigned long long inc = late ? kLateUnit + 1ull : 1ull;
  return atomicAdd(word, inc) + inc;
}

// r for the tokens of one 16-byte vector of each row; rv[e] gets token e.
template <typename T>
__device__ __forceinline__ void resid_vec(const uint4& zv, const uint4& yv, const Job& job, bool has_p,
                                          float (&rv)[Elem<T>::kVec]) {
  using E = Elem<T>;
  const uint64_t k2 = f2pack(job.k, job.k);
  const uint64_t nq2 = f2pack(-job.cq, -job.cq), iq2 = f2pack(job.inv_sq, job.inv_sq);
  const uint64_t np2 = f2pack(-job.cp, -job.cp), ip2 = f2pack(job.inv_sp, job.inv_sp);
#pragma unroll
  for (int e = 0; e < E::kPairs; ++e) {
    float a0, a1;
    f2unpack(f2fma(E::pair(zv, e), k2, nq2), a0, a1);
    float q0, q1;
    f2unpack(f2mul(f2pack(ex2(a0), ex2(a1)), iq2), q0, q1);
    if (has_p) {
      float b0, b1;
      f2unpack(f2fma(E::pair(yv, e), k2, np2), b0, b1);
      float p0, p1;
      f2unpack(f2mul(f2pack(ex2(b0), ex2(b1)), ip2), p0, p1);
      q0 = fmaxf(q0 - p0, 0.f);
      q1 = fmaxf(q1 - p1, 0.f);
    }
    rv[2 * e] = q0;
    rv[2 * e + 1] = q1;
  }
}

// Scalar form (rows that are not 16-byte aligned, and level 4): bit for bit
// the value resid_vec gives the token.
__device__ __forceinline__ float resid1(float zt, float yt, const Job& job, bool has_p) {
  const float q = ex2(fmaf(zt, job.k, -job.cq)) * job.inv_sq;
  if (!has_p) return q;
  return fmaxf(q - ex2(fmaf(yt, job.k, -job.cp)) * job.inv_sp, 0.f);
}

// The two level-3 masses of one thread's 32 tokens [t0, t0 + 32) (0 past
// cend), without keeping the individual r values.
template <typename T, bool kVecPath>
__device__ __forceinline__ void resid_halves(const T* z, const T* y, int t0, int cend, const Job& job,
                                             bool has_p, float& h0, float& h1) {
  using E = Elem<T>;
  h0 = 0.f;
  h1 = 0.f;
  if (kVecPath) {
    constexpr int kVec = E::kVec;
    constexpr int kVecs = kSegTok / kVec;
    const uint4 pad = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
    uint4 zv[kVecs], yv[kVecs];
#pragma unroll
    for (int i = 0; i < kVecs; ++i) {
      const int e0 = t0 + i * kVec;
      const bool in = e0 < cend;
      zv[i] = in ? __ldg(reinterpret_cast<const uint4*>(z + e0)) : pad;
      yv[i] = (in && has_p) ? __ldg(reinterpret_cast<const uint4*>(y + e0)) : pad;
    }
#pragma unroll
    for (int i = 0; i < kVecs; ++i) {
      float rv[kVec];
      resid_vec<T>(zv[i], yv[i], job, has_p, rv);
      float part = 0.f;
#pragma unroll
      for (int e = 0; e < kVec; ++e) part += rv[e];
      if (i < kVecs / 2)
        h0 += part;
      else
        h1 += part;
    }
  } else {
    for (int i = 0; i < kSegTok; ++i) {
      const int t = t0 + i;
      const float r = t < cend ? resid1(E::load1(z + t), has_p ? E::load1(y + t) : 0.f, job, has_p) : 0.f;
      if (i < kLevel3)
        h0 += r;
      else
        h1 += r;
    }
  }
}

// One element of a staged row (shared memory), as float.
__device__ __forceinline__ float staged1(const float* p) { return *p; }
__device__ __forceinline__ float staged1(const __nv_bfloat16* p) {
  return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(p)) << 16);
}

// Stage this thread's tokens [32t, 32t + 32) of the level-1 block starting at
// cbeg into sz / sy; vectors at or past cend get -inf.
template <typename T>
__device__ __forceinline__ void stage_block(const T* z, const T* y, int cbeg, int cend, bool has_p,
                                            T* sz, T* sy) {
  using E = Elem<T>;
  constexpr int kVec = E::kVec;
  const uint4 pad = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
#pragma unroll
  for (int i = 0; i < kSegTok / kVec; ++i) {
    const int e = threadIdx.x * kSegTok + i * kVec;
    const int at = (i * kST + threadIdx.x) * kVec;
    if (cbeg + e < cend) {
      cp_async16(sz + at, z + cbeg + e);
      if (has_p) cp_async16(sy + at, y + cbeg + e);
    } else {
      *reinterpret_cast<uint4*>(sz + at) = pad;
      if (has_p) *reinterpret_cast<uint4*>(sy + at) = pad;
    }
  }
}

// The two level-3 masses of this thread's 32 staged tokens.
template <typename T>
__device__ __forceinline__ void staged_halves(const T* sz, const T* sy, const Job& job, bool has_p,
                                              float& h0, float& h1) {
  using E = Elem<T>;
  constexpr int kVec = E::kVec;
  constexpr int kVecs = kSegTok / kVec;
  h0 = 0.f;
  h1 = 0.f;
#pragma unroll
  for (int i = 0; i < kVecs; ++i) {
    const int e = (i * kST + threadIdx.x) * kVec;
    const uint4 zv = *reinterpret_cast<const uint4*>(sz + e);
    const uint4 yv = has_p ? *reinterpret_cast<const uint4*>(sy + e) : zv;
    float rv[kVec];
    resid_vec<T>(zv, yv, job, has_p, rv);
    float part = 0.f;
#pragma unroll
    for (int q = 0; q < kVec; ++q) part += rv[q];
    if (i < kVecs / 2)
      h0 += part;
    else
      h1 += part;
  }
}

// Masses and candidate of one level-1 block read straight from global memory
// (rows that are not 16-byte aligned, and the q-only redo).
template <typename T, bool kVecPath>
__device__ int block_candidate_global(const T* z, const T* y, int cbeg, int V, const Job& job,
                                      bool has_p, BlockScratch& sc, float* mass) {
  using E = Elem<T>;
  const int cend = min(V, cbeg + kLevel1);
  float h0, h1;
  resid_halves<T, kVecPath>(z, y, cbeg + threadIdx.x * kSegTok, cend, job, has_p, h0, h1);
  return block_pick(
      h0, h1, cbeg, cend, job,
      [&](int t) { return resid1(E::load1(z + t), has_p ? E::load1(y + t) : 0.f, job, has_p); }, sc,
      mass);
}

// Resident CTAs per SM the sampler is built for (its registers per thread
// follow); build-time override -DSV_SAMPLE_MINB=<n>.
#ifndef SV_SAMPLE_MINB
#define SV_SAMPLE_MINB 3
#endif

template <typename T, bool kVecPath, int kB>
__global__ void __launch_bounds__(kST, SV_SAMPLE_MINB) sample_kernel(Problem p, Workspace w) {
  extern __shared__ __align__(16) unsigned char s_rows[];  // staged rows (vector path)
  __shared__ BlockScratch scs[kB];
  BlockScratch& sc = scs[0];
  __shared__ Job s_job;
  __shared__ int s_last;
  const int S3 = w.S3;
  const int G = (S3 + kB - 1) / kB;  // CTAs per request
  const int b = blockIdx.x / G;
  const int g = blockIdx.x - b * G;
  walk_request<T>(p, w, b, g == 0, &s_job, g == p.debug_late_cta);
  __syncthreads();
  const Job job = s_job;
  if (job.kind == kJobNone) return;  // nothing to sample for this request
  const bool late = job.kind == kJobLate;
  // the walk failed the request and wrote its outputs; the CTA only counts in
  const bool failed = job.kind == kJobFailed;
  const int N = p.N, V = p.V;
  const T* z = static_cast<const T*>(p.target) + (static_cast<size_t>(b) * (N + 1) + job.row) * V;
  const T* y = job.kind == kJobResidual
                   ? static_cast<const T*>(p.draft) + (static_cast<size_t>(b) * N + job.row) * V
                   : z;
  const bool has_p = job.kind == kJobResidual;
  float* masses = w.chunk_sums + static_cast<size_t>(b) * S3;
  int* cands = w.blk_tok + static_cast<size_t>(b) * S3;
  const int c0 = g * kB;
  const int nb = min(kB, S3 - c0);

  if (late || failed) {
    // no blocks: the CTA only counts in (below)
  } else if (kVecPath) {
    T* sz = reinterpret_cast<T*>(s_rows);
    T* sy = sz + kB * kLevel1;
    // one group of copies per block, so block i is reduced while the
    // blocks after it are still arriving
#pragma unroll
    for (int i = 0; i < kB; ++i) {
      if (i < nb) stage_block<T>(z, y, (c0 + i) * kLevel1, V, has_p, sz + i * kLevel1, sy + i * kLevel1);
      cp_async_commit();
    }
    // every block's level-3 masses first, then the picks of all blocks
    // together (warp i picks inside block i)
    float h0[kB], h1[kB], mass[kB];
    int cand[kB];
#pragma unroll
    for (int i = 0; i < kB; ++i) {
      h0[i] = 0.f;
      h1[i] = 0.f;
      cp_async_wait_pending(kB - 1 - i);  // this thread's copies of block i; it alone reads them here
      if (i < nb) staged_halves<T>(sz + i * kLevel1, sy + i * kLevel1, job, has_p, h0[i], h1[i]);
    }
    blocks_pick<kB>(
        h0, h1, c0 * kLevel1, V, nb, job,
        [&](int i, int t) {
          const int e = i * kLevel1 + staged_at<T>(t - (c0 + i) * kLevel1);
          return resid1(staged1(sz + e), has_p ? staged1(sy + e) : 0.f, job, has_p);
        },
        scs, mass, cand);
    if (threadIdx.x == 0) {
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        if (i < nb) {
          masses[c0 + i] = mass[i];
          cands[c0 + i] = cand[i];
        }
      }
    }
  } else {
    for (int i = 0; i < nb; ++i) {
      float mass;
      const int cand = block_candidate_global<T, false>(z, y, (c0 + i) * kLevel1, V, job, has_p, sc, &mass);
      if (threadIdx.x == 0) {
        masses[c0 + i] = mass;
        cands[c0 + i] = cand;
      }
    }
  }
  if (threadIdx.x == 0) {
    __threadfence();  // publish before counting in
    const unsigned long long state = count_in(w.arrivals + b, late);
    const bool last = static_cast<unsigned>(state) == static_cast<unsigned>(G);
    // 0: not last; 1: last, sample; 2: last, some CTA's wait ran out;
    // 3: last, the walk failed the request (then no CTA sampled, and only a
    // CTA whose wait ran out can have seen otherwise)
    s_last = !last ? 0 : (state >> 32) != 0 ? 2 : failed ? 3 : 1;
    if (last) w.arrivals[b] = 0;  // every CTA of the request has counted in
  }
  __syncthreads();
  if (s_last == 0 || s_last == 3) return;
  __threadfence();  // see the other CTAs' masses and candidates
  if (s_last == 2) {
    // Some CTA of the request gave up waiting for its row statistics, so
    // not every block was evaluated: the request fails as a whole.
    if (threadIdx.x <= N) p.out_tokens[static_cast<size_t>(b) * (N + 1) + threadIdx.x] = -1;
    if (threadIdx.x == 0) {
      p.out_accept[b] = -1;
      p.out_kv[b] = 0;
      atomicOr(w.err, kErrWait);
    }
    return;
  }

  // Level 1 over the blocks' masses; with at most 32 blocks lane i fetches
  // block i's candidate together with its mass.
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int mine = (S3 <= 32 && lane < S3) ? __ldcg(cands + lane) : -1;
    const int c1 = warp_pick([&](int i) { return __ldcg(masses + i); }, S3, job.u[0]);
    const int tok = S3 <= 32 ? __shfl_sync(kFull, mine, c1 & 31) : (c1 >= 0 ? __ldcg(cands + c1) : 0);
    if (lane == 0) {
      sc.pick = c1;
      sc.tok = tok;
    }
  }
  __syncthreads();
  int c1 = sc.pick;
  if (c1 < 0 && has_p) {
    // The residual has no mass anywhere: draw from q (same levels, same
    // uniforms), every block redone by this CTA.
    for (int cc = 0; cc < S3; ++cc) {
      float mq;
      const int cq = block_candidate_global<T, kVecPath>(z, z, cc * kLevel1, V, job, false, sc, &mq);
      if (threadIdx.x == 0) {
        masses[cc] = mq;
        cands[cc] = cq;
      }
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      const int cq1 = warp_pick([&](int i) { return __ldcg(masses + i); }, S3, job.u[0]);
      if (threadIdx.x == 0) sc.tok = cq1 >= 0 ? __ldcg(cands + cq1) : 0;
    }
    __syncthreads();
  } else if (c1 < 0) {
    if (threadIdx.x == 0) sc.tok = 0;  // no mass at all (cannot happen for q)
    __syncthreads();
  }
  if (threadIdx.x == 0) p.out_tokens[static_cast<size_t>(b) * (N + 1) + job.row] = sc.tok;
}

template <typename T, bool kVecPath, int kB>
cudaError_t launch_sample_k(const Problem& p, const Workspace& w, cudaStream_t s) {
  const long long blocks = static_cast<long long>(p.B) * ((w.S3 + kB - 1) / kB);
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const int smem = kVecPath ? stage_bytes<T, kB>() : 0;
  if (kVecPath) {
    // above the default 48 KB of dynamic shared memory: opt in (cheap, idempotent)
    const cudaError_t e = cudaFuncSetAttribute(sample_kernel<T, kVecPath, kB>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  // Programmatic dependent launch: the grid may be scheduled once every
  // row-statistics CTA has started (they are all resident or done, so CTAs
  // of this grid that poll for partials never hold back a CTA they wait for).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kST);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sample_kernel<T, kVecPath, kB>, p, w);
}

template <typename T, bool kVecPath>
cudaError_t launch_sample_t(const Problem& p, const Workspace& w, cudaStream_t s) {
  constexpr int kB = blocks_per_cta<T>();
  if (kB > 1 && SV_SAMPLE_SMALL_PER_SM > 0) {
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    if (static_cast<long long>(p.B) * w.S3 <= static_cast<long long>(sms) * SV_SAMPLE_SMALL_PER_SM)
      return launch_sample_k<T, kVecPath, 1>(p, w, s);
  }
  return launch_sample_k<T, kVecPath, kB>(p, w, s);
}

}  // namespace

cudaError_t launch_sample(int dtype, bool vec, const Problem& p, const Workspace& w,
                          cudaStream_t s) {
  if (dtype == 1)
    return vec ? launch_sample_t<__nv_bfloat16, true>(p, w, s)
               : launch_sample_t<__nv_bfloat16, false>(p, w, s);
  return vec ? launch_sample_t<float, true>(p, w, s) : launch_sample_t<float, false>(p, w, s);
}

}  // namespace sv
