// The accept/reject walk and the correction / bonus sampling, touching only
// the one row (or row pair) per request that the walk selected.
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
// Grid: one cluster of kSampleCluster CTAs of kSampleThreads threads per
// request.  Every CTA first runs the request's accept/reject walk itself from
// the row-statistics partials (cheap, and no CTA waits for another to get
// it); rank 0 writes the walk's outputs.  For a sampled request each CTA then
// takes level-1 blocks rank, rank + cluster, ...: thread t evaluates tokens
// [32t, 32t + 32) of a block, which gives the block's level-3 masses (two per
// thread), level-2 masses (eight threads) and level-1 mass (the CTA) in one
// pass, kept in the CTA's shared memory.  After a cluster barrier rank 0 reads
// the masses it needs from the owners' shared memory (distributed shared
// memory), picks levels 1-3, re-evaluates only the 16 tokens of the chosen
// level-3 block for level 4, and writes the token; a second cluster barrier
// keeps the owners alive until then.  When a CTA owns more blocks than it can
// keep (V > kSampleCluster * kKeepBlocks * 8192) or the residual has no mass,
// rank 0 instead picks level 1 from masses in global memory and rescans the
// chosen block itself.
//
// r_t = max(q_t - p_t, 0) with q_t = 2^(z_t k - c_q) / s_q and likewise p_t,
// evaluated two tokens at a time with the paired float instructions.  Its
// rounding (a few float32 ulps of q_t per token) moves the level edges by
// ~1e-7 of the level mass, well inside the 1e-5 near-threshold window.

#include <climits>
#include <cuda_bf16.h>

#include "sv_device.cuh"
#include "sv_walk.cuh"

namespace sv {
namespace {

constexpr int kST = kSampleThreads;      // threads per sampler CTA
constexpr int kSegTok = kLevel1 / kST;   // tokens per thread in a level-1 block (32)
constexpr int kL2 = kLevel1 / kLevel2;   // level-2 blocks per level-1 block (32)
constexpr int kL3 = kLevel1 / kLevel3;   // level-3 blocks per level-1 block (512)
constexpr int kL3PerL2 = kLevel2 / kLevel3;  // 16
constexpr int kKeepBlocks = 4;           // level-1 blocks whose masses a CTA keeps
static_assert(kSegTok == 2 * kLevel3, "two level-3 blocks per thread");

__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Hardware barrier over all threads of all CTAs of the cluster; orders the
// memory accesses before it (release) with those after it (acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Load a float from the shared memory of CTA `rank` of this cluster, at the
// place where `local` lives in this CTA's shared memory.
__device__ __forceinline__ float ld_dsmem(const float* local, unsigned rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(local))), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

__device__ __forceinline__ float cta_sum(float v, float* scratch) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  v = 0.f;
#pragma unroll
  for (int w = 0; w < kST / 32; ++w) v += scratch[w];
  __syncthreads();
  return v;
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

// Scalar form for rows that are not 16-byte aligned (same arithmetic).
__device__ __forceinline__ float resid1(float zt, float yt, const Job& job, bool has_p) {
  const float q = ex2(fmaf(zt, job.k, -job.cq)) * job.inv_sq;
  if (!has_p) return q;
  return fmaxf(q - ex2(fmaf(yt, job.k, -job.cp)) * job.inv_sp, 0.f);
}

// r at tokens [t0, t0 + kSegTok) of the row pair (0 past cend): one thread's
// contiguous share of a level-1 block.
template <typename T, bool kVecPath>
__device__ __forceinline__ void resid_seg(const T* z, const T* y, int t0, int cend, const Job& job,
                                          bool has_p, float (&r)[kSegTok]) {
  using E = Elem<T>;
  if (kVecPath) {
    constexpr int kVec = E::kVec;
    const uint4 pad = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
    uint4 zv[kSegTok / kVec], yv[kSegTok / kVec];
#pragma unroll
    for (int i = 0; i < kSegTok / kVec; ++i) {
      const int e0 = t0 + i * kVec;
      const bool in = e0 < cend;
      zv[i] = in ? __ldg(reinterpret_cast<const uint4*>(z + e0)) : pad;
      yv[i] = (in && has_p) ? __ldg(reinterpret_cast<const uint4*>(y + e0)) : pad;
    }
#pragma unroll
    for (int i = 0; i < kSegTok / kVec; ++i) {
      float rv[kVec];
      resid_vec<T>(zv[i], yv[i], job, has_p, rv);
#pragma unroll
      for (int e = 0; e < kVec; ++e) r[i * kVec + e] = rv[e];
    }
  } else {
#pragma unroll
    for (int i = 0; i < kSegTok; ++i) {
      const int t = t0 + i;
      r[i] = t < cend ? resid1(E::load1(z + t), has_p ? E::load1(y + t) : 0.f, job, has_p) : 0.f;
    }
  }
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

// Inverse CDF over n masses, evaluated by one whole warp (all lanes get the
// result): the smallest c with running sum C_c > u * C_{n-1}; if none, the
// last c with mass > 0; -1 if every mass is 0.  Masses are read through
// `get(i)`, once each when n <= 32; longer lists are scanned in tiles of 32
// twice (total, then the crossing) with identical arithmetic.
template <typename Get>
__device__ int warp_pick(Get get, int n, float u) {
  const int lane = threadIdx.x & 31;
  if (n <= 32) {
    const float m = lane < n ? get(lane) : 0.f;
    float incl = m;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned pos = __ballot_sync(kFull, m > 0.f);
    if (!pos) return -1;
    const float target = u * __shfl_sync(kFull, incl, 31);
    const unsigned hit = __ballot_sync(kFull, lane < n && incl > target);
    return hit ? __ffs(hit) - 1 : 31 - __clz(pos);
  }
  float carry = 0.f;
  int last_pos = -1;
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    const float m = i < n ? get(i) : 0.f;
    float incl = m;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned pos = __ballot_sync(kFull, m > 0.f);
    if (pos) last_pos = base + 31 - __clz(pos);
    carry += __shfl_sync(kFull, incl, 31);
  }
  if (last_pos < 0) return -1;
  const float target = u * carry;
  carry = 0.f;
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    const float m = i < n ? get(i) : 0.f;
    float incl = m;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned hit = __ballot_sync(kFull, i < n && carry + incl > target);
    if (hit) return base + __ffs(hit) - 1;
    carry += __shfl_sync(kFull, incl, 31);
  }
  return last_pos;
}

template <typename T, bool kVecPath>
__global__ void __cluster_dims__(kSampleCluster, 1, 1) __launch_bounds__(kST, 3)
    sample_kernel(Problem p, Workspace w) {
  using E = Elem<T>;
  __shared__ float red[kST / 32];
  __shared__ float s_l1[kKeepBlocks];        // level-1 masses of the kept own blocks
  __shared__ float s_l2[kKeepBlocks][kL2];   // their level-2 masses
  __shared__ float s_l3[kKeepBlocks][kL3];   // their level-3 masses
  __shared__ float s_l4[kLevel3];            // the chosen level-3 block's token masses
  __shared__ int s_sel, s_g2, s_g3, s_tok;
  __shared__ Job s_job;
  const int S3 = w.S3;
  const int b = blockIdx.x / kSampleCluster;
  const unsigned rank = cluster_rank();
  // Only sampled requests need the other CTAs of the cluster (the choice is
  // the same in every CTA of a cluster, so either all of them reach the
  // cluster barriers below or none does); rank 0 writes the outputs.
  if (rank != 0 && temp_mode(p.temperature[b]) != kModeSampled) return;
  walk_request<T>(p, w, b, rank == 0, &s_job);
  __syncthreads();
  const Job job = s_job;
  if (job.kind == kJobNone) return;  // identical in every CTA of the cluster
  const int N = p.N, V = p.V;
  const T* z = static_cast<const T*>(p.target) + (static_cast<size_t>(b) * (N + 1) + job.row) * V;
  const T* y = job.kind == kJobResidual
                   ? static_cast<const T*>(p.draft) + (static_cast<size_t>(b) * N + job.row) * V
                   : z;
  bool has_p = job.kind == kJobResidual;
  float* sums = w.chunk_sums + static_cast<size_t>(b) * S3;
  const bool keep_all = S3 <= kSampleCluster * kKeepBlocks;

  // One pass over this CTA's level-1 blocks: masses at all three levels.
  int kept = 0;
  for (int c = static_cast<int>(rank); c < S3; c += kSampleCluster, ++kept) {
    const int cbeg = c * kLevel1;
    float h0, h1;
    resid_halves<T, kVecPath>(z, y, cbeg + threadIdx.x * kSegTok, min(V, cbeg + kLevel1), job, has_p,
                              h0, h1);
    float m2 = h0 + h1;  // level-2 mass: the 8 consecutive threads of a 256-token block
#pragma unroll
    for (int o = 1; o < kL3PerL2 / 2; o <<= 1) m2 += __shfl_xor_sync(kFull, m2, o);
    const float m1 = cta_sum(h0 + h1, red);
    if (keep_all) {
      s_l3[kept][2 * threadIdx.x] = h0;
      s_l3[kept][2 * threadIdx.x + 1] = h1;
      if ((threadIdx.x & (kL3PerL2 / 2 - 1)) == 0) s_l2[kept][threadIdx.x / (kL3PerL2 / 2)] = m2;
      if (threadIdx.x == 0) s_l1[kept] = m1;
    } else if (threadIdx.x == 0) {
      sums[c] = m1;
    }
  }
  if (!keep_all) __threadfence();
  cluster_sync();  // every owner's masses are in place
  if (rank != 0) {
    cluster_sync();  // stay resident until rank 0 has read them
    return;
  }

  // ---- rank 0 of request b.
  int sel = -1;
  if (keep_all) {
    if (threadIdx.x < 32) {
      const int c1 = warp_pick(
          [&](int c) { return ld_dsmem(&s_l1[c / kSampleCluster], c % kSampleCluster); }, S3, job.u[0]);
      int g2 = -1, g3 = -1;
      if (c1 >= 0) {
        const unsigned own = c1 % kSampleCluster;
        const int li = c1 / kSampleCluster;
        g2 = max(warp_pick([&](int i) { return ld_dsmem(&s_l2[li][i], own); }, kL2, job.u[1]), 0);
        g3 = max(warp_pick([&](int i) { return ld_dsmem(&s_l3[li][g2 * kL3PerL2 + i], own); }, kL3PerL2,
                           job.u[2]),
                 0);
      }
      if (threadIdx.x == 0) {
        s_sel = c1;
        s_g2 = g2;
        s_g3 = g3;
      }
    }
    __syncthreads();
    sel = s_sel;
  }
  cluster_sync();  // the owners may leave now
  int token = 0;
  if (keep_all && sel >= 0) {
    // Level 4: the 16 tokens of the chosen level-3 block.
    const int t0 = sel * kLevel1 + (s_g2 * kL3PerL2 + s_g3) * kLevel3;
    if (threadIdx.x < kLevel3) {
      const int t = t0 + threadIdx.x;
      s_l4[threadIdx.x] = t < V ? resid1(E::load1(z + t), has_p ? E::load1(y + t) : 0.f, job, has_p) : 0.f;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      const int g4 = max(warp_pick([&](int i) { return s_l4[i]; }, kLevel3, job.u[3]), 0);
      if (threadIdx.x == 0) s_tok = t0 + g4;
    }
    __syncthreads();
    token = s_tok;
  } else {
    // Level 1 from global masses (many blocks, or a residual without mass,
    // which falls back to q), then a rescan of the chosen block.
    if (keep_all) has_p = false;  // the residual had no mass
    for (int pass = 0; pass < 2; ++pass) {
      if (!keep_all || pass == 1) {
        if (threadIdx.x < 32) {
          const int s1 = warp_pick([&](int i) { return __ldcg(sums + i); }, S3, job.u[0]);
          if (threadIdx.x == 0) s_sel = s1;
        }
        __syncthreads();
        if (s_sel >= 0 || !has_p || pass == 1) break;
      }
      // q-only masses of every block (the residual had no mass)
      has_p = false;
      for (int c = 0; c < S3; ++c) {
        const int cbeg = c * kLevel1;
        float h0, h1;
        resid_halves<T, kVecPath>(z, y, cbeg + threadIdx.x * kSegTok, min(V, cbeg + kLevel1), job,
                                  false, h0, h1);
        const float m1 = cta_sum(h0 + h1, red);
        if (threadIdx.x == 0) sums[c] = m1;
      }
      __threadfence_block();
    }
    sel = s_sel;
    if (sel >= 0) {
      const int cbeg = sel * kLevel1;
      float r[kSegTok];
      resid_seg<T, kVecPath>(z, y, cbeg + threadIdx.x * kSegTok, min(V, cbeg + kLevel1), job, has_p, r);
      float h0 = 0.f, h1 = 0.f;
#pragma unroll
      for (int i = 0; i < kLevel3; ++i) {
        h0 += r[i];
        h1 += r[kLevel3 + i];
      }
      s_l3[0][2 * threadIdx.x] = h0;
      s_l3[0][2 * threadIdx.x + 1] = h1;
      float m2 = h0 + h1;
#pragma unroll
      for (int o = 1; o < kL3PerL2 / 2; o <<= 1) m2 += __shfl_xor_sync(kFull, m2, o);
      if ((threadIdx.x & (kL3PerL2 / 2 - 1)) == 0) s_l2[0][threadIdx.x / (kL3PerL2 / 2)] = m2;
      __syncthreads();
      if (threadIdx.x < 32) {
        const int g2 = max(warp_pick([&](int i) { return s_l2[0][i]; }, kL2, job.u[1]), 0);
        const int g3 = max(warp_pick([&](int i) { return s_l3[0][g2 * kL3PerL2 + i]; }, kL3PerL2,
                                     job.u[2]),
                           0);
        if (threadIdx.x == 0) {
          s_g2 = g2;
          s_g3 = g3;
        }
      }
      __syncthreads();
      const int blk3 = s_g2 * kL3PerL2 + s_g3;  // thread blk3 / 2 holds its tokens
      if (threadIdx.x == (blk3 >> 1)) {
#pragma unroll
        for (int i = 0; i < kLevel3; ++i) s_l4[i] = (blk3 & 1) ? r[kLevel3 + i] : r[i];
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        const int g4 = max(warp_pick([&](int i) { return s_l4[i]; }, kLevel3, job.u[3]), 0);
        if (threadIdx.x == 0) s_tok = cbeg + blk3 * kLevel3 + g4;
      }
      __syncthreads();
      token = s_tok;
    }
  }
  if (threadIdx.x == 0) p.out_tokens[static_cast<size_t>(b) * (N + 1) + job.row] = token;
}

}  // namespace

cudaError_t launch_sample(int dtype, bool vec, const Problem& p, const Workspace& w,
                          cudaStream_t s) {
  const long long blocks = static_cast<long long>(p.B) * kSampleCluster;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const dim3 grid(static_cast<unsigned>(blocks));
  if (dtype == 1) {
    if (vec)
      sample_kernel<__nv_bfloat16, true><<<grid, kST, 0, s>>>(p, w);
    else
      sample_kernel<__nv_bfloat16, false><<<grid, kST, 0, s>>>(p, w);
  } else {
    if (vec)
      sample_kernel<float, true><<<grid, kST, 0, s>>>(p, w);
    else
      sample_kernel<float, false><<<grid, kST, 0, s>>>(p, w);
  }
  return cudaGetLastError();
}

}  // namespace sv
