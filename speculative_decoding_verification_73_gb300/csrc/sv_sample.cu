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
// sums r over its share of the level-1 blocks (blocks rank, rank + cluster,
// ...), the cluster meets at one hardware cluster barrier, and rank 0 picks
// the level-1 block, rescans only that block for levels 2-4 (thread t holds
// the 16 tokens of level-3 block t) and writes the token.
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

constexpr int kST = kSampleThreads;        // threads per sampler CTA
constexpr int kSegTok = kLevel1 / kST;      // tokens per thread in a level-1 block (16)
static_assert(kSegTok == kLevel3, "one thread per level-3 block in the rescan");

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

// r for the (up to) 8 tokens of one 16-byte vector of each row; rv[e] gets
// token e of the vector.
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

// Residual mass of level-1 block [beg, end) (all threads; result in all).
template <typename T, bool kVecPath>
__device__ float block_mass(const T* z, const T* y, int beg, int end, const Job& job, bool has_p,
                            float* scratch) {
  using E = Elem<T>;
  float s = 0.f;
  if (kVecPath) {
    constexpr int kVec = E::kVec;
    constexpr int kPer = kLevel1 / kVec / kST;
    const uint4* zp = reinterpret_cast<const uint4*>(z + beg);
    const uint4* yp = reinterpret_cast<const uint4*>(y + beg);
    const int nv = (end - beg) / kVec;
    const uint4 pad = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
    uint4 zr[kPer], yr[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int v = threadIdx.x + i * kST;
      const bool in = v < nv;
      zr[i] = in ? __ldg(zp + v) : pad;
      yr[i] = (in && has_p) ? __ldg(yp + v) : pad;
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      float rv[kVec];
      resid_vec<T>(zr[i], yr[i], job, has_p, rv);
#pragma unroll
      for (int e = 0; e < kVec; ++e) s += rv[e];
    }
  } else {
    for (int t = beg + threadIdx.x; t < end; t += kST)
      s += resid1(E::load1(z + t), has_p ? E::load1(y + t) : 0.f, job, has_p);
  }
  return cta_sum(s, scratch);
}

// Inverse CDF over n masses, evaluated by one whole warp (all lanes get the
// result): the smallest c with running sum C_c > u * C_{n-1}; if none, the
// last c with mass > 0; -1 if every mass is 0.  Masses are read through
// `get(i)`.  Tiles of 32 are scanned in index order twice (total, then the
// crossing) with identical arithmetic.
template <typename Get>
__device__ int warp_pick(Get get, int n, float u) {
  const int lane = threadIdx.x & 31;
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

template <typename T, bool kVecPath>
__global__ void __cluster_dims__(kSampleCluster, 1, 1) __launch_bounds__(kST)
    sample_kernel(Problem p, Workspace w) {
  using E = Elem<T>;
  __shared__ float red[kST / 32];
  __shared__ float s_l2[kLevel1 / kLevel2];         // 32 level-2 masses
  __shared__ float s_l3[kLevel1 / kLevel3];         // 512 level-3 masses
  __shared__ float s_l4[kLevel3];                   // 16 token masses
  __shared__ int s_sel, s_g2, s_g3, s_tok;
  __shared__ Job s_job;
  const int S3 = w.S3;
  const int b = blockIdx.x / kSampleCluster;
  const unsigned rank = cluster_rank();
  // Only sampled requests need the other CTAs of the cluster (the choice is
  // the same in every CTA of a cluster, so either all of them reach the
  // cluster barrier below or none does); rank 0 writes the outputs.
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

  // Level-1 block masses: this CTA takes blocks rank, rank + cluster, ...
  for (int c = static_cast<int>(rank); c < S3; c += kSampleCluster) {
    const int beg = c * kLevel1;
    const float part = block_mass<T, kVecPath>(z, y, beg, min(V, beg + kLevel1), job, has_p, red);
    if (threadIdx.x == 0) sums[c] = part;
  }
  __threadfence();
  cluster_sync();
  if (rank != 0) return;

  // ---- rank 0 of request b.  Level 1: pick the block.
  for (int pass = 0; pass < 2; ++pass) {
    if (threadIdx.x < 32) {
      const int sel = warp_pick([&](int i) { return __ldcg(sums + i); }, S3, job.u[0]);
      if (threadIdx.x == 0) s_sel = sel;
    }
    __syncthreads();
    if (s_sel >= 0 || !has_p || pass == 1) break;
    // The residual has no mass: sample from q instead.
    has_p = false;
    for (int i = 0; i < S3; ++i) {
      const int bi = i * kLevel1;
      const float v = block_mass<T, kVecPath>(z, y, bi, min(V, bi + kLevel1), job, false, red);
      if (threadIdx.x == 0) sums[i] = v;
    }
    __threadfence_block();
  }
  const int sel = s_sel;
  int token = 0;
  if (sel >= 0) {
    // Rescan the chosen block: thread t holds tokens [16t, 16t + 16) of it,
    // i.e. level-3 block t; 16 threads make a level-2 block.
    const int cbeg = sel * kLevel1;
    const int cend = min(V, cbeg + kLevel1);
    const int t0 = cbeg + threadIdx.x * kSegTok;
    float r[kSegTok];
    if (kVecPath) {
      constexpr int kVec = E::kVec;
      const uint4 pad = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
#pragma unroll
      for (int i = 0; i < kSegTok / kVec; ++i) {
        const int e0 = t0 + i * kVec;
        const bool in = e0 < cend;
        const uint4 zv = in ? __ldg(reinterpret_cast<const uint4*>(z + e0)) : pad;
        const uint4 yv = (in && has_p) ? __ldg(reinterpret_cast<const uint4*>(y + e0)) : pad;
        float rv[kVec];
        resid_vec<T>(zv, yv, job, has_p, rv);
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
    float h = 0.f;
#pragma unroll
    for (int i = 0; i < kSegTok; ++i) h += r[i];
    s_l3[threadIdx.x] = h;
    float m2 = h;  // level-2 mass: the 16 consecutive threads of one 256-token block
#pragma unroll
    for (int o = 1; o < kLevel2 / kLevel3; o <<= 1) m2 += __shfl_xor_sync(kFull, m2, o);
    if ((threadIdx.x & (kLevel2 / kLevel3 - 1)) == 0) s_l2[threadIdx.x / (kLevel2 / kLevel3)] = m2;
    __syncthreads();
    if (threadIdx.x < 32) {
      // a chosen block has mass > 0, so each level below finds a sub-block
      // with mass; max(.., 0) only keeps the indices in range regardless
      const int g2 = max(warp_pick([&](int i) { return s_l2[i]; }, kLevel1 / kLevel2, job.u[1]), 0);
      const int g3 = max(warp_pick([&](int i) { return s_l3[g2 * (kLevel2 / kLevel3) + i]; },
                                   kLevel2 / kLevel3, job.u[2]),
                         0);
      if (threadIdx.x == 0) {
        s_g2 = g2;
        s_g3 = g3;
      }
    }
    __syncthreads();
    const int blk3 = s_g2 * (kLevel2 / kLevel3) + s_g3;  // level-3 block = thread index
    if (threadIdx.x == blk3) {
#pragma unroll
      for (int i = 0; i < kLevel3; ++i) s_l4[i] = r[i];
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      const int g4 = max(warp_pick([&](int i) { return s_l4[i]; }, kLevel3, job.u[3]), 0);
      if (threadIdx.x == 0) s_tok = cbeg + blk3 * kLevel3 + g4;
    }
    __syncthreads();
    token = s_tok;
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
