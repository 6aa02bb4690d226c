// Correction / bonus sampling by inverse CDF, touching only the one row (or
// row pair) per request that the walk selected.
//
// "Speculative Decoding and EAGLE-3" lesson, "Invariant: Leviathan rejection
// sampling" and "Build it" step 2: after a rejection at position j the token
// comes from the residual r_t = (q_j(t) - p_j(t))_+ normalised by its sum
// (from q_j itself if that sum is 0); after a full acceptance it comes from
// q_{N+1}.  The sample is the smallest vocabulary index t whose running sum
// of r exceeds u * sum(r).
//
// Grid: B x S3 CTAs, one per (request, 16 KB chunk).  Each CTA sums r over its
// chunk; the last CTA of a request to finish (counted with an atomic, no
// waiting) turns the chunk sums into a prefix, finds the chunk holding
// u * sum(r), rescans only that chunk with a CTA-wide scan, and writes the
// token.  It then resets the request's counter for the next call.

#include <climits>
#include <cuda_bf16.h>

#include "sv_device.cuh"

namespace sv {
namespace {

// r_t from one target value (and one draft value when has_p).  Both the
// chunk sums and the rescan evaluate exactly this expression.
__device__ __forceinline__ float resid(float zt, float yt, const Job& job, bool has_p) {
  const float q = ex2(fmaf(zt, job.k, -job.cq)) * job.inv_sq;
  if (!has_p) return q;
  const float pr = ex2(fmaf(yt, job.k, -job.cp)) * job.inv_sp;
  return fmaxf(q - pr, 0.f);
}

template <typename T, bool kVecPath>
__device__ float chunk_sum(const T* z, const T* y, int beg, int end, const Job& job, bool has_p,
                           float* scratch) {
  using E = Elem<T>;
  float s = 0.f;
  if (kVecPath) {
    constexpr int kVec = E::kVec;
    constexpr int kPer = kSampleChunkBytes / 16 / kThreads;
    const uint4* zp = reinterpret_cast<const uint4*>(z + beg);
    const uint4* yp = reinterpret_cast<const uint4*>(y + beg);
    const int nv = (end - beg) / kVec;
    uint4 zr[kPer], yr[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int v = threadIdx.x + i * kThreads;
      const bool in = v < nv;
      zr[i] = in ? __ldg(zp + v) : make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
      yr[i] = (in && has_p) ? __ldg(yp + v) : zr[i];
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
#pragma unroll
      for (int e = 0; e < kVec; ++e) s += resid(E::get(zr[i], e), E::get(yr[i], e), job, has_p);
    }
  } else {
    for (int t = beg + threadIdx.x; t < end; t += kThreads) {
      const float zt = E::load1(z + t);
      const float yt = has_p ? E::load1(y + t) : 0.f;
      s += resid(zt, yt, job, has_p);
    }
  }
  return block_sum(s, scratch);
}

template <typename T, bool kVecPath>
__global__ void __launch_bounds__(kThreads) sample_kernel(Problem p, Workspace w) {
  using E = Elem<T>;
  constexpr int kChunk = kSampleChunkBytes / static_cast<int>(sizeof(T));
  constexpr int kSeg = kChunk / kThreads;  // contiguous elements per thread in the rescan
  __shared__ float red[kThreads / 32];
  __shared__ float red2[kThreads / 32];
  __shared__ int red_i[kThreads / 32];
  __shared__ int red_j[kThreads / 32];
  __shared__ int s_last;
  __shared__ float s_sel[3];  // chunk index (as bits), prefix before it, target
  const int S3 = w.S3;
  const int b = blockIdx.x / S3;
  const int c = blockIdx.x - b * S3;
  const Job job = w.jobs[b];
  if (job.kind == kJobNone) return;  // CTA-uniform
  const int N = p.N, V = p.V;
  const T* z = static_cast<const T*>(p.target) + (static_cast<size_t>(b) * (N + 1) + job.row) * V;
  const T* y = job.kind == kJobResidual
                   ? static_cast<const T*>(p.draft) + (static_cast<size_t>(b) * N + job.row) * V
                   : z;
  bool has_p = job.kind == kJobResidual;
  float* sums = w.chunk_sums + static_cast<size_t>(b) * S3;

  const int beg = c * kChunk;
  const float part = chunk_sum<T, kVecPath>(z, y, beg, min(V, beg + kChunk), job, has_p, red);
  if (threadIdx.x == 0) {
    sums[c] = part;
    __threadfence();
    const unsigned prev = atomicAdd(w.counters + b, 1u);
    s_last = prev == static_cast<unsigned>(S3 - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- last CTA of request b: locate the chunk, then the token.
  for (int pass = 0; pass < 2; ++pass) {
    if (threadIdx.x == 0) {
      float prefix = 0.f;
      for (int i = 0; i < S3; ++i) prefix += __ldcg(sums + i);
      const float total = prefix;
      const float target = job.u * total;
      int sel = -1, last_pos = -1;
      float before = 0.f, before_last = 0.f, run = 0.f;
      for (int i = 0; i < S3; ++i) {
        const float v = __ldcg(sums + i);
        if (v > 0.f) {
          last_pos = i;
          before_last = run;
        }
        if (sel < 0 && run + v > target) {
          sel = i;
          before = run;
        }
        run += v;
      }
      if (sel < 0) {  // rounding put the target at or past the end
        sel = last_pos;
        before = before_last;
      }
      s_sel[0] = __int_as_float(total > 0.f ? sel : -1);
      s_sel[1] = before;
      s_sel[2] = target;
    }
    __syncthreads();
    if (__float_as_int(s_sel[0]) >= 0) break;
    // The residual has no mass: sample from q instead (recompute every chunk).
    if (!has_p || pass == 1) break;
    has_p = false;
    for (int i = 0; i < S3; ++i) {
      const int bi = i * kChunk;
      const float v = chunk_sum<T, kVecPath>(z, y, bi, min(V, bi + kChunk), job, false, red);
      if (threadIdx.x == 0) sums[i] = v;
      __syncthreads();
    }
    __threadfence_block();
  }
  const int sel = __float_as_int(s_sel[0]);
  int token = 0;
  if (sel >= 0) {
    const float before = s_sel[1], target = s_sel[2];
    const int cbeg = sel * kChunk;
    const int cend = min(V, cbeg + kChunk);
    const int t0 = cbeg + threadIdx.x * kSeg;
    float r[kSeg];
    if (kVecPath) {
      constexpr int kVec = E::kVec;
      constexpr int kVecs = kSeg / kVec;
#pragma unroll
      for (int i = 0; i < kVecs; ++i) {
        const int e0 = t0 + i * kVec;
        const bool in = e0 < cend;
        const uint4 zv = in ? __ldg(reinterpret_cast<const uint4*>(z + e0))
                            : make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
        const uint4 yv = (in && has_p) ? __ldg(reinterpret_cast<const uint4*>(y + e0)) : zv;
#pragma unroll
        for (int e = 0; e < kVec; ++e) r[i * kVec + e] = resid(E::get(zv, e), E::get(yv, e), job, has_p);
      }
    } else {
#pragma unroll
      for (int i = 0; i < kSeg; ++i) {
        const int t = t0 + i;
        if (t < cend) {
          r[i] = resid(E::load1(z + t), has_p ? E::load1(y + t) : 0.f, job, has_p);
        } else {
          r[i] = 0.f;
        }
      }
    }
    float mine = 0.f;
#pragma unroll
    for (int i = 0; i < kSeg; ++i) mine += r[i];
    float total;
    float run = before + block_exclusive_scan(mine, red2, &total);
    int hit = INT_MAX, lastpos = -1;
#pragma unroll
    for (int i = 0; i < kSeg; ++i) {
      run += r[i];
      if (hit == INT_MAX && run > target) hit = t0 + i;
      if (r[i] > 0.f) lastpos = t0 + i;
    }
    hit = block_min_int(hit, red_i);
    lastpos = block_max_int(lastpos, red_j);
    token = hit != INT_MAX ? hit : lastpos;
  }
  if (threadIdx.x == 0) {
    p.out_tokens[static_cast<size_t>(b) * (N + 1) + job.row] = token;
    w.counters[b] = 0u;
  }
}

}  // namespace

cudaError_t launch_sample(int dtype, bool vec, const Problem& p, const Workspace& w,
                          cudaStream_t s) {
  const long long blocks = static_cast<long long>(p.B) * w.S3;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const dim3 grid(static_cast<unsigned>(blocks));
  if (dtype == 1) {
    if (vec)
      sample_kernel<__nv_bfloat16, true><<<grid, kThreads, 0, s>>>(p, w);
    else
      sample_kernel<__nv_bfloat16, false><<<grid, kThreads, 0, s>>>(p, w);
  } else {
    if (vec)
      sample_kernel<float, true><<<grid, kThreads, 0, s>>>(p, w);
    else
      sample_kernel<float, false><<<grid, kThreads, 0, s>>>(p, w);
  }
  return cudaGetLastError();
}

}  // namespace sv
