// Row statistics: one streaming pass over every logit row the verify step
// needs, producing per-chunk partials that the walk merges.
//
// For a sampled request (T > 0) both its N+1 target rows and its N draft rows
// are reduced to (c, s): c = fl(M k) with M the chunk maximum and
// k = log2(e)/T, s = sum_t 2^(x_t k - c); the walk merges chunks into
// log2 sum_t 2^(x_t k), the normaliser of softmax(x / T) ("Speculative
// Decoding and EAGLE-3" lesson, "Invariant: Leviathan rejection sampling":
// q and p are the verifier's and the drafter's next-token laws).  For a
// greedy request (T = 0) only its target rows are read and reduced to the
// maximum and the lowest index holding it; its draft rows are skipped.
//
// Grid: one CTA per (row, 32 KB chunk).  Each thread issues all of its 16-byte
// loads up front (8 per thread), so a CTA has 32 KB in flight; the chunk
// maximum is reduced over the CTA first, and every exponent then uses that
// one reference, so no per-thread rescaling is needed.
//
// The CTA that finishes the last chunk of a request (counted with an atomic
// per request; nothing waits) then runs that request's accept/reject walk,
// so walks overlap the other requests' streaming.

#include <climits>
#include <cuda_bf16.h>

#include "sv_device.cuh"
#include "sv_walk.cuh"

namespace sv {
namespace {

struct RowRef {
  int b;
  bool draft;
  size_t offset;  // element offset of the row in its tensor
};

// CTAs are numbered request-major: request b owns rows b(2N+1) .. b(2N+1)+2N,
// its N+1 target rows first, then its N draft rows, so a request's chunks are
// streamed together and its walk runs soon after.
__device__ __forceinline__ RowRef locate_row(const Problem& p, int row) {
  const int per = 2 * p.N + 1;
  RowRef r;
  r.b = row / per;
  const int i = row - r.b * per;
  r.draft = i > p.N;
  r.offset = r.draft ? (static_cast<size_t>(r.b) * p.N + (i - p.N - 1)) * p.V
                     : (static_cast<size_t>(r.b) * (p.N + 1) + i) * p.V;
  return r;
}

// Sampled-row partial from the chunk maximum M and the per-thread sum.
__device__ __forceinline__ bool sampled_reference(float chunk_max, float k, float* c) {
  // -inf chunk: nothing to add.  NaN / +inf / a maximum whose scaled value
  // leaves the float range: the partial is marked bad (NaN sum).
  *c = chunk_max * k;
  return chunk_max > -INFINITY && chunk_max < INFINITY && fabsf(*c) <= 3.40282347e38f;
}

template <typename T>
__device__ void chunk_vec(const T* row, int beg, int end, bool greedy, float k, Partial* slot) {
  using E = Elem<T>;
  constexpr int kVec = E::kVec;
  constexpr int kPer = kRowChunkBytes / 16 / kThreads;
  __shared__ float red_f[kThreads / 32];
  __shared__ float red_g[kThreads / 32];
  __shared__ int red_i[kThreads / 32];

  const uint4* vp = reinterpret_cast<const uint4*>(row + beg);
  const int nv = (end - beg) / kVec;
  uint4 raw[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int v = threadIdx.x + i * kThreads;
    if (v < nv) {
      raw[i] = ld_stream16(vp + v);
    } else {
      raw[i] = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
    }
  }
  float m = E::vmax_nan(raw[0]);
#pragma unroll
  for (int i = 1; i < kPer; ++i) m = fmax_nan(m, E::vmax_nan(raw[i]));
  const float cmax = block_max_nan(m, red_f);

  Partial out;
  out.pad = 0;
  if (greedy) {
    int idx = INT_MAX;
    if (m == cmax) {
      // lowest index of this thread holding the chunk maximum
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
          if (idx == INT_MAX && E::get(raw[i], e) == cmax)
            idx = beg + (threadIdx.x + i * kThreads) * kVec + e;
        }
      }
    }
    idx = block_min_int(idx, red_i);
    out.a = cmax;
    out.s = (cmax != cmax) ? __int_as_float(0x7fc00000) : 0.f;
    out.idx = idx;
  } else {
    float c;
    float s = 0.f;
    const bool ok = sampled_reference(cmax, k, &c);
    if (ok) {
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
#pragma unroll
        for (int e = 0; e < kVec; ++e) s += ex2(fmaf(E::get(raw[i], e), k, -c));
      }
    }
    s = block_sum(s, red_g);
    if (!ok) {
      if (cmax == -INFINITY) {
        c = -INFINITY;
        s = 0.f;
      } else {
        s = __int_as_float(0x7fc00000);
      }
    }
    out.a = c;
    out.s = s;
    out.idx = 0;
  }
  if (threadIdx.x == 0) *slot = out;
}

// Any V or alignment: scalar loads, two passes over the chunk (the second
// pass hits L1/L2).
template <typename T>
__device__ void chunk_scalar(const T* row, int beg, int end, bool greedy, float k, Partial* slot) {
  using E = Elem<T>;
  __shared__ float red_f[kThreads / 32];
  __shared__ float red_g[kThreads / 32];
  __shared__ int red_i[kThreads / 32];
  float m = -INFINITY;
  for (int t = beg + threadIdx.x; t < end; t += kThreads) m = fmax_nan(m, E::load1(row + t));
  const float cmax = block_max_nan(m, red_f);
  Partial out;
  out.pad = 0;
  if (greedy) {
    int idx = INT_MAX;
    if (m == cmax) {
      for (int t = beg + threadIdx.x; t < end; t += kThreads) {
        if (E::load1(row + t) == cmax) {
          idx = t;
          break;
        }
      }
    }
    idx = block_min_int(idx, red_i);
    out.a = cmax;
    out.s = (cmax != cmax) ? __int_as_float(0x7fc00000) : 0.f;
    out.idx = idx;
  } else {
    float c;
    float s = 0.f;
    const bool ok = sampled_reference(cmax, k, &c);
    if (ok) {
      for (int t = beg + threadIdx.x; t < end; t += kThreads) s += ex2(fmaf(E::load1(row + t), k, -c));
    }
    s = block_sum(s, red_g);
    if (!ok) {
      if (cmax == -INFINITY) {
        c = -INFINITY;
        s = 0.f;
      } else {
        s = __int_as_float(0x7fc00000);
      }
    }
    out.a = c;
    out.s = s;
    out.idx = 0;
  }
  if (threadIdx.x == 0) *slot = out;
}

template <typename T, bool kVecPath>
__global__ void __launch_bounds__(kThreads) rowstats_kernel(Problem p, Workspace w) {
  __shared__ int s_last;
  const int S1 = w.S1;
  const int row = blockIdx.x / S1;
  const int chunk = blockIdx.x - row * S1;
  const RowRef r = locate_row(p, row);
  const float t = p.temperature[r.b];
  const int mode = temp_mode(t);
  if (mode == kModeGreedy && r.draft) return;  // CTA-uniform; not counted
  if (mode == kModeInvalid && r.draft) return;
  if (mode != kModeInvalid) {
    const T* base = static_cast<const T*>(r.draft ? p.draft : p.target) + r.offset;
    constexpr int kChunk = kRowChunkBytes / static_cast<int>(sizeof(T));
    const int beg = chunk * kChunk;
    const int end = min(p.V, beg + kChunk);
    const bool greedy = mode == kModeGreedy;
    const float k = greedy ? 0.f : scale_of(t);
    Partial* slot = w.partials + static_cast<size_t>(row) * S1 + chunk;
    if (kVecPath) {
      chunk_vec<T>(base, beg, end, greedy, k, slot);
    } else {
      chunk_scalar<T>(base, beg, end, greedy, k, slot);
    }
  }
  // Count this chunk for its request: target rows always, draft rows only
  // when the request is sampled.  The CTA that brings the count to its total
  // runs the walk.
  if (threadIdx.x == 0) {
    const unsigned total =
        static_cast<unsigned>(S1) * static_cast<unsigned>(p.N + 1 + (mode == kModeSampled ? p.N : 0));
    __threadfence();
    const unsigned prev = atomicAdd(w.walk_counters + r.b, 1u);
    s_last = prev + 1 == total;
    if (s_last) w.walk_counters[r.b] = 0u;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  walk_request<T>(p, w, r.b);
}

}  // namespace

cudaError_t launch_rowstats(int dtype, bool vec, const Problem& p, const Workspace& w,
                            cudaStream_t s) {
  const long long rows = static_cast<long long>(p.B) * (2 * p.N + 1);
  const long long blocks = rows * w.S1;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const dim3 grid(static_cast<unsigned>(blocks));
  if (dtype == 1) {
    if (vec)
      rowstats_kernel<__nv_bfloat16, true><<<grid, kThreads, 0, s>>>(p, w);
    else
      rowstats_kernel<__nv_bfloat16, false><<<grid, kThreads, 0, s>>>(p, w);
  } else {
    if (vec)
      rowstats_kernel<float, true><<<grid, kThreads, 0, s>>>(p, w);
    else
      rowstats_kernel<float, false><<<grid, kThreads, 0, s>>>(p, w);
  }
  return cudaGetLastError();
}

}  // namespace sv
