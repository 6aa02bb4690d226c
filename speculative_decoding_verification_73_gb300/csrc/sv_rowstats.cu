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
// maximum and the lowest index holding it; its draft rows are never read.
//
// Rows are numbered request-major: request b owns rows b(2N+1) .. b(2N+1)+2N,
// its N+1 target rows first, then its N draft rows.  A row is cut into
// 32 KB chunks; partials[row][chunk] receives each chunk's statistics.
//
// Two kernels compute the same partials:
//  * ring: one persistent CTA per SM streams its share of the chunks
//    through a ring of kRingStages shared-memory stages filled by bulk
//    copies (cp.async.bulk) that complete on mbarriers, so several chunks
//    per SM are always in flight while the CTA reduces the current one.  The
//    active chunks (the draft rows of greedy requests are skipped) are dealt
//    out round robin: chunk k of the request-major list goes to CTA k mod G.
//  * direct: one CTA per chunk reading global memory with 16-byte loads (or
//    scalar loads when rows are not 16-byte aligned); used when the ring's
//    requirements (aligned rows, B <= kRingMaxB) do not hold.
// In both, the chunk maximum is reduced over the CTA first and every
// exponent then uses that one reference.

#include <climits>
#include <cuda_bf16.h>

#include "sv_device.cuh"

namespace sv {
namespace {

constexpr int kPer = kRowChunkBytes / 16 / kThreads;  // 16-byte vectors per thread per chunk
constexpr unsigned kWaitTries = 1u << 22;              // mbarrier polls before giving up

struct RowRef {
  bool draft;
  size_t offset;  // element offset of the row in its tensor
};

__device__ __forceinline__ RowRef row_of(const Problem& p, int b, int slot) {
  RowRef r;
  r.draft = slot > p.N;
  r.offset = r.draft ? (static_cast<size_t>(b) * p.N + (slot - p.N - 1)) * p.V
                     : (static_cast<size_t>(b) * (p.N + 1) + slot) * p.V;
  return r;
}

// c = M k; false for a chunk that contributes nothing (-inf maximum) or is
// bad (NaN, +inf, or a scaled maximum outside the float range).
__device__ __forceinline__ bool sampled_reference(float chunk_max, float k, float* c) {
  *c = chunk_max * k;
  return chunk_max > -INFINITY && chunk_max < INFINITY && fabsf(*c) <= 3.40282347e38f;
}

// Statistics of one chunk whose 16-byte vectors (vector v of the chunk in
// raw[i] with v = threadIdx.x + i * kThreads, -inf padding past the end) are
// in registers.  All threads call it; the result is valid in every thread.
template <typename T>
__device__ __forceinline__ Partial chunk_partial(const uint4 (&raw)[kPer], int beg, bool greedy,
                                                 float k) {
  using E = Elem<T>;
  constexpr int kVec = E::kVec;
  __shared__ float red_f[kThreads / 32];
  __shared__ float red_g[kThreads / 32];
  __shared__ int red_i[kThreads / 32];
  float m = E::vmax_nan(raw[0]);
#pragma unroll
  for (int i = 1; i < kPer; ++i) m = fmax_nan(m, E::vmax_nan(raw[i]));
  const float cmax = block_max_nan(m, red_f);
  Partial out;
  out.pad = 0;
  if (greedy) {
    int idx = INT_MAX;
    if (m == cmax) {  // lowest index of this thread holding the chunk maximum
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
          if (idx == INT_MAX && E::get(raw[i], e) == cmax)
            idx = beg + (threadIdx.x + i * kThreads) * kVec + e;
        }
      }
    }
    out.idx = block_min_int(idx, red_i);
    out.a = cmax;
    out.s = (cmax != cmax) ? __int_as_float(0x7fc00000) : 0.f;
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
  return out;
}

// Same statistics from scalar loads (rows not 16-byte aligned); two passes
// over the chunk, the second hitting L1/L2.
template <typename T>
__device__ Partial chunk_partial_scalar(const T* row, int beg, int end, bool greedy, float k) {
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
    out.idx = block_min_int(idx, red_i);
    out.a = cmax;
    out.s = (cmax != cmax) ? __int_as_float(0x7fc00000) : 0.f;
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
  return out;
}

// ------------------------------------------------------------------ direct

template <typename T, bool kVecPath>
__global__ void __launch_bounds__(kThreads) rowstats_direct_kernel(Problem p, Workspace w) {
  using E = Elem<T>;
  const int S1 = w.S1;
  const int per = 2 * p.N + 1;
  const int row = blockIdx.x / S1;
  const int chunk = blockIdx.x - row * S1;
  const int b = row / per;
  const int slot = row - b * per;
  const int mode = temp_mode(p.temperature[b]);
  if (mode == kModeInvalid || (mode == kModeGreedy && slot > p.N)) return;  // CTA-uniform
  const RowRef r = row_of(p, b, slot);
  const T* base = static_cast<const T*>(r.draft ? p.draft : p.target) + r.offset;
  constexpr int kChunk = kRowChunkBytes / static_cast<int>(sizeof(T));
  const int beg = chunk * kChunk;
  const int end = min(p.V, beg + kChunk);
  const bool greedy = mode == kModeGreedy;
  const float k = greedy ? 0.f : scale_of(p.temperature[b]);
  Partial out;
  if (kVecPath) {
    const uint4* vp = reinterpret_cast<const uint4*>(base + beg);
    const int nv = (end - beg) / E::kVec;
    uint4 raw[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int v = threadIdx.x + i * kThreads;
      raw[i] = v < nv ? ld_stream16(vp + v)
                      : make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
    }
    out = chunk_partial<T>(raw, beg, greedy, k);
  } else {
    out = chunk_partial_scalar<T>(base, beg, end, greedy, k);
  }
  if (threadIdx.x == 0) w.partials[static_cast<size_t>(row) * S1 + chunk] = out;
}

// ------------------------------------------------------------------ ring

// Chunks a request contributes: none for an invalid temperature (the walk
// reports it), the target rows for a greedy request, all rows otherwise.
__device__ __forceinline__ unsigned request_chunks(int mode, int N, int S1) {
  if (mode == kModeInvalid) return 0u;
  return static_cast<unsigned>(S1) * static_cast<unsigned>(mode == kModeGreedy ? N + 1 : 2 * N + 1);
}

struct Item {
  int b, slot, chunk;
  bool greedy;
};

// Active chunk k -> (request, row slot, chunk).  prefix[b] is the number of
// active chunks before request b; `cursor` only moves forward.
__device__ __forceinline__ Item decode_item(unsigned k, const unsigned* prefix,
                                            const unsigned char* modes, int& cursor, int S1) {
  while (prefix[cursor + 1] <= k) ++cursor;
  Item it;
  it.b = cursor;
  const unsigned l = k - prefix[cursor];
  it.slot = static_cast<int>(l / static_cast<unsigned>(S1));
  it.chunk = static_cast<int>(l - static_cast<unsigned>(it.slot) * S1);
  it.greedy = modes[cursor] == kModeGreedy;
  return it;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) rowstats_ring_kernel(Problem p, Workspace w) {
  using E = Elem<T>;
  constexpr int kChunk = kRowChunkBytes / static_cast<int>(sizeof(T));
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kRingStages * kRowChunkBytes);
  unsigned* prefix = reinterpret_cast<unsigned*>(bars + kRingStages);
  unsigned char* modes = reinterpret_cast<unsigned char*>(prefix + p.B + 1);
  __shared__ unsigned scan_scratch[kThreads / 32];
  __shared__ int s_abort;

  const int B = p.B, N = p.N, S1 = w.S1;

  // Per-request active chunk counts and their exclusive prefix.
  const int per_thread = (B + kThreads - 1) / kThreads;
  const int b0 = threadIdx.x * per_thread;
  unsigned local = 0;
  for (int i = 0; i < per_thread; ++i) {
    const int b = b0 + i;
    if (b < B) {
      const int mode = temp_mode(p.temperature[b]);
      modes[b] = static_cast<unsigned char>(mode);
      local += request_chunks(mode, N, S1);
    }
  }
  unsigned total;
  unsigned run = block_exclusive_scan_u32(local, scan_scratch, &total);
  for (int i = 0; i < per_thread; ++i) {
    const int b = b0 + i;
    if (b < B) {
      prefix[b] = run;
      run += request_chunks(modes[b], N, S1);
    }
  }
  if (threadIdx.x == 0) {
    prefix[B] = total;
    s_abort = 0;
    for (int s = 0; s < kRingStages; ++s) mbar_init(smem_u32(bars + s), 1);
    fence_mbar_init();
  }
  __syncthreads();

  const unsigned G = gridDim.x, g = blockIdx.x;
  const unsigned my_items = total > g ? (total - g + G - 1) / G : 0u;

  // Producer (thread 0): start the copy of this CTA's m-th chunk into stage
  // m % kRingStages.
  int pcursor = 0;
  auto issue = [&](unsigned m) {
    if (m >= my_items) return;
    const Item it = decode_item(g + m * G, prefix, modes, pcursor, S1);
    const RowRef r = row_of(p, it.b, it.slot);
    const T* src = static_cast<const T*>(r.draft ? p.draft : p.target) + r.offset +
                   static_cast<size_t>(it.chunk) * kChunk;
    const int n = min(p.V - it.chunk * kChunk, kChunk);
    const uint32_t bytes = static_cast<uint32_t>(n) * sizeof(T);
    const int s = static_cast<int>(m % kRingStages);
    const uint32_t bar = smem_u32(bars + s);
    mbar_arrive_expect_tx(bar, bytes);
    bulk_copy_g2s(smem_u32(ring + s * kRowChunkBytes), src, bytes, bar);
  };
  if (threadIdx.x == 0) {
    for (unsigned m = 0; m + 1 < kRingStages; ++m) issue(m);
  }

  int ccursor = 0;
  unsigned m = 0;
  for (; m < my_items; ++m) {
    if (threadIdx.x == 0) {
      // Refill the stage consumed in iteration m - 1.  Every thread has
      // passed that iteration's last barrier, so its reads of the stage are
      // done; the proxy fence orders them before the bulk copy's writes.
      fence_proxy_async_smem();
      issue(m + kRingStages - 1);
    }
    const Item it = decode_item(g + m * G, prefix, modes, ccursor, S1);
    const int s = static_cast<int>(m % kRingStages);
    const uint32_t parity = (m / kRingStages) & 1u;
    if (!mbar_wait_bounded(smem_u32(bars + s), parity, kWaitTries)) {
      atomicOr(w.err, kErrTimeout);
      s_abort = 1;
    }
    __syncthreads();
    if (s_abort) break;
    const int beg = it.chunk * kChunk;
    const int nv = (min(p.V, beg + kChunk) - beg) / E::kVec;
    const uint4* stage = reinterpret_cast<const uint4*>(ring + s * kRowChunkBytes);
    uint4 raw[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int v = threadIdx.x + i * kThreads;
      raw[i] = v < nv ? stage[v]
                      : make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
    }
    const float k = it.greedy ? 0.f : scale_of(p.temperature[it.b]);
    const Partial out = chunk_partial<T>(raw, beg, it.greedy, k);
    if (threadIdx.x == 0) {
      const size_t row = static_cast<size_t>(it.b) * (2 * N + 1) + it.slot;
      w.partials[row * S1 + it.chunk] = out;
    }
  }
  if (s_abort && threadIdx.x == 0) {
    // Do not leave while copies into this CTA's shared memory may still be
    // in flight: wait (bounded) on every copy issued after the one that
    // timed out.
    const unsigned issued = min(my_items, m + kRingStages);  // items m .. m+kRingStages-1 may be in flight
    for (unsigned q = m; q < issued; ++q)
      mbar_wait_bounded(smem_u32(bars + q % kRingStages), (q / kRingStages) & 1u, kWaitTries);
  }
}

}  // namespace

size_t ring_smem_bytes(int B) {
  return static_cast<size_t>(kRingStages) * kRowChunkBytes + kRingStages * sizeof(uint64_t) +
         (static_cast<size_t>(B) + 1) * sizeof(unsigned) + static_cast<size_t>(B);
}

cudaError_t prepare_rowstats(int max_B) {
  const int bytes = static_cast<int>(ring_smem_bytes(max_B < kRingMaxB ? max_B : kRingMaxB));
  cudaError_t e = cudaFuncSetAttribute(rowstats_ring_kernel<__nv_bfloat16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(rowstats_ring_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              bytes);
}

cudaError_t launch_rowstats(int dtype, bool vec, int ring_ctas, const Problem& p, const Workspace& w,
                            cudaStream_t s) {
  const long long blocks = static_cast<long long>(p.B) * (2 * p.N + 1) * w.S1;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (vec && ring_ctas > 0 && p.B <= kRingMaxB) {
    const size_t smem = ring_smem_bytes(p.B);
    if (dtype == 1)
      rowstats_ring_kernel<__nv_bfloat16><<<ring_ctas, kThreads, smem, s>>>(p, w);
    else
      rowstats_ring_kernel<float><<<ring_ctas, kThreads, smem, s>>>(p, w);
    return cudaGetLastError();
  }
  const dim3 grid(static_cast<unsigned>(blocks));
  if (dtype == 1) {
    if (vec)
      rowstats_direct_kernel<__nv_bfloat16, true><<<grid, kThreads, 0, s>>>(p, w);
    else
      rowstats_direct_kernel<__nv_bfloat16, false><<<grid, kThreads, 0, s>>>(p, w);
  } else {
    if (vec)
      rowstats_direct_kernel<float, true><<<grid, kThreads, 0, s>>>(p, w);
    else
      rowstats_direct_kernel<float, false><<<grid, kThreads, 0, s>>>(p, w);
  }
  return cudaGetLastError();
}

}  // namespace sv
