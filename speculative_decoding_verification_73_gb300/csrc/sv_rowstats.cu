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
// chunks; partials[row][chunk] receives each chunk's statistics.
//
// Two kernels compute the partials:
//  * ring (8 KB chunks): one persistent CTA per SM.  A producer warp streams
//    the CTA's share of the chunks through kRingStages shared-memory stages
//    with bulk copies (cp.async.bulk) that complete on "full" mbarriers;
//    kRingWarps consumer warps each reduce whole chunks on their own (warp
//    shuffles only, no CTA barrier) and release the stage on an "empty"
//    mbarrier.  The active chunks (draft rows of greedy requests are
//    skipped) are dealt round robin: chunk k of the request-major list goes
//    to CTA k mod G, and a CTA's m-th chunk to consumer warp m mod kRingWarps.
//  * direct (32 KB chunks): one CTA per chunk reading global memory with
//    16-byte loads (or scalar loads when rows are not 16-byte aligned); used
//    when the ring's requirements (aligned rows, B <= kRingMaxB) do not hold.
// In both, a chunk's maximum is found first and every exponent uses that one
// reference.

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

constexpr int kRingThreads = (kRingWarps + 1) * 32;  // consumer warps + one producer warp
constexpr int kWarpVecs = kRingChunkBytes / 16 / 32;  // 16-byte vectors per lane per chunk

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

__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmax_nan(v, __shfl_xor_sync(kFull, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ int warp_min_int(int v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// One warp reduces one chunk held in shared memory (nv 16-byte vectors, the
// chunk starting at element beg of its row): two passes over the stage,
// the chunk maximum first, then the exponent sum or the argmax.
template <typename T>
__device__ __forceinline__ Partial warp_chunk_partial(const uint4* stage, int nv, int beg, bool greedy,
                                                      float k) {
  using E = Elem<T>;
  constexpr int kVec = E::kVec;
  const int lane = threadIdx.x & 31;
  float m = -INFINITY;
#pragma unroll 8
  for (int i = 0; i < kWarpVecs; ++i) {
    const int v = lane + i * 32;
    if (v < nv) m = fmax_nan(m, E::vmax_nan(stage[v]));
  }
  const float cmax = warp_max_nan(m);
  Partial out;
  out.pad = 0;
  if (greedy) {
    int idx = INT_MAX;
    if (m == cmax) {  // lowest index of this lane holding the chunk maximum
      for (int i = 0; i < kWarpVecs && idx == INT_MAX; ++i) {
        const int v = lane + i * 32;
        if (v >= nv) break;
        const uint4 x = stage[v];
#pragma unroll
        for (int e = 0; e < kVec; ++e)
          if (idx == INT_MAX && E::get(x, e) == cmax) idx = beg + v * kVec + e;
      }
    }
    out.idx = warp_min_int(idx);
    out.a = cmax;
    out.s = (cmax != cmax) ? __int_as_float(0x7fc00000) : 0.f;
  } else {
    float c;
    float s = 0.f;
    const bool ok = sampled_reference(cmax, k, &c);
    if (ok) {
#pragma unroll 4
      for (int i = 0; i < kWarpVecs; ++i) {
        const int v = lane + i * 32;
        if (v < nv) {
          const uint4 x = stage[v];
#pragma unroll
          for (int e = 0; e < kVec; ++e) s += ex2(fmaf(E::get(x, e), k, -c));
        }
      }
    }
    s = warp_sum(s);
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

template <typename T>
__global__ void __launch_bounds__(kRingThreads, 1) rowstats_ring_kernel(Problem p, Workspace w) {
  using E = Elem<T>;
  constexpr int kChunk = kRingChunkBytes / static_cast<int>(sizeof(T));
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kRingStages * kRingChunkBytes);
  uint64_t* empty = full + kRingStages;
  unsigned* prefix = reinterpret_cast<unsigned*>(empty + kRingStages);
  unsigned char* modes = reinterpret_cast<unsigned char*>(prefix + p.B + 1);
  __shared__ unsigned scan_scratch[32];

  const int B = p.B, N = p.N, S1 = w.S1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Per-request active chunk counts and their exclusive prefix (whole CTA).
  const int nthreads = blockDim.x;
  const int per_thread = (B + nthreads - 1) / nthreads;
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
  unsigned incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) scan_scratch[warp] = incl;
  __syncthreads();
  unsigned run = incl - local, total = 0;
  for (int q = 0; q < (nthreads >> 5); ++q) {
    const unsigned t = scan_scratch[q];
    if (q < warp) run += t;
    total += t;
  }
  for (int i = 0; i < per_thread; ++i) {
    const int b = b0 + i;
    if (b < B) {
      prefix[b] = run;
      run += request_chunks(modes[b], N, S1);
    }
  }
  if (threadIdx.x == 0) {
    prefix[B] = total;
    for (int s = 0; s < kRingStages; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const unsigned G = gridDim.x, g = blockIdx.x;
  const unsigned my_items = total > g ? (total - g + G - 1) / G : 0u;

  if (warp == kRingWarps) {
    // Producer: one lane issues the bulk copy of item m into stage
    // m % kRingStages once the consumer of item m - kRingStages released it.
    if (lane == 0) {
      int cursor = 0;
      for (unsigned m = 0; m < my_items; ++m) {
        const int s = static_cast<int>(m % kRingStages);
        const unsigned use = m / kRingStages;
        if (use > 0 && !mbar_wait_bounded(smem_u32(empty + s), (use - 1) & 1u, kWaitTries)) {
          atomicOr(w.err, kErrTimeout);
          break;
        }
        fence_proxy_async_smem();
        const Item it = decode_item(g + m * G, prefix, modes, cursor, S1);
        const RowRef r = row_of(p, it.b, it.slot);
        const T* src = static_cast<const T*>(r.draft ? p.draft : p.target) + r.offset +
                       static_cast<size_t>(it.chunk) * kChunk;
        const int n = min(p.V - it.chunk * kChunk, kChunk);
        const uint32_t bytes = static_cast<uint32_t>(n) * sizeof(T);
        const uint32_t bar = smem_u32(full + s);
        mbar_arrive_expect_tx(bar, bytes);
        bulk_copy_g2s(smem_u32(ring + s * kRingChunkBytes), src, bytes, bar);
      }
    }
    return;
  }

  // Consumers: warp q reduces items q, q + kRingWarps, ... of this CTA.
  int cursor = 0;
  for (unsigned m = warp; m < my_items; m += kRingWarps) {
    const Item it = decode_item(g + m * G, prefix, modes, cursor, S1);
    const int s = static_cast<int>(m % kRingStages);
    const bool ready = mbar_wait_bounded(smem_u32(full + s), (m / kRingStages) & 1u, kWaitTries);
    if (ready) {
      const int beg = it.chunk * kChunk;
      const int nv = (min(p.V, beg + kChunk) - beg) / E::kVec;
      const float k = it.greedy ? 0.f : scale_of(p.temperature[it.b]);
      const Partial out = warp_chunk_partial<T>(
          reinterpret_cast<const uint4*>(ring + s * kRingChunkBytes), nv, beg, it.greedy, k);
      if (lane == 0) {
        const size_t row = static_cast<size_t>(it.b) * (2 * N + 1) + it.slot;
        w.partials[row * S1 + it.chunk] = out;
      }
    } else if (lane == 0) {
      atomicOr(w.err, kErrTimeout);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(empty + s));
  }
}

}  // namespace

size_t ring_smem_bytes(int B) {
  return static_cast<size_t>(kRingStages) * kRingChunkBytes + 2 * kRingStages * sizeof(uint64_t) +
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
      rowstats_ring_kernel<__nv_bfloat16><<<ring_ctas, kRingThreads, smem, s>>>(p, w);
    else
      rowstats_ring_kernel<float><<<ring_ctas, kRingThreads, smem, s>>>(p, w);
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
