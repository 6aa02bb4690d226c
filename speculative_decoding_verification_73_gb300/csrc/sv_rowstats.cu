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
// spans of kSpanBytes; one CTA reduces one span in a single streaming pass
// (16-byte non-allocating loads, the next group of loads in flight while the
// current one is reduced, a running maximum with a rescaled sum per thread,
// one CTA-wide merge per span) and writes partials[row][span].  Rows that
// are not 16-byte aligned take a scalar two-pass path over the same spans.

#include <climits>
#include <cuda_bf16.h>

#include "sv_device.cuh"

namespace sv {
namespace {



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

// ------------------------------------------------------------------ online

// One CTA reduces one span of kSpanBytes of a row in a single pass: thread t
// reads 16-byte vectors t, t + kThreads, ... of the span in groups of kGroup,
// the next group's loads issued before the current group is reduced, and
// keeps a running maximum with its sum rescaled whenever the maximum grows
// (or, for a greedy row, the running maximum and its lowest index).  The
// threads' states are merged once at the end.  kFull: the span is complete,
// so no vector needs a bounds check.  Exponent arguments and sums use the
// paired float instructions, two elements per instruction.
template <typename T, bool kGreedy, bool kFull>
__device__ __forceinline__ Partial span_partial_vec(const T* row, int beg, int end, float k) {
  using E = Elem<T>;
  constexpr int kVec = E::kVec;
  constexpr int kVecs = kSpanBytes / 16 / kThreads;  // vectors per thread
  constexpr int kGroups = kVecs / kGroup;
  __shared__ float red_f[kThreads / 32];
  __shared__ float red_g[kThreads / 32];
  __shared__ int red_i[kThreads / 32];
  const uint4* vp = reinterpret_cast<const uint4*>(row + beg);
  const int nv = kFull ? kVecs * kThreads : (end - beg) / kVec;
  const uint4 pad = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);

  uint4 buf[2][kGroup];
#pragma unroll
  for (int u = 0; u < kGroup; ++u) {
    const int v = threadIdx.x + u * kThreads;
    buf[0][u] = (kFull || v < nv) ? ld_stream16(vp + v) : pad;
  }
  float m = -INFINITY;      // running maximum (raw logits)
  float c = -INFINITY;      // fl(m k), the exponent reference of the sum
  uint64_t s2 = f2pack(0.f, 0.f);  // sum of 2^(x k - c), two lanes
  bool bad = false;         // a NaN / +inf / out-of-range maximum was seen
  int idx = INT_MAX;        // greedy: lowest index holding m
  const uint64_t k2 = f2pack(k, k);
#pragma unroll
  for (int gi = 0; gi < kGroups; ++gi) {
    const int cur = gi & 1;
    if (gi + 1 < kGroups) {
#pragma unroll
      for (int u = 0; u < kGroup; ++u) {
        const int v = threadIdx.x + ((gi + 1) * kGroup + u) * kThreads;
        buf[cur ^ 1][u] = (kFull || v < nv) ? ld_stream16(vp + v) : pad;
      }
    }
    float gm = E::vmax_nan(buf[cur][0]);
#pragma unroll
    for (int u = 1; u < kGroup; ++u) gm = fmax_nan(gm, E::vmax_nan(buf[cur][u]));
    if (gm != gm) bad = true;
    if (kGreedy) {
      if (gm > m) {  // strict: an equal value later in the row keeps the earlier index
        m = gm;
        idx = INT_MAX;
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
#pragma unroll
          for (int e = 0; e < kVec; ++e) {
            if (idx == INT_MAX && E::get(buf[cur][u], e) == gm)
              idx = beg + (threadIdx.x + (gi * kGroup + u) * kThreads) * kVec + e;
          }
        }
      }
    } else {
      if (gm > m) {
        const float cn = gm * k;
        if (gm == INFINITY || !(fabsf(cn) <= 3.40282347e38f)) bad = true;
        const float r = c > -INFINITY ? ex2(c - cn) : 0.f;
        s2 = f2mul(s2, f2pack(r, r));
        c = cn;
        m = gm;
      }
      if (m > -INFINITY && !bad) {
        const uint64_t nc2 = f2pack(-c, -c);
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
#pragma unroll
          for (int e = 0; e < E::kPairs; ++e) {
            float a0, a1;
            f2unpack(f2fma(E::pair(buf[cur][u], e), k2, nc2), a0, a1);
            s2 = f2add(s2, f2pack(ex2(a0), ex2(a1)));
          }
        }
      }
    }
  }
  Partial out;
  out.pad = 0;
  if (kGreedy) {
    const float best = block_max_nan(bad ? __int_as_float(0x7fc00000) : m, red_f);
    out.idx = block_min_int(m == best ? idx : INT_MAX, red_i);
    out.a = best;
    out.s = (best != best) ? __int_as_float(0x7fc00000) : 0.f;
  } else {
    float s_lo, s_hi;
    f2unpack(s2, s_lo, s_hi);
    const float s = s_lo + s_hi;
    // merge (c, s) over the CTA; any bad thread makes the span bad
    const float cmax = block_max_nan(bad ? __int_as_float(0x7fc00000) : c, red_f);
    float part = 0.f;
    if (cmax == cmax && cmax > -INFINITY && c > -INFINITY) part = s * ex2(c - cmax);
    const float tot = block_sum(part, red_g);
    out.a = cmax;
    out.s = (cmax != cmax) ? __int_as_float(0x7fc00000) : (cmax > -INFINITY ? tot : 0.f);
    out.idx = 0;
  }
  return out;
}

template <typename T, bool kVecPath>
__global__ void __launch_bounds__(kThreads, kSpanMinBlocks) rowstats_kernel(Problem p, Workspace w) {
  const int S1 = w.S1;
  const int per = 2 * p.N + 1;
  const int row = blockIdx.x / S1;
  const int span = blockIdx.x - row * S1;
  const int b = row / per;
  const int slot = row - b * per;
  const int mode = temp_mode(p.temperature[b]);
  if (mode == kModeInvalid || (mode == kModeGreedy && slot > p.N)) return;  // CTA-uniform
  const RowRef r = row_of(p, b, slot);
  const T* base = static_cast<const T*>(r.draft ? p.draft : p.target) + r.offset;
  constexpr int kSpan = kSpanBytes / static_cast<int>(sizeof(T));
  const int beg = span * kSpan;
  const int end = min(p.V, beg + kSpan);
  const bool greedy = mode == kModeGreedy;
  const float k = greedy ? 0.f : scale_of(p.temperature[b]);
  Partial out;
  if (!kVecPath) {
    out = chunk_partial_scalar<T>(base, beg, end, greedy, k);
  } else if (end - beg == kSpan) {
    out = greedy ? span_partial_vec<T, true, true>(base, beg, end, k)
                 : span_partial_vec<T, false, true>(base, beg, end, k);
  } else {
    out = greedy ? span_partial_vec<T, true, false>(base, beg, end, k)
                 : span_partial_vec<T, false, false>(base, beg, end, k);
  }
  if (threadIdx.x == 0) w.partials[static_cast<size_t>(row) * S1 + span] = out;
}

// ------------------------------------------------------------------ stream

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

// Running per-lane state of one row segment.
struct LaneState {
  float m;      // running maximum (raw logits)
  float c;      // fl(m k): exponent reference of the sum (sampled rows)
  uint64_t s2;  // sum of 2^(x k - c), two lanes of paired floats
  int idx;      // lowest index holding m (greedy rows)
  bool bad;     // NaN / +inf / out-of-range maximum seen
  float tok;    // logit at the draft token, if this lane read it
  bool has_tok;
};

// Fold one group of kGroup vectors (vector indices vfirst + 32u) into the
// lane state; vectors at or past vend hold -inf padding.
template <typename T, bool kGreedy>
__device__ __forceinline__ void fold_group(LaneState& st, const uint4 (&buf)[kGroup], int vfirst,
                                           int vend, float k, uint64_t k2, int d) {
  using E = Elem<T>;
  constexpr int kVec = E::kVec;
#pragma unroll
  for (int u = 0; u < kGroup; ++u) {
    const int v = vfirst + 32 * u;
    if (d >= v * kVec && d < v * kVec + kVec && v < vend) {
      st.tok = E::get(buf[u], d - v * kVec);
      st.has_tok = true;
    }
  }
  float gm = E::vmax_nan(buf[0]);
#pragma unroll
  for (int u = 1; u < kGroup; ++u) gm = fmax_nan(gm, E::vmax_nan(buf[u]));
  if (gm != gm) st.bad = true;
  if (kGreedy) {
    if (gm > st.m) {  // strict: a later equal value keeps the earlier index
      st.m = gm;
      st.idx = INT_MAX;
#pragma unroll
      for (int u = 0; u < kGroup; ++u) {
#pragma unroll
        for (int e = 0; e < kVec; ++e)
          if (st.idx == INT_MAX && E::get(buf[u], e) == gm) st.idx = (vfirst + 32 * u) * kVec + e;
      }
    }
  } else {
    if (gm > st.m) {
      const float cn = gm * k;
      if (gm == INFINITY || !(fabsf(cn) <= 3.40282347e38f)) st.bad = true;
      const float r = st.c > -INFINITY ? ex2(st.c - cn) : 0.f;
      st.s2 = f2mul(st.s2, f2pack(r, r));
      st.c = cn;
      st.m = gm;
    }
    if (st.m > -INFINITY && !st.bad) {
      const uint64_t nc2 = f2pack(-st.c, -st.c);
#pragma unroll
      for (int u = 0; u < kGroup; ++u) {
#pragma unroll
        for (int e = 0; e < E::kPairs; ++e) {
          float a0, a1;
          f2unpack(f2fma(E::pair(buf[u], e), k2, nc2), a0, a1);
          st.s2 = f2add(st.s2, f2pack(ex2(a0), ex2(a1)));
        }
      }
    }
  }
}

constexpr int kWarpRingVecs = kStreamStages * kGroup * 32;  // 16-byte slots per warp
constexpr int kStreamSmem = (kThreads / 32) * kWarpRingVecs * 16;

// One warp reduces vectors [v0, v1) of one row (16-byte vector indices) and
// writes the partial to `slot`; the lane that reads the draft token's logit
// stores it to *tok_out.  Loads go through the warp's ring of kStreamStages
// groups in shared memory (cp.async), kStreamStages - 1 groups in flight.
template <typename T, bool kGreedy>
__device__ void stream_segment(const T* row, int v0, int v1, float k, int d, uint4* ring,
                               Partial* slot, float* tok_out) {
  using E = Elem<T>;
  constexpr int kStep = 32 * kGroup;
  const int lane = threadIdx.x & 31;
  const uint4* rowv = reinterpret_cast<const uint4*>(row);
  const uint4 pad = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
  LaneState st;
  st.m = -INFINITY;
  st.c = -INFINITY;
  st.s2 = f2pack(0.f, 0.f);
  st.idx = INT_MAX;
  st.bad = false;
  st.tok = 0.f;
  st.has_tok = false;
  const uint64_t k2 = f2pack(k, k);
  const int groups = (v1 - v0 + kStep - 1) / kStep;
  const int vlane = v0 + lane;
  // group g -> stage g % kStreamStages; every issue commits one (maybe empty)
  // group so that wait_group counts stay aligned with g
  auto issue = [&](int g) {
    if (g < groups) {
      uint4* stage = ring + (g % kStreamStages) * kGroup * 32 + lane;
#pragma unroll
      for (int u = 0; u < kGroup; ++u) {
        const int v = vlane + g * kStep + 32 * u;
        if (v < v1) cp_async16(smem_u32(stage + 32 * u), rowv + v);
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int g = 0; g < kStreamStages - 1; ++g) issue(g);
  for (int g = 0; g < groups; ++g) {
    issue(g + kStreamStages - 1);
    cp_async_wait<kStreamStages - 1>();
    const uint4* stage = ring + (g % kStreamStages) * kGroup * 32 + lane;
    const int vfirst = vlane + g * kStep;
    uint4 buf[kGroup];
#pragma unroll
    for (int u = 0; u < kGroup; ++u) buf[u] = vfirst + 32 * u < v1 ? stage[32 * u] : pad;
    fold_group<T, kGreedy>(st, buf, vfirst, v1, k, k2, d);
  }
  cp_async_wait<0>();
  if (st.has_tok) *tok_out = st.tok;
  Partial out;
  out.pad = 0;
  if (kGreedy) {
    const float best = warp_max_nan(st.bad ? __int_as_float(0x7fc00000) : st.m);
    out.idx = warp_min_int(st.m == best ? st.idx : INT_MAX);
    out.a = best;
    out.s = (best != best) ? __int_as_float(0x7fc00000) : 0.f;
  } else {
    float s_lo, s_hi;
    f2unpack(st.s2, s_lo, s_hi);
    const float cmax = warp_max_nan(st.bad ? __int_as_float(0x7fc00000) : st.c);
    float part = 0.f;
    if (cmax == cmax && cmax > -INFINITY && st.c > -INFINITY) part = (s_lo + s_hi) * ex2(st.c - cmax);
    const float tot = warp_sum(part);
    out.a = cmax;
    out.s = (cmax != cmax) ? __int_as_float(0x7fc00000) : (cmax > -INFINITY ? tot : 0.f);
    out.idx = 0;
  }
  if (lane == 0) *slot = out;
}

// Chunks a request contributes to the stream: its rows that are read.
__device__ __forceinline__ unsigned request_rows(int mode, int N) {
  if (mode == kModeInvalid) return 0u;
  return mode == kModeGreedy ? static_cast<unsigned>(N + 1) : static_cast<unsigned>(2 * N + 1);
}

template <typename T>
__global__ void __launch_bounds__(kThreads, kStreamCtasPerSm) rowstats_stream_kernel(Problem p,
                                                                                    Workspace w) {
  extern __shared__ __align__(16) uint4 stream_ring[];
  __shared__ unsigned rows_before[kStreamMaxB + 1];
  __shared__ unsigned char modes[kStreamMaxB];
  __shared__ unsigned scan_scratch[kThreads / 32];
  const int B = p.B, N = p.N;
  uint4* ring = stream_ring + (threadIdx.x >> 5) * kWarpRingVecs;

  // Active rows per request and their exclusive prefix (same in every CTA).
  const int per_thread = (B + kThreads - 1) / kThreads;
  const int b0 = threadIdx.x * per_thread;
  unsigned local = 0;
  for (int i = 0; i < per_thread; ++i) {
    const int b = b0 + i;
    if (b < B) {
      const int mode = temp_mode(p.temperature[b]);
      modes[b] = static_cast<unsigned char>(mode);
      local += request_rows(mode, N);
    }
  }
  unsigned total_rows;
  unsigned run = block_exclusive_scan_u32(local, scan_scratch, &total_rows);
  for (int i = 0; i < per_thread; ++i) {
    const int b = b0 + i;
    if (b < B) {
      rows_before[b] = run;
      if (blockIdx.x == 0) w.row_prefix[b] = run;
      run += request_rows(modes[b], N);
    }
  }
  if (threadIdx.x == 0) {
    rows_before[B] = total_rows;
    if (blockIdx.x == 0) w.row_prefix[B] = total_rows;
  }
  __syncthreads();

  using E = Elem<T>;
  const unsigned long long row_bytes = static_cast<unsigned long long>(p.V) * sizeof(T);
  const unsigned long long total = static_cast<unsigned long long>(total_rows) * row_bytes;
  const unsigned long long warps = static_cast<unsigned long long>(gridDim.x) * (kThreads / 32);
  const unsigned long long rb = stream_range_bytes(total, row_bytes, warps);
  const unsigned long long ranges = (total + rb - 1) / rb;
  const int per = 2 * N + 1;
  int cursor = 0;
  for (unsigned long long rho = static_cast<unsigned long long>(blockIdx.x) * (kThreads / 32) +
                                (threadIdx.x >> 5);
       rho < ranges; rho += warps) {
    const unsigned long long start = rho * rb;
    const unsigned long long end = start + rb < total ? start + rb : total;
    unsigned long long q = start / row_bytes;
    unsigned long long off = start - q * row_bytes;
    for (int part = 0; part < 2; ++part) {
      const unsigned long long row_end = (q + 1) * row_bytes;
      const unsigned long long seg_end = end < row_end ? end : row_end;
      if (q * row_bytes + off >= seg_end) break;
      while (rows_before[cursor + 1] <= q) ++cursor;
      const int b = cursor;
      const int slot = static_cast<int>(q - rows_before[b]);
      const bool greedy = modes[b] == kModeGreedy;
      const RowRef r = row_of(p, b, slot);
      const T* row = static_cast<const T*>(r.draft ? p.draft : p.target) + r.offset;
      const int d = (!greedy && slot != N) ? p.tokens[static_cast<size_t>(b) * N + (slot <= N ? slot : slot - N - 1)]
                                           : -1;
      const int v0 = static_cast<int>(off / 16);
      const int v1 = static_cast<int>((seg_end - q * row_bytes) / 16);
      Partial* dst = w.partials + 2 * rho + part;
      float* tok = w.tok_logit + static_cast<size_t>(b) * per + slot;
      if (greedy)
        stream_segment<T, true>(row, v0, v1, 0.f, -1, ring, dst, tok);
      else
        stream_segment<T, false>(row, v0, v1, scale_of(p.temperature[b]), d, ring, dst, tok);
      ++q;
      off = 0;
    }
  }
  (void)sizeof(E);
}

}  // namespace

cudaError_t prepare_rowstats() {
  cudaError_t e = cudaFuncSetAttribute(rowstats_stream_kernel<__nv_bfloat16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kStreamSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(rowstats_stream_kernel<float>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kStreamSmem);
}

cudaError_t launch_rowstats(int dtype, bool vec, const Problem& p, const Workspace& w,
                            cudaStream_t s) {
  if (w.layout == kLayoutStream) {
    if (!vec || p.B > kStreamMaxB || w.stream_warps % (kThreads / 32) != 0)
      return cudaErrorInvalidValue;
    const unsigned grid = static_cast<unsigned>(w.stream_warps / (kThreads / 32));
    if (dtype == 1)
      rowstats_stream_kernel<__nv_bfloat16><<<grid, kThreads, kStreamSmem, s>>>(p, w);
    else
      rowstats_stream_kernel<float><<<grid, kThreads, kStreamSmem, s>>>(p, w);
    return cudaGetLastError();
  }
  const long long blocks = static_cast<long long>(p.B) * (2 * p.N + 1) * w.S1;
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
