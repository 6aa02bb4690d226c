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
// one CTA-wide merge per span) and writes partials[row][span].  The CTA
// whose span holds the row's draft token also stores that token's logit, so
// the walk never reads the logits again.  Rows that are not 16-byte aligned
// take a scalar two-pass path over the same spans.  Small per-thread state
// and groups of two loads keep eight CTAs resident per SM, which measured
// best (more warps in flight, fewer registers per byte in flight).

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
__device__ Partial chunk_partial_scalar(const T* row, int beg, int end, bool greedy, float k, int d,
                                        float* tok_out) {
  using E = Elem<T>;
  if (threadIdx.x == 0 && !greedy && d >= beg && d < end) *tok_out = E::load1(row + d);
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
__device__ __forceinline__ Partial span_partial_vec(const T* row, int beg, int end, float k, int d,
                                                    float* tok_out) {
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
    if (!kGreedy) {
      // the thread whose vector holds the draft token stores its logit
#pragma unroll
      for (int u = 0; u < kGroup; ++u) {
        const int e0 = beg + (threadIdx.x + (gi * kGroup + u) * kThreads) * kVec;
        if (d >= e0 && d < e0 + kVec && (kFull || d < end)) *tok_out = E::get(buf[cur][u], d - e0);
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
  allow_dependents();  // the sampler may be scheduled behind the last wave
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
  // draft token of a sampled row (none for the bonus row, slot N); its logit
  // is captured in the same pass for the walk
  const int j = slot <= p.N ? slot : slot - p.N - 1;
  const int d = (!greedy && slot != p.N) ? p.tokens[static_cast<size_t>(b) * p.N + j] : -1;
  float* tok = w.tok_logit + row;
  Partial out;
  if (!kVecPath) {
    out = chunk_partial_scalar<T>(base, beg, end, greedy, k, d, tok);
  } else if (end - beg == kSpan) {
    out = greedy ? span_partial_vec<T, true, true>(base, beg, end, k, -1, tok)
                 : span_partial_vec<T, false, true>(base, beg, end, k, d, tok);
  } else {
    out = greedy ? span_partial_vec<T, true, false>(base, beg, end, k, -1, tok)
                 : span_partial_vec<T, false, false>(base, beg, end, k, d, tok);
  }
  if (threadIdx.x == 0) w.partials[static_cast<size_t>(row) * S1 + span] = out;
}

template <typename T, bool kVecPath>
cudaError_t launch_rowstats_t(const Problem& p, const Workspace& w, cudaStream_t s) {
  const long long blocks = static_cast<long long>(p.B) * (2 * p.N + 1) * w.S1;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  rowstats_kernel<T, kVecPath><<<dim3(static_cast<unsigned>(blocks)), kThreads, 0, s>>>(p, w);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rowstats(int dtype, bool vec, const Problem& p, const Workspace& w,
                            cudaStream_t s) {
  if (dtype == 1)
    return vec ? launch_rowstats_t<__nv_bfloat16, true>(p, w, s)
               : launch_rowstats_t<__nv_bfloat16, false>(p, w, s);
  return vec ? launch_rowstats_t<float, true>(p, w, s) : launch_rowstats_t<float, false>(p, w, s);
}

}  // namespace sv
