// Statistics of one span of one logit row, shared by the chain and tree
// row-statistics kernels (see sv_rowstats.cu for the method and the grid).
// One CTA of kThreads threads reduces the span [beg, end) of a row: for a
// sampled row to (c, s) with c = fl(M k), M the span maximum, k = log2(e)/T,
// s = sum_t 2^(x_t k - c); for a greedy row to the maximum and the lowest
// index holding it.  The thread whose vector holds token d (if d is in the
// span) stores x_d at *tok_out.
#pragma once

#include <climits>
#include <cuda_bf16.h>

#include "sv_device.cuh"

namespace sv {
namespace {

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
  out.tag = 0;
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
// kSmem: `row` + beg points to a copy of the span staged in shared memory
// (plain loads) instead of global memory (streaming loads); the arithmetic
// is the same either way.
template <typename T, bool kGreedy, bool kFull, bool kSmem = false>
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
    buf[0][u] = (kFull || v < nv) ? (kSmem ? vp[v] : ld_stream16(vp + v)) : pad;
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
        buf[cur ^ 1][u] = (kFull || v < nv) ? (kSmem ? vp[v] : ld_stream16(vp + v)) : pad;
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
  out.tag = 0;
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

}  // namespace
}  // namespace sv
