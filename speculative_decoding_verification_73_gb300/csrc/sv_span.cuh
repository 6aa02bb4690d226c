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
// reads 16-byte vectors t, t + kThreads, ... of the span in groups of kGroup
// and keeps a running maximum with its sum rescaled whenever the maximum
// grows (or, for a greedy row, the running maximum and its lowest index).
// The threads' states are merged once at the end.  Exponent arguments and
// sums use the paired float instructions, two elements per instruction.
// The per-thread state, the per-group update and the final merge are
// written out separately below, so that the order of operations that every
// span partial depends on reads in one place.

struct SpanAcc {
  float m;      // running maximum (raw logits)
  float c;      // fl(m k), the exponent reference of the sum
  uint64_t s2;  // sum of 2^(x k - c), two lanes
  bool bad;     // a NaN / +inf / out-of-range maximum was seen
  int idx;      // greedy: lowest index holding m
};

__device__ __forceinline__ SpanAcc span_acc_init() {
  SpanAcc a;
  a.m = -INFINITY;
  a.c = -INFINITY;
  a.s2 = f2pack(0.f, 0.f);
  a.bad = false;
  a.idx = INT_MAX;
  return a;
}

// Where the draft token d sits among this thread's vectors of the span
// [beg, end): group gi, vector u of the group, element e (gi = -1 if this
// thread does not hold it), worked out once per span.
struct TokAt {
  int gi, u, e;
};

template <typename T>
__device__ __forceinline__ TokAt tok_at(int beg, int end, int d) {
  constexpr int kVec = Elem<T>::kVec;
  TokAt t{-1, 0, 0};
  if (d >= beg && d < end) {
    const int r = d - beg;
    const int v = r / kVec;
    if (v % kThreads == static_cast<int>(threadIdx.x)) {
      const int i = v / kThreads;
      t.gi = i / kGroup;
      t.u = i - t.gi * kGroup;
      t.e = r - v * kVec;
    }
  }
  return t;
}

// Fold group gi of this thread's vectors (vector i of the group is span
// vector threadIdx.x + (gi kGroup + i) kThreads) into the state.  A vector
// past the span's end must hold -inf words.  The thread whose vector holds
// the draft token (ta, from tok_at) stores its logit at *tok_out.
template <typename T, bool kGreedy>
__device__ __forceinline__ void span_group(SpanAcc& a, const uint4 (&g)[kGroup], int beg, int gi, uint64_t k2,
                                           float k, const TokAt& ta, float* tok_out) {
  using E = Elem<T>;
  constexpr int kVec = E::kVec;
  if (!kGreedy && gi == ta.gi) {
    uint4 v = g[0];
#pragma unroll
    for (int u = 1; u < kGroup; ++u)
      if (u == ta.u) v = g[u];
    *tok_out = E::get(v, ta.e);
  }
  float gm = E::vmax_nan(g[0]);
#pragma unroll
  for (int u = 1; u < kGroup; ++u) gm = fmax_nan(gm, E::vmax_nan(g[u]));
  if (gm != gm) a.bad = true;
  if (kGreedy) {
    if (gm > a.m) {  // strict: an equal value later in the row keeps the earlier index
      a.m = gm;
      a.idx = INT_MAX;
#pragma unroll
      for (int u = 0; u < kGroup; ++u) {
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
          if (a.idx == INT_MAX && E::get(g[u], e) == gm)
            a.idx = beg + (static_cast<int>(threadIdx.x) + (gi * kGroup + u) * kThreads) * kVec + e;
        }
      }
    }
  } else {
    if (gm > a.m) {
      const float cn = gm * k;
      if (gm == INFINITY || !(fabsf(cn) <= 3.40282347e38f)) a.bad = true;
      const float r = a.c > -INFINITY ? ex2(a.c - cn) : 0.f;
      a.s2 = f2mul(a.s2, f2pack(r, r));
      a.c = cn;
      a.m = gm;
    }
    if (a.m > -INFINITY && !a.bad) {
      const uint64_t nc2 = f2pack(-a.c, -a.c);
#pragma unroll
      for (int u = 0; u < kGroup; ++u) {
#pragma unroll
        for (int e = 0; e < E::kPairs; ++e) {
          float a0, a1;
          f2unpack(f2fma(E::pair(g[u], e), k2, nc2), a0, a1);
          a.s2 = f2add(a.s2, f2pack(ex2(a0), ex2(a1)));
        }
      }
    }
  }
}

// Merge the threads' states into the span's partial (every thread of the
// CTA gets it).  red_f, red_g, red_i: kThreads/32 slots each.
template <bool kGreedy>
__device__ __forceinline__ Partial span_finish(const SpanAcc& a, float* red_f, float* red_g, int* red_i) {
  Partial out;
  out.tag = 0;
  if (kGreedy) {
    const float best = block_max_nan(a.bad ? __int_as_float(0x7fc00000) : a.m, red_f);
    out.idx = block_min_int(a.m == best ? a.idx : INT_MAX, red_i);
    out.a = best;
    out.s = (best != best) ? __int_as_float(0x7fc00000) : 0.f;
  } else {
    float s_lo, s_hi;
    f2unpack(a.s2, s_lo, s_hi);
    const float s = s_lo + s_hi;
    // merge (c, s) over the CTA; any bad thread makes the span bad
    const float cmax = block_max_nan(a.bad ? __int_as_float(0x7fc00000) : a.c, red_f);
    float part = 0.f;
    if (cmax == cmax && cmax > -INFINITY && a.c > -INFINITY) part = s * ex2(a.c - cmax);
    const float tot = block_sum(part, red_g);
    out.a = cmax;
    out.s = (cmax != cmax) ? __int_as_float(0x7fc00000) : (cmax > -INFINITY ? tot : 0.f);
    out.idx = 0;
  }
  return out;
}

// The span [beg, end) of a row, read from global memory (the next group's
// loads issued before the current group is reduced) or, kSmem, from a copy
// staged in shared memory at `row` + beg (plain loads).  kFull: the span is
// complete, so no vector needs a bounds check.
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
  SpanAcc acc = span_acc_init();
  const uint64_t k2 = f2pack(k, k);
  const TokAt ta = kGreedy ? TokAt{-1, 0, 0} : tok_at<T>(beg, end, d);
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
    span_group<T, kGreedy>(acc, buf[cur], beg, gi, k2, k, ta, tok_out);
  }
  return span_finish<kGreedy>(acc, red_f, red_g, red_i);
}

// The span [beg, end) of a row read through a ring in shared memory: each
// thread fetches its own vectors with cp.async into its own slots kDepth
// groups ahead of the group it reduces, so more of the span is in flight
// than registers would hold (a thread reads only slots it filled itself,
// after its own cp.async.wait_group: no CTA barrier).  `ring` holds
// kDepth * kGroup * kThreads vectors.  The same partial as span_partial_vec
// (same vectors per thread, same groups, same order).
template <int kDepth>
constexpr int span_ring_bytes() {
  return kDepth * kGroup * kThreads * 16;
}
template <typename T, bool kGreedy, bool kFull, int kDepth>
__device__ __forceinline__ Partial span_partial_ring(const T* row, int beg, int end, float k, int d,
                                                     float* tok_out, uint4* ring) {
  using E = Elem<T>;
  constexpr int kVecs = kSpanBytes / 16 / kThreads;  // vectors per thread
  constexpr int kGroups = kVecs / kGroup;
  static_assert(kDepth >= 1 && kDepth <= 3 && kDepth <= kGroups, "ring depth");
  __shared__ float red_f[kThreads / 32];
  __shared__ float red_g[kThreads / 32];
  __shared__ int red_i[kThreads / 32];
  const uint4* vp = reinterpret_cast<const uint4*>(row + beg);
  const int nv = kFull ? kVecs * kThreads : (end - beg) / E::kVec;
  const uint4 pad = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
  auto slot = [&](int gi, int u) { return ring + ((gi % kDepth) * kGroup + u) * kThreads + threadIdx.x; };
  auto issue = [&](int gi) {
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
      const int v = threadIdx.x + (gi * kGroup + u) * kThreads;
      if (kFull || v < nv)
        cp_async16(slot(gi, u), vp + v);
      else
        *slot(gi, u) = pad;
    }
    cp_async_commit();
  };
#pragma unroll
  for (int gi = 0; gi < kDepth; ++gi) issue(gi);
  SpanAcc acc = span_acc_init();
  const uint64_t k2 = f2pack(k, k);
  const TokAt ta = kGreedy ? TokAt{-1, 0, 0} : tok_at<T>(beg, end, d);
#pragma unroll
  for (int gi = 0; gi < kGroups; ++gi) {
    cp_async_wait_group<kDepth - 1>();  // this thread's copies of group gi have landed
    uint4 g[kGroup];
#pragma unroll
    for (int u = 0; u < kGroup; ++u) g[u] = *slot(gi, u);
    if (gi + kDepth < kGroups)
      issue(gi + kDepth);  // into the slot just read
    else
      cp_async_commit();  // an empty group keeps the count of groups in step
    span_group<T, kGreedy>(acc, g, beg, gi, k2, k, ta, tok_out);
  }
  return span_finish<kGreedy>(acc, red_f, red_g, red_i);
}

}  // namespace
}  // namespace sv
