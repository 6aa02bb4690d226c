// The accept/reject walk of one request, run by each sampler CTA of the
// request (see sv_sample.cu); thread j handles row j.  Every CTA of a request
// computes the same result from the row-statistics partials; only the one
// asked to (write_outputs) stores the outputs.
//
// Thread j merges the row-statistics partials of target row j (and, for a
// sampled request, draft row j), checks the inputs, and evaluates position
// j+1 of the chain.  The partials are polled by their tags (below), so a
// request's walk starts as soon as its own rows are reduced.  "Speculative Decoding and EAGLE-3" lesson:
//   * "Build it", step 1: a draft with p(d) = 0 is accepted; otherwise it is
//     accepted iff u < min(1, q(d) / p(d));
//   * "Invariant: Leviathan rejection sampling": the walk goes left to right
//     and stops at the first rejection; if all N are accepted a bonus token
//     comes from q_{N+1};
//   * "KV cache rollback" / "Build it" step 4: the committed KV length stops
//     right after the correction token, i.e. accepted + 1 entries of this
//     window.
// Greedy requests (T = 0) accept d_j iff it equals the argmax of target row
// j; the emitted token after the prefix is the argmax of the next row.
//
// All arithmetic is float32 (double-precision transcendentals are very slow
// on this part).  The acceptance ratio is formed as
//   log2(q(d)/p(d)) = (z_d - y_d) k - (c_q - c_p) + log2(s_p / s_q),
// so every term stays small when q(d) and p(d) are close.  The correction /
// bonus token of a sampled request is left to the sampler as a Job.
#pragma once

#include <climits>

#include "sv_device.cuh"

namespace sv {

// log2 sum_t 2^(x_t k) = c + log2(s)
struct RowNorm {
  float c;
  float s;
  bool ok;
};

// The first kPre partials of every row are loaded together with the walk's
// other inputs (one L2 round trip for V up to kPre spans); any further ones
// kBatch at a time, every load of a batch issued before any is used.
constexpr int kPre = 4;
constexpr int kBatch = 8;

// A partial, or an empty one (maximum -inf, nothing summed) when !take.
__device__ __forceinline__ float4 partial_or_empty(const Partial* at, bool take) {
  return take ? __ldcg(reinterpret_cast<const float4*>(at))
              : make_float4(-INFINITY, 0.f, __int_as_float(INT_MAX), 0.f);
}

template <int kN>
__device__ __forceinline__ void absorb_sampled(const float4 (&pt)[kN], float& c, float& s, bool& bad) {
  float cb = c;
#pragma unroll
  for (int i = 0; i < kN; ++i) {
    if (pt[i].y != pt[i].y || pt[i].x != pt[i].x) bad = true;
    cb = fmaxf(cb, pt[i].x);
  }
  if (cb > -INFINITY) {
    float sb = c > -INFINITY ? s * exp2f(c - cb) : 0.f;
#pragma unroll
    for (int i = 0; i < kN; ++i)
      if (pt[i].x > -INFINITY) sb += pt[i].y * exp2f(pt[i].x - cb);
    s = sb;
    c = cb;
  }
}

// Merge the n partials of a sampled row; `pre` holds the first kPre and
// load(i0, pt) fetches the kBatch partials from index i0 on (empty past n).
template <class Load>
__device__ __forceinline__ RowNorm merge_sampled_by(const float4 (&pre)[kPre], int n, Load load) {
  float c = -INFINITY, s = 0.f;
  bool bad = false;
  absorb_sampled(pre, c, s, bad);
  for (int i0 = kPre; i0 < n; i0 += kBatch) {
    float4 pt[kBatch];
    load(i0, pt);
    absorb_sampled(pt, c, s, bad);
  }
  RowNorm r;
  r.c = c;
  r.s = s;
  r.ok = !bad && c > -INFINITY && c < INFINITY && s > 0.f && s < INFINITY;
  return r;
}

// The same with plain loads (partials written by a kernel that has ended).
__device__ __forceinline__ RowNorm merge_sampled(const float4 (&pre)[kPre], const Partial* parts,
                                                 int n) {
  return merge_sampled_by(pre, n, [&](int i0, float4(&pt)[kBatch]) {
#pragma unroll
    for (int i = 0; i < kBatch; ++i) pt[i] = partial_or_empty(parts + i0 + i, i0 + i < n);
  });
}

struct RowMax {
  int idx;
  bool ok;
};

template <int kN>
__device__ __forceinline__ void absorb_greedy(const float4 (&pt)[kN], float& best, int& idx,
                                              bool& bad) {
#pragma unroll
  for (int i = 0; i < kN; ++i) {
    if (pt[i].y != pt[i].y || pt[i].x != pt[i].x) bad = true;
    if (pt[i].x > best) {
      best = pt[i].x;
      idx = __float_as_int(pt[i].z);
    }
  }
}

// Greedy rows: partials come in increasing index order, so strict > keeps
// the lowest index among equal maxima.
template <class Load>
__device__ __forceinline__ RowMax merge_greedy_by(const float4 (&pre)[kPre], int n, Load load) {
  float best = -INFINITY;
  int idx = INT_MAX;
  bool bad = false;
  absorb_greedy(pre, best, idx, bad);
  for (int i0 = kPre; i0 < n; i0 += kBatch) {
    float4 pt[kBatch];
    load(i0, pt);
    absorb_greedy(pt, best, idx, bad);
  }
  RowMax r;
  r.idx = idx;
  r.ok = !bad && best > -INFINITY && best < INFINITY;
  return r;
}

__device__ __forceinline__ RowMax merge_greedy(const float4 (&pre)[kPre], const Partial* parts, int n) {
  return merge_greedy_by(pre, n, [&](int i0, float4(&pt)[kBatch]) {
#pragma unroll
    for (int i = 0; i < kBatch; ++i) pt[i] = partial_or_empty(parts + i0 + i, i0 + i < n);
  });
}

// The same merges over partials gathered into this CTA's shared memory
// (plain loads; the merge arithmetic is the same).
__device__ __forceinline__ float4 partial_local(const Partial* at, bool take) {
  return take ? *reinterpret_cast<const float4*>(at) : make_float4(-INFINITY, 0.f, __int_as_float(INT_MAX), 0.f);
}

__device__ __forceinline__ RowNorm merge_row_local(const Partial* parts, int n) {
  float4 pre[kPre];
#pragma unroll
  for (int i = 0; i < kPre; ++i) pre[i] = partial_local(parts + i, i < n);
  return merge_sampled_by(pre, n, [&](int i0, float4(&pt)[kBatch]) {
#pragma unroll
    for (int i = 0; i < kBatch; ++i) pt[i] = partial_local(parts + i0 + i, i0 + i < n);
  });
}

__device__ __forceinline__ RowMax merge_row_greedy_local(const Partial* parts, int n) {
  float4 pre[kPre];
#pragma unroll
  for (int i = 0; i < kPre; ++i) pre[i] = partial_local(parts + i, i < n);
  return merge_greedy_by(pre, n, [&](int i0, float4(&pt)[kBatch]) {
#pragma unroll
    for (int i = 0; i < kBatch; ++i) pt[i] = partial_local(parts + i0 + i, i0 + i < n);
  });
}

// ------------------------------------------------------- tagged partials
// The chain sampler does not wait for the row-statistics grid to end: each
// partial it needs is read with a relaxed 128-bit load and used once its tag
// is this call's sequence number.  A partial not yet written is polled again
// after a short sleep; a thread gives up after kPollLimit polls (about a
// second), which only a stalled row-statistics grid could cause, and its
// request is then reported with kErrWait.
constexpr int kPollLimit = 1 << 20;

struct Poll {
  unsigned epoch;
  int budget;
  bool late;  // a partial never showed this call's tag
};

__device__ __forceinline__ bool tagged(const float4& v, unsigned epoch) { return __float_as_uint(v.w) == epoch; }

// Settle the partials a[i] (from pa + i) for i < na and b[i] (from pb + i)
// for i < nb, whose first loads are already issued: every round sleeps
// briefly and re-issues the loads of all those still untagged before it
// looks at any of them, so a row's spans are waited for together, not one
// after another.
template <int kN>
__device__ __forceinline__ void settle(float4 (&a)[kN], const Partial* pa, int na, float4 (&b)[kN],
                                       const Partial* pb, int nb, Poll& pl) {
  auto pending = [&]() {
    bool any = false;
#pragma unroll
    for (int i = 0; i < kN; ++i) {
      any |= i < na && !tagged(a[i], pl.epoch);
      any |= i < nb && !tagged(b[i], pl.epoch);
    }
    return any;
  };
  while (pending() && pl.budget > 0) {
    --pl.budget;
    __nanosleep(100);
#pragma unroll
    for (int i = 0; i < kN; ++i) {
      if (i < na && !tagged(a[i], pl.epoch)) a[i] = ld_partial_relaxed(pa + i);
      if (i < nb && !tagged(b[i], pl.epoch)) b[i] = ld_partial_relaxed(pb + i);
    }
  }
  if (pending()) pl.late = true;
}

// The same for one array.
template <int kN>
__device__ __forceinline__ void settle(float4 (&a)[kN], const Partial* pa, int na, Poll& pl) {
  float4 none[kN];
  settle(a, pa, na, none, pa, 0, pl);
}

// Batch loader for merge_*_by: every load issued, then the batch settled.
struct TaggedLoad {
  const Partial* parts;
  int n;
  Poll* pl;
  __device__ __forceinline__ void operator()(int i0, float4 (&pt)[kBatch]) const {
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
      pt[i] = i0 + i < n ? ld_partial_relaxed(parts + i0 + i)
                         : make_float4(-INFINITY, 0.f, __int_as_float(INT_MAX), 0.f);
    settle(pt, parts + i0, n - i0, *pl);
  }
};

// force_late: the test hook that makes this CTA act as if its waits ran out.
template <typename T>
__device__ __forceinline__ void walk_request(const Problem& p, const Workspace& w, int b,
                                             bool write_outputs, Job* job_out,
                                             bool force_late = false) {
  const int j = threadIdx.x;
  const int N = p.N, V = p.V;
  const bool row_thread = j <= N;
  const bool pos_thread = j < N;

  __shared__ int s_bad_token, s_bad_logit, s_first, s_late;

  // The inputs first (temperature, draft token), then every partial of the
  // request's rows that this thread merges, all loads issued before any is
  // used; a partial whose tag is not yet this call's is polled until it is.
  // (the partial loads go out before the temperature is back, so the
  // request's mode costs no extra round trip; loads a mode does not need
  // are never settled or used)
  const float t = p.temperature[b];
  const int d = pos_thread ? p.tokens[static_cast<size_t>(b) * N + j] : -1;
  const int S1 = w.S1;
  const Partial* req_parts = w.partials + static_cast<size_t>(b) * (2 * N + 1) * S1;
  const Partial* tparts = req_parts + static_cast<size_t>(j) * S1;
  const Partial* dparts = req_parts + static_cast<size_t>(N + 1 + j) * S1;
  const float4 empty = make_float4(-INFINITY, 0.f, __int_as_float(INT_MAX), 0.f);
  float4 tpre[kPre], dpre[kPre];
#pragma unroll
  for (int i = 0; i < kPre; ++i) {
    tpre[i] = (row_thread && i < S1) ? ld_partial_relaxed(tparts + i) : empty;
    dpre[i] = (pos_thread && i < S1) ? ld_partial_relaxed(dparts + i) : empty;
  }
  const int mode = temp_mode(t);
  if (!write_outputs && mode != kModeSampled) {  // CTA-uniform: nothing to sample
    if (j == 0) job_out->kind = kJobNone;
    return;
  }
  const bool take_t = row_thread && mode != kModeInvalid;
  const bool take_d = pos_thread && mode == kModeSampled;
  if (j == 0) {
    s_bad_token = 0;
    s_bad_logit = 0;
    s_first = N;
    s_late = 0;
  }
  Poll pl{p.epoch, kPollLimit, false};
  settle(tpre, tparts, take_t ? S1 : 0, dpre, dparts, take_d ? S1 : 0, pl);
  // The logits at d_j in target row j and draft row j: the row-statistics
  // CTA of the span holding d_j put them in that span's partial.
  float zd = 0.f, yd = 0.f;
  if (take_d && d >= 0 && d < V) {
    constexpr int kSpanElems = kSpanBytes / static_cast<int>(sizeof(T));
    const int sp = d / kSpanElems;
    if (sp < kPre) {
#pragma unroll
      for (int i = 0; i < kPre; ++i) {
        if (i == sp) {
          zd = tpre[i].z;
          yd = dpre[i].z;
        }
      }
    } else {
      float4 zt[1] = {ld_partial_relaxed(tparts + sp)}, yt[1] = {ld_partial_relaxed(dparts + sp)};
      settle(zt, tparts + sp, 1, yt, dparts + sp, 1, pl);
      zd = zt[0].z;
      yd = yt[0].z;
    }
  }
  __syncthreads();
  if (pos_thread && (d < 0 || d >= V)) atomicOr(&s_bad_token, 1);
  RowNorm q{}, pn{};
  RowMax g{};
  if (mode == kModeGreedy && row_thread) {
    g = merge_greedy_by(tpre, S1, TaggedLoad{tparts, S1, &pl});
    if (!g.ok) atomicOr(&s_bad_logit, 1);
  } else if (mode == kModeSampled && row_thread) {
    q = merge_sampled_by(tpre, S1, TaggedLoad{tparts, S1, &pl});
    if (!q.ok) atomicOr(&s_bad_logit, 1);
    if (pos_thread) {
      pn = merge_sampled_by(dpre, S1, TaggedLoad{dparts, S1, &pl});
      if (!pn.ok) atomicOr(&s_bad_logit, 1);
    }
  }
  if (pl.late || force_late) atomicOr(&s_late, 1);
  __syncthreads();

  // checks of the inputs first; a wait that ran out comes before the logit
  // check, whose partials it leaves unread
  unsigned err = 0;
  if (mode == kModeInvalid)
    err = kErrTemp;
  else if (s_bad_token)
    err = kErrToken;
  else if (s_late)
    err = kErrWait;
  else if (s_bad_logit)
    err = kErrLogit;

  int32_t* out_tok = p.out_tokens + static_cast<size_t>(b) * (N + 1);
  float* dbg_acc = w.dbg_accept + static_cast<size_t>(b) * N;
  float* dbg_lz = w.dbg_logz + static_cast<size_t>(b) * (2 * N + 1);
  const float qnan = __int_as_float(0x7fc00000);
  constexpr float kLn2 = 0.693147180559945309f;

  if (err || mode == kModeGreedy) {
    int a = -1;
    if (!err) {
      if (pos_thread && d != g.idx) atomicMin(&s_first, j);
      __syncthreads();
      a = s_first;
    }
    if (write_outputs) {
      if (row_thread) {
        out_tok[j] = (!err && j <= a) ? g.idx : -1;
        dbg_lz[j] = qnan;
        if (pos_thread) {
          dbg_acc[j] = qnan;
          dbg_lz[N + 1 + j] = qnan;
        }
      }
      if (j == 0) {
        p.out_accept[b] = err ? -1 : a;
        p.out_kv[b] = err ? 0 : a + 1;
        if (err) atomicOr(w.err, err);
      }
    }
    // every sampler CTA of a sampled request counts in, whatever stopped it
    // (see sv_sample.cu): a wait that ran out is this CTA's alone, so the
    // request's other CTAs may have reached the logit check instead
    if (j == 0)
      job_out->kind = mode != kModeSampled ? kJobNone : (err == kErrWait ? kJobLate : kJobFailed);
    return;
  }

  // Sampled request.
  const float k = scale_of(t);
  if (pos_thread) {
    float thr = 1.f;
    bool accepted = true;
    if (yd != -INFINITY) {  // p(d) > 0
      const float lr = fmaf(zd - yd, k, -(q.c - pn.c)) + log2f(pn.s / q.s);  // log2 q(d)/p(d)
      thr = fminf(1.f, exp2f(lr));
      accepted = philox_uniform(p.seed, b, j + 1, 0) < thr;
    }
    if (write_outputs) {
      dbg_acc[j] = thr;
      dbg_lz[N + 1 + j] = (pn.c + log2f(pn.s)) * kLn2;
    }
    if (!accepted) atomicMin(&s_first, j);
  }
  if (write_outputs && row_thread) dbg_lz[j] = (q.c + log2f(q.s)) * kLn2;
  __syncthreads();
  const int a = s_first;
  if (write_outputs && row_thread) out_tok[j] = j < a ? d : -1;
  if (j == a) {
    Job job;
    job.kind = a < N ? kJobResidual : kJobBonus;
    job.row = a;
    philox_uniforms4(p.seed, b, a + 1, 1, job.u);
    job.k = k;
    job.cq = q.c;
    job.inv_sq = 1.f / q.s;
    job.cp = a < N ? pn.c : 0.f;
    job.inv_sp = a < N ? 1.f / pn.s : 0.f;
    *job_out = job;
    if (write_outputs) {
      p.out_accept[b] = a;
      p.out_kv[b] = a + 1;
    }
  }
}

}  // namespace sv
