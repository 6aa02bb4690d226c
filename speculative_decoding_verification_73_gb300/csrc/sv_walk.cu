// The accept/reject walk: one CTA per request, one thread per row j = 0..N.
//
// Thread j merges the row-statistics partials of target row j (and, for a
// sampled request, draft row j), checks the inputs, and evaluates position
// j+1 of the chain.  "Speculative Decoding and EAGLE-3" lesson:
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
// The few per-row scalars are merged and compared in double precision
// (products of two floats are exact there), so the accept thresholds carry
// only the rounding of the fp32 row sums.  The correction / bonus token of a
// sampled request is left to the sampler as a Job.

#include <climits>
#include <cuda_bf16.h>

#include "sv_device.cuh"

namespace sv {
namespace {

constexpr double kLn2 = 0.69314718055994530942;

struct RowNorm {
  float c;      // reference exponent (max over chunks of fl(M k))
  double s;     // sum_t 2^(x_t k - c)
  double l2z;   // c + log2(s) = log2 sum_t 2^(x_t k)
  bool ok;
};

__device__ RowNorm merge_sampled(const Partial* parts, int S1) {
  float c = -INFINITY;
  bool bad = false;
  for (int i = 0; i < S1; ++i) {
    const Partial pt = parts[i];
    if (pt.s != pt.s) bad = true;
    c = fmaxf(c, pt.a);
  }
  RowNorm r;
  r.c = c;
  r.s = 0.0;
  if (!bad && c > -INFINITY) {
    for (int i = 0; i < S1; ++i) {
      const Partial pt = parts[i];
      if (pt.a > -INFINITY) r.s += static_cast<double>(pt.s) * exp2(static_cast<double>(pt.a) - c);
    }
  }
  r.ok = !bad && c > -INFINITY && r.s > 0.0 && r.s < 1e300;
  r.l2z = r.ok ? static_cast<double>(c) + log2(r.s) : 0.0;
  return r;
}

struct RowMax {
  int idx;
  bool ok;
};

__device__ RowMax merge_greedy(const Partial* parts, int S1) {
  float best = -INFINITY;
  int idx = INT_MAX;
  bool bad = false;
  for (int i = 0; i < S1; ++i) {
    const Partial pt = parts[i];
    if (pt.s != pt.s || pt.a != pt.a) bad = true;
    if (pt.a > best) {  // chunks are in index order: strict > keeps the lowest index
      best = pt.a;
      idx = pt.idx;
    }
  }
  RowMax r;
  r.idx = idx;
  r.ok = !bad && best > -INFINITY && best < INFINITY;
  return r;
}

template <typename T>
__device__ __forceinline__ float load_elem(const void* base, size_t off) {
  return Elem<T>::load1(static_cast<const T*>(base) + off);
}

template <typename T>
__global__ void __launch_bounds__(kWalkMaxThreads) walk_kernel(Problem p, Workspace w) {
  const int b = blockIdx.x;
  const int j = threadIdx.x;
  const int N = p.N, V = p.V, S1 = w.S1;
  const bool row_thread = j <= N;
  const bool pos_thread = j < N;

  __shared__ int s_bad_token, s_bad_logit, s_first;
  if (j == 0) {
    s_bad_token = 0;
    s_bad_logit = 0;
    s_first = N;
  }
  __syncthreads();

  const float t = p.temperature[b];
  const int mode = temp_mode(t);
  int d = -1;
  if (pos_thread) {
    d = p.tokens[static_cast<size_t>(b) * N + j];
    if (d < 0 || d >= V) atomicOr(&s_bad_token, 1);
  }

  const size_t trow = static_cast<size_t>(b) * (N + 1) + j;          // target row index
  const size_t drow = static_cast<size_t>(p.B) * (N + 1) +            // draft row index in
                      static_cast<size_t>(b) * N + j;                 // the partials array
  RowNorm q{}, pn{};
  RowMax g{};
  if (mode == kModeGreedy && row_thread) {
    g = merge_greedy(w.partials + trow * S1, S1);
    if (!g.ok) atomicOr(&s_bad_logit, 1);
  } else if (mode == kModeSampled && row_thread) {
    q = merge_sampled(w.partials + trow * S1, S1);
    if (!q.ok) atomicOr(&s_bad_logit, 1);
    if (pos_thread) {
      pn = merge_sampled(w.partials + drow * S1, S1);
      if (!pn.ok) atomicOr(&s_bad_logit, 1);
    }
  }
  __syncthreads();

  unsigned err = 0;
  if (mode == kModeInvalid)
    err = kErrTemp;
  else if (s_bad_token)
    err = kErrToken;
  else if (s_bad_logit)
    err = kErrLogit;

  int32_t* out_tok = p.out_tokens + static_cast<size_t>(b) * (N + 1);
  float* dbg_acc = w.dbg_accept + static_cast<size_t>(b) * N;
  float* dbg_lz = w.dbg_logz + static_cast<size_t>(b) * (2 * N + 1);
  const float qnan = __int_as_float(0x7fc00000);

  if (err) {
    if (row_thread) {
      out_tok[j] = -1;
      dbg_lz[j] = qnan;
      if (pos_thread) {
        dbg_acc[j] = qnan;
        dbg_lz[N + 1 + j] = qnan;
      }
    }
    if (j == 0) {
      p.out_accept[b] = -1;
      p.out_kv[b] = 0;
      w.jobs[b].kind = kJobNone;
      atomicOr(w.err, err);
    }
    return;
  }

  if (mode == kModeGreedy) {
    if (pos_thread && d != g.idx) atomicMin(&s_first, j);
    __syncthreads();
    const int a = s_first;
    if (row_thread) {
      out_tok[j] = j <= a ? g.idx : -1;
      dbg_lz[j] = qnan;
      if (pos_thread) {
        dbg_acc[j] = qnan;
        dbg_lz[N + 1 + j] = qnan;
      }
    }
    if (j == 0) {
      p.out_accept[b] = a;
      p.out_kv[b] = a + 1;
      w.jobs[b].kind = kJobNone;
    }
    return;
  }

  // Sampled request.
  const float k = scale_of(t);
  bool accepted = true;
  if (pos_thread) {
    const float zd = load_elem<T>(p.target, trow * V + d);
    const float yd = load_elem<T>(p.draft, (static_cast<size_t>(b) * N + j) * V + d);
    double thr = 1.0;
    if (yd != -INFINITY) {  // p(d) > 0
      // log2 q(d) - log2 p(d), each x*k exact in double
      const double l2q = static_cast<double>(zd) * k - q.l2z;
      const double l2p = static_cast<double>(yd) * k - pn.l2z;
      thr = fmin(1.0, exp2(l2q - l2p));
      const float u = philox_uniform(p.seed, b, j + 1, 0);
      accepted = static_cast<double>(u) < thr;
    }
    dbg_acc[j] = static_cast<float>(thr);
    dbg_lz[N + 1 + j] = static_cast<float>(pn.l2z * kLn2);
    if (!accepted) atomicMin(&s_first, j);
  }
  if (row_thread) dbg_lz[j] = static_cast<float>(q.l2z * kLn2);
  __syncthreads();
  const int a = s_first;
  if (row_thread) out_tok[j] = j < a ? d : -1;
  if (j == a) {
    Job job;
    job.kind = a < N ? kJobResidual : kJobBonus;
    job.row = a;
    philox_uniforms4(p.seed, b, a + 1, 1, job.u);
    job.k = k;
    job.cq = q.c;
    job.inv_sq = static_cast<float>(1.0 / q.s);
    // log2 Z_q - log2 Z_p as a float pair, so that log2(q_t / p_t) keeps its
    // precision when q_t and p_t are close
    const double dl = a < N ? q.l2z - pn.l2z : 0.0;
    job.dhi = static_cast<float>(dl);
    job.dlo = static_cast<float>(dl - static_cast<double>(job.dhi));
    w.jobs[b] = job;
    p.out_accept[b] = a;
    p.out_kv[b] = a + 1;
  }
}

__global__ void philox_probe_kernel(unsigned long long seed, const uint32_t* ctr3, uint32_t* out4,
                                    int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint2 key = make_uint2(static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  const uint4 r = philox4x32_10(make_uint4(ctr3[3 * i], ctr3[3 * i + 1], ctr3[3 * i + 2], 0u), key);
  out4[4 * i] = r.x;
  out4[4 * i + 1] = r.y;
  out4[4 * i + 2] = r.z;
  out4[4 * i + 3] = r.w;
}

}  // namespace

cudaError_t launch_walk(int dtype, const Problem& p, const Workspace& w, cudaStream_t s) {
  if (p.B <= 0) return cudaSuccess;
  const int threads = ((p.N + 1 + 31) / 32) * 32;
  if (dtype == 1)
    walk_kernel<__nv_bfloat16><<<p.B, threads, 0, s>>>(p, w);
  else
    walk_kernel<float><<<p.B, threads, 0, s>>>(p, w);
  return cudaGetLastError();
}

cudaError_t launch_philox_probe(unsigned long long seed, const uint32_t* ctr3, uint32_t* out4,
                                int n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  philox_probe_kernel<<<(n + 255) / 256, 256, 0, s>>>(seed, ctr3, out4, n);
  return cudaGetLastError();
}

}  // namespace sv
