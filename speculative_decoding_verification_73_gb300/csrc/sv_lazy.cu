// Lazy (early-exit) verify: the chain of spec_verify, reading a request's
// rows only as far as its walk goes.
//
// "Speculative Decoding and EAGLE-3" lesson, "Invariant: Leviathan rejection
// sampling": the walk goes left to right and stops at the first rejection,
// so the rows after it never influence the result.  Position j needs target
// row j-1 and draft row j-1 (target row j-1 alone at T = 0); the bonus, or
// the last argmax of a fully matched greedy request, needs target row N.
// Fewer bytes when drafts are rejected early, at the price of one dependent
// pass per position.
//
// One cluster of kLazyCluster CTAs per request.  For each position the
// cluster splits the row pair's 64 KB spans among its CTAs, brings each span
// on chip at once (most of it staged in shared memory, the rest in
// registers) and reduces it with the chain's per-group span arithmetic
// (sv_span.cuh; the span holding the draft token also stores its logit),
// keeps the partials in its shared memory (rows of more than kLazyMaxS1
// spans: in the chain's workspace layout), and meets at a cluster barrier;
// then every CTA gathers the position's partials from its peers through
// distributed shared memory and merges
// the same partials and takes the same accept decision, with the walk's
// arithmetic, so the results are those of spec_verify bit for bit.  The
// final token is drawn like the tree walk's: per level-1 block the mass and
// the candidate of levels 2-4, then rank 0 picks level 1.  Errors: the
// temperature and every token are checked first; a row is checked when the
// walk reads it, so a bad row past the stop is not an error.

#include <climits>
#include <cuda_bf16.h>

#include "sv_device.cuh"
#include "sv_law.cuh"
#include "sv_pick.cuh"
#include "sv_span.cuh"
#include "sv_walk.cuh"

namespace sv {
namespace {

#ifndef SV_LAZY_CLUSTER
#define SV_LAZY_CLUSTER 8
#endif
#ifndef SV_LAZY_MINB
#define SV_LAZY_MINB 4
#endif
constexpr int kLazyCluster = SV_LAZY_CLUSTER;  // CTAs per request

// One 64 KB span of a row: the chain's reduction.  On the vector path the
// first kStagedVecs vectors of every thread (thread t's vectors t,
// t + kThreads, ...) are staged in shared memory with cp.async and the
// rest are loaded into registers at the same time -- all of the span in
// flight at once, one round trip instead of the streaming loop's sixteen
// dependent ones, which is what one position of one request costs here --
// and then reduced group by group with the chain's per-group update, so the
// partials equal the chain's.  Staging 48 of the 64 KB lets four CTAs share
// an SM, so all the clusters of a 64-request batch are resident at once
// (measured on 64 requests at V = 128256: 78.5 / 41.4 / 34.6 us per step at
// 3.1 / 0.28 / 0.03 accepted drafts, against 90.0 / 46.3 / 39.0 us with the
// whole span staged and three CTAs per SM).
#ifndef SV_LAZY_STAGE_VECS
#define SV_LAZY_STAGE_VECS 12
#endif
constexpr int kSpanVecs = kSpanBytes / 16 / kThreads;  // vectors per thread of a span
constexpr int kStagedVecs = SV_LAZY_STAGE_VECS < kSpanVecs ? SV_LAZY_STAGE_VECS : kSpanVecs;
constexpr int kHeldVecs = kSpanVecs - kStagedVecs;      // held in registers
constexpr int kLazyStageBytes = kStagedVecs * kThreads * 16;
static_assert(kStagedVecs >= 1 && kStagedVecs <= kSpanVecs, "staged vectors per thread");

template <typename T, bool kGreedy>
__device__ __forceinline__ Partial reduce_span_split(const T* row, int beg, int end, float k, int d,
                                                     float* tok, T* stage) {
  using E = Elem<T>;
  __shared__ float red_f[kThreads / 32];
  __shared__ float red_g[kThreads / 32];
  __shared__ int red_i[kThreads / 32];
  const int nv = (end - beg) / E::kVec;
  const uint4* src = reinterpret_cast<const uint4*>(row + beg);
  uint4* dst = reinterpret_cast<uint4*>(stage);
  const uint4 pad = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
  const int staged = min(nv, kStagedVecs * kThreads);
  for (int v = threadIdx.x; v < staged; v += kThreads) cp_async16(dst + v, src + v);
  uint4 held[kHeldVecs > 0 ? kHeldVecs : 1];
#pragma unroll
  for (int r = 0; r < kHeldVecs; ++r) {
    const int v = threadIdx.x + (kStagedVecs + r) * kThreads;
    held[r] = v < nv ? ld_stream16(src + v) : pad;
  }
  cp_async_wait_all();  // thread t reads back exactly the vectors it copied
  SpanAcc acc = span_acc_init();
  const uint64_t k2 = f2pack(k, k);
  const TokAt ta = kGreedy ? TokAt{-1, 0, 0} : tok_at<T>(beg, end, d);
#pragma unroll
  for (int gi = 0; gi < kSpanVecs / kGroup; ++gi) {
    uint4 g[kGroup];
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
      const int i = gi * kGroup + u;
      const int v = threadIdx.x + i * kThreads;
      if (i < kStagedVecs)
        g[u] = v < nv ? dst[v] : pad;
      else
        g[u] = held[i - kStagedVecs];
    }
    span_group<T, kGreedy>(acc, g, beg, gi, k2, k, ta, tok);
  }
  return span_finish<kGreedy>(acc, red_f, red_g, red_i);
}

template <typename T, bool kVecPath>
__device__ __forceinline__ Partial reduce_row_span(const T* row, int span, int V, bool greedy, float k,
                                                   int d, float* tok, T* stage) {
  constexpr int kSpan = kSpanBytes / static_cast<int>(sizeof(T));
  const int beg = span * kSpan;
  const int end = min(V, beg + kSpan);
  if (!kVecPath) return chunk_partial_scalar<T>(row, beg, end, greedy, k, d, tok);
  return greedy ? reduce_span_split<T, true>(row, beg, end, k, -1, tok, stage)
                : reduce_span_split<T, false>(row, beg, end, k, d, tok, stage);
}

__device__ __forceinline__ RowNorm merge_row(const Partial* parts, int n) {
  float4 pre[kPre];
#pragma unroll
  for (int i = 0; i < kPre; ++i) pre[i] = partial_or_empty(parts + i, i < n);
  return merge_sampled(pre, parts, n);
}

// Rows of up to kLazyMaxS1 spans exchange their partials through
// distributed shared memory (each CTA keeps the partials of its own spans
// of the position in double-buffered slots; after the cluster barrier every
// CTA gathers the row pair's); longer rows go through the workspace.
constexpr int kLazyMaxS1 = 32;
constexpr int kLazySlots = (2 * kLazyMaxS1 + kLazyCluster - 1) / kLazyCluster;  // items per CTA

__device__ __forceinline__ RowMax merge_row_greedy(const Partial* parts, int n) {
  float4 pre[kPre];
#pragma unroll
  for (int i = 0; i < kPre; ++i) pre[i] = partial_or_empty(parts + i, i < n);
  return merge_greedy(pre, parts, n);
}

constexpr int kGo = 0, kStopToken = 1, kStopDraw = 2, kStopError = 3;

template <typename T, bool kVecPath>
__global__ void __cluster_dims__(kLazyCluster, 1, 1) __launch_bounds__(kThreads, SV_LAZY_MINB)
    lazy_kernel(Problem p, Workspace w) {
  using E = Elem<T>;
  extern __shared__ __align__(16) unsigned char s_stage[];  // one span (vector path)
  __shared__ BlockScratch sc;
  __shared__ int s_bad_token, s_state, s_final, s_a, s_row;
  __shared__ float s_law[5];  // k, cq, inv_sq, cp, inv_sp of the draw
  __shared__ float s_u[4];
  __shared__ int s_kind;
  __shared__ __align__(16) Partial s_own[2][kLazySlots];  // this CTA's spans of a position, by parity
  __shared__ float s_owntok[2][kLazySlots];               // their token logits
  __shared__ __align__(16) Partial s_gather[2 * kLazyMaxS1];  // the position's row pair, gathered
  const int b = blockIdx.x / kLazyCluster;
  const unsigned rank = cluster_rank();
  const int N = p.N, V = p.V, S1 = w.S1;
  const int tid = threadIdx.x;
  const float temp = p.temperature[b];
  const int mode = temp_mode(temp);
  const bool greedy = mode == kModeGreedy;
  const float k = mode == kModeSampled ? scale_of(temp) : 0.f;
  int32_t* out_tok = p.out_tokens + static_cast<size_t>(b) * (N + 1);
  const int32_t* toks = p.tokens + static_cast<size_t>(b) * N;

  if (tid == 0) s_bad_token = 0;
  __syncthreads();
  if (tid < N) {
    const int d = toks[tid];
    if (d < 0 || d >= V) atomicOr(&s_bad_token, 1);
  }
  __syncthreads();
  unsigned err = mode == kModeInvalid ? kErrTemp : (s_bad_token ? kErrToken : 0u);

  const int per = 2 * N + 1;
  Partial* parts = w.partials + static_cast<size_t>(b) * per * S1;
  float* tok_logit = w.tok_logit + static_cast<size_t>(b) * per;
  int a = N;
  const bool dsm = S1 <= kLazyMaxS1;  // partials through distributed shared memory
  constexpr int kSpanElems = kSpanBytes / static_cast<int>(sizeof(T));
  if (!err) {
    for (int j = 1; j <= N + 1; ++j) {
      const bool last = j == N + 1;
      const int trow = j - 1;  // target row of this step
      const bool with_draft = !greedy && !last;
      const int nitems = with_draft ? 2 * S1 : S1;
      const int d = last ? -1 : toks[j - 1];
      const int par = j & 1;
      for (int it = static_cast<int>(rank), li = 0; it < nitems; it += kLazyCluster, ++li) {
        const bool dr = it >= S1;
        const int span = dr ? it - S1 : it;
        const int slot = dr ? N + 1 + trow : trow;
        const T* row = dr ? static_cast<const T*>(p.draft) + (static_cast<size_t>(b) * N + trow) * V
                          : static_cast<const T*>(p.target) + (static_cast<size_t>(b) * (N + 1) + trow) * V;
        float* tokp = dsm ? &s_owntok[par][li] : tok_logit + slot;
        const Partial out = reduce_row_span<T, kVecPath>(row, span, V, greedy, k, greedy ? -1 : d, tokp,
                                                         reinterpret_cast<T*>(s_stage));
        if (tid == 0) {
          if (dsm)
            s_own[par][li] = out;
          else
            parts[static_cast<size_t>(slot) * S1 + span] = out;
        }
      }
      if (!dsm) __threadfence();
      cluster_sync();  // the step's partials and token logits are stored
      if (dsm) {
        // item i (span i of the target row, then of the draft row) is in
        // slot i / kLazyCluster of CTA i % kLazyCluster
        if (tid < nitems)
          *reinterpret_cast<float4*>(&s_gather[tid]) =
              ld_dsmem16(&s_own[par][tid / kLazyCluster], static_cast<unsigned>(tid % kLazyCluster));
        __syncthreads();
      }
      if (tid == 0) {
        int state = kGo;
        if (greedy) {
          const RowMax g = dsm ? merge_row_greedy_local(s_gather, S1)
                               : merge_row_greedy(parts + static_cast<size_t>(trow) * S1, S1);
          if (!g.ok) {
            state = kStopError;
          } else if (last || d != g.idx) {
            state = kStopToken;
            s_final = g.idx;
            s_a = j - 1;
          }
        } else {
          const RowNorm q = dsm ? merge_row_local(s_gather, S1) : merge_row(parts + static_cast<size_t>(trow) * S1, S1);
          RowNorm pn{0.f, 1.f, true};
          if (with_draft)
            pn = dsm ? merge_row_local(s_gather + S1, S1)
                     : merge_row(parts + static_cast<size_t>(N + 1 + trow) * S1, S1);
          if (!q.ok || !pn.ok) {
            state = kStopError;
          } else {
            bool accepted = !last;
            if (!last) {
              float zd, yd;
              if (dsm) {  // the items holding d: span d / kSpanElems of each row
                const int it_z = d / kSpanElems, it_y = S1 + d / kSpanElems;
                zd = ld_dsmem(&s_owntok[par][it_z / kLazyCluster], static_cast<unsigned>(it_z % kLazyCluster));
                yd = ld_dsmem(&s_owntok[par][it_y / kLazyCluster], static_cast<unsigned>(it_y % kLazyCluster));
              } else {
                zd = __ldcg(tok_logit + trow);
                yd = __ldcg(tok_logit + N + 1 + trow);
              }
              if (yd != -INFINITY) {  // p(d) > 0
                const float lr = fmaf(zd - yd, k, -(q.c - pn.c)) + log2f(pn.s / q.s);
                accepted = philox_uniform(p.seed, b, j, 0) < fminf(1.f, exp2f(lr));
              }
            }
            if (!accepted) {
              state = kStopDraw;
              s_a = j - 1;
              s_row = trow;
              s_kind = last ? NodeLaw::kQ : NodeLaw::kSampled;
              s_law[0] = k;
              s_law[1] = q.c;
              s_law[2] = 1.f / q.s;
              s_law[3] = pn.c;
              s_law[4] = 1.f / pn.s;
              philox_uniforms4(p.seed, b, j, 1, s_u);
            }
          }
        }
        s_state = state;
      }
      __syncthreads();
      if (s_state != kGo) break;
    }
    // no CTA leaves (or reuses a slot) while another may still read its
    // shared memory
    cluster_sync();
    if (s_state == kStopError) err = kErrLogit;
    a = s_a;
  }
  if (err) {
    if (rank == 0) {
      if (tid <= N) out_tok[tid] = -1;
      if (tid == 0) {
        p.out_accept[b] = -1;
        p.out_kv[b] = 0;
        atomicOr(w.err, err);
      }
    }
    return;  // the same in every CTA of the cluster
  }

  int token = 0;
  if (s_state == kStopToken) {
    token = s_final;
  } else {
    // the drawn token: residual at the rejected row or bonus from row N
    const int row = s_row;
    const NodeLaw law{s_kind, s_law[0], s_law[1], s_law[2], s_law[3], s_law[4], 1.f, 1.f, 0, nullptr};
    const bool need_y = s_kind == NodeLaw::kSampled;
    const T* z = static_cast<const T*>(p.target) + (static_cast<size_t>(b) * (N + 1) + row) * V;
    const T* y = need_y ? static_cast<const T*>(p.draft) + (static_cast<size_t>(b) * N + row) * V : z;
    Job job;
#pragma unroll
    for (int i = 0; i < 4; ++i) job.u[i] = s_u[i];
    const int S3 = w.S3;
    float* masses = w.chunk_sums + static_cast<size_t>(b) * S3;
    int* cands = w.blk_tok + static_cast<size_t>(b) * S3;
    // the blocks' masses and candidates reach rank 0 through distributed
    // shared memory (block c in slot c / kLazyCluster of CTA c % kLazyCluster)
    // when they fit the slots, else through the workspace
    constexpr int kPickSlots = 16;
    __shared__ float s_bmass[kPickSlots];
    __shared__ float s_bcand[kPickSlots];  // the candidate token's bits
    const bool dsm_pick = S3 <= kPickSlots * kLazyCluster;
    auto rf = [&](float zt, float yt, int t) { return law.r(zt, yt, t); };
    int bi = 0;
    for (int c = static_cast<int>(rank); c < S3; c += kLazyCluster, ++bi) {
      const int cbeg = c * kLevel1, cend = min(V, cbeg + kLevel1);
      float h0, h1, mass;
      seg_sums<T, kVecPath>(z, y, need_y, cbeg + tid * kSegTok, cend, rf, h0, h1);
      const int cand = block_pick(
          h0, h1, cbeg, cend, job,
          [&](int t) { return law.r(E::load1(z + t), need_y ? E::load1(y + t) : 0.f, t); }, sc, &mass);
      if (tid == 0) {
        if (dsm_pick) {
          s_bmass[bi] = mass;
          s_bcand[bi] = __int_as_float(cand);
        } else {
          masses[c] = mass;
          cands[c] = cand;
        }
      }
    }
    if (dsm_pick) {
      cluster_sync();  // every block's mass and candidate are in its CTA's shared memory
      if (rank == 0 && tid < 32) {
        const int c1 = warp_pick(
            [&](int i) { return ld_dsmem(&s_bmass[i / kLazyCluster], static_cast<unsigned>(i % kLazyCluster)); },
            S3, job.u[0]);
        if (tid == 0)
          s_final = c1 >= 0 ? __float_as_int(ld_dsmem(&s_bcand[c1 / kLazyCluster],
                                                      static_cast<unsigned>(c1 % kLazyCluster)))
                            : -1;
      }
      cluster_sync();  // rank 0 has read the other CTAs' shared memory
      if (rank != 0) return;
    } else {
      __threadfence();
      cluster_sync();  // every block's mass and candidate are stored
      if (rank != 0) return;
      if (tid < 32) {
        const int c1 = warp_pick([&](int i) { return __ldcg(masses + i); }, S3, job.u[0]);
        if (tid == 0) s_final = c1 >= 0 ? __ldcg(cands + c1) : -1;
      }
      __syncthreads();
    }
    if (s_final < 0 && need_y) {
      // the residual has no mass (float32 rounding only): draw from q
      const NodeLaw lq{NodeLaw::kQ, s_law[0], s_law[1], s_law[2], 0.f, 0.f, 1.f, 1.f, 0, nullptr};
      auto qf = [&](float zt, float yt, int t) { return lq.r(zt, yt, t); };
      for (int c = 0; c < S3; ++c) {
        const int cbeg = c * kLevel1, cend = min(V, cbeg + kLevel1);
        float h0, h1, mass;
        seg_sums<T, kVecPath>(z, z, false, cbeg + tid * kSegTok, cend, qf, h0, h1);
        const int cand = block_pick(
            h0, h1, cbeg, cend, job, [&](int t) { return lq.r(E::load1(z + t), 0.f, t); }, sc, &mass);
        if (tid == 0) {
          masses[c] = mass;
          cands[c] = cand;
        }
      }
      __syncthreads();
      if (tid < 32) {
        const int c1 = warp_pick([&](int i) { return __ldcg(masses + i); }, S3, job.u[0]);
        if (tid == 0) s_final = c1 >= 0 ? __ldcg(cands + c1) : 0;
      }
      __syncthreads();
    }
    token = s_final < 0 ? 0 : s_final;
  }
  if (rank != 0) return;
  if (tid <= N) out_tok[tid] = tid < a ? toks[tid] : (tid == a ? token : -1);
  if (tid == 0) {
    p.out_accept[b] = a;
    p.out_kv[b] = a + 1;
  }
}

template <typename T, bool kVecPath>
cudaError_t launch_lazy_t(const Problem& p, const Workspace& w, cudaStream_t s) {
  const long long blocks = static_cast<long long>(p.B) * kLazyCluster;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const int smem = kVecPath ? kLazyStageBytes : 0;
  if (kVecPath) {
    const cudaError_t e =
        cudaFuncSetAttribute(lazy_kernel<T, kVecPath>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  lazy_kernel<T, kVecPath><<<dim3(static_cast<unsigned>(blocks)), kThreads, smem, s>>>(p, w);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lazy(int dtype, bool vec, const Problem& p, const Workspace& w, cudaStream_t s) {
  if (dtype == 1)
    return vec ? launch_lazy_t<__nv_bfloat16, true>(p, w, s) : launch_lazy_t<__nv_bfloat16, false>(p, w, s);
  return vec ? launch_lazy_t<float, true>(p, w, s) : launch_lazy_t<float, false>(p, w, s);
}

}  // namespace sv
