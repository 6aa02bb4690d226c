// Verification of a draft tree (EAGLE-2's dynamic draft tree).
//
// "Speculative Decoding and EAGLE-3" lesson: the "Key terms" entry on
// EAGLE-2 (a small candidate tree scored by one verifier pass, the walk
// following the most probable path), its tree-mask remark in "KV cache
// rollback", exercise 3 (the [2, 2, 2] tree), and "Invariant: Leviathan
// rejection sampling" for the test at each node.
//
// Node 0 is the root, draft nodes 1..M (parent of node i in [0, i-1], token
// tokens[i-1]); target row r and draft row r belong to node r.  From the
// root, the children of the current node are tried in increasing index: a
// child with token x is accepted iff p(x) = 0 or u < min(1, r(x) / p(x)),
// r the node's current distribution (q at first).  Accepting descends;
// rejecting turns r into (r - p)_+ normalised (r itself if that is all 0).
// When every child is rejected a token is drawn from the final r; at a leaf
// a bonus token is drawn from its q.  SAMPLED mode: the children were drawn
// independently from the node's draft row.  TOPK mode: they are fixed
// candidates, whose drafting law is a point mass on their own token, so
// accept iff u < r(x) and the residual is r with x removed; draft logits are
// not read.  Uniforms: the i-th child tried at depth j uses Philox counter
// (b, j, i == 0 ? 0 : i + 1, 0); the token drawn at depth j uses draw 1 and
// the grouped inverse CDF (levels of 8192 / 256 / 16 / 1 tokens).  T = 0
// descends into the first child whose token is the node's target argmax and
// emits the argmax where there is none.
//
// Two kernels.  tree_rowstats_kernel streams every target row and, for a
// sampled request in SAMPLED mode, the draft rows of nodes that have
// children, one CTA per 64 KB span (the chain's span reduction).
// tree_walk_kernel gives each request a cluster of kTreeCluster CTAs.  Every
// CTA merges the partials of all rows and fetches the logits of every child
// at its token (thread i holds node i), then all of them run the same walk:
// one thread decides, and each rejection in SAMPLED mode of a child that has
// a later sibling triggers a pass in which every CTA sums max(r(t) - p(t), 0)
// over its share of the vocabulary and the cluster's partial sums are
// exchanged through distributed shared memory after a cluster barrier, so
// every CTA holds the same normaliser for that sibling's test.  After the
// last sibling is rejected no pass runs: the draw is scale-free and needs
// only the new residual's offset, known already.  The final draw computes,
// per level-1 block, the block's mass and the token levels 2-4 would pick in
// it (each CTA its own blocks), then rank 0 picks level 1.  All arithmetic is float32; each CTA takes the same decisions
// from the same numbers, so the cluster stays in step.

#include <climits>
#include <cuda_bf16.h>

#include "sv_device.cuh"
#include "sv_law.cuh"
#include "sv_pick.cuh"
#include "sv_span.cuh"
#include "sv_walk.cuh"

namespace sv {
namespace {

// Tuning constants, overridable at build time (-D<name>=<value>): CTAs per
// request cluster and resident CTAs per SM the walk kernel is built for.
#ifndef SV_TREE_CLUSTER
#define SV_TREE_CLUSTER 8
#endif
#ifndef SV_TREE_MINB
#define SV_TREE_MINB 2
#endif
// Resident CTAs per SM the lazy walk is built for (all the request clusters
// of a 64-request batch at once at four).
#ifndef SV_TREE_LAZY_MINB
#define SV_TREE_LAZY_MINB 4
#endif
constexpr int kTreeCluster = SV_TREE_CLUSTER;
constexpr int kMaxNodes = kST;  // root + up to 255 draft nodes, one thread each
constexpr int kNoNode = INT_MAX;

// ------------------------------------------------------------ row statistics

template <typename T, bool kVecPath>
__global__ void __launch_bounds__(kThreads, kSpanMinBlocks) tree_rowstats_kernel(TreeProblem p,
                                                                                   Workspace w) {
  allow_dependents();  // the walk may be scheduled behind the last wave
  const int S1 = w.S1;
  const int per = 2 * (p.M + 1);
  const int row = blockIdx.x / S1;
  const int span = blockIdx.x - row * S1;
  const int b = row / per;
  const int slot = row - b * per;
  const bool draft = slot > p.M;
  const int node = draft ? slot - p.M - 1 : slot;
  const int mode = temp_mode(p.temperature[b]);
  if (mode == kModeInvalid) return;  // CTA-uniform
  if (draft) {
    if (mode == kModeGreedy || p.mode != kTreeSampled) return;
    int has_children = 0;  // only draft rows of inner nodes are read
    const int32_t* par = p.parents + static_cast<size_t>(b) * p.M;
    for (int i = threadIdx.x; i < p.M; i += kThreads) has_children |= par[i] == node;
    if (!__syncthreads_or(has_children)) return;
  }
  const T* base = static_cast<const T*>(draft ? p.draft : p.target) +
                  (static_cast<size_t>(b) * (p.M + 1) + node) * p.V;
  constexpr int kSpan = kSpanBytes / static_cast<int>(sizeof(T));
  const int beg = span * kSpan;
  const int end = min(p.V, beg + kSpan);
  const bool greedy = mode == kModeGreedy;
  const float k = greedy ? 0.f : scale_of(p.temperature[b]);
  Partial out;
  if (!kVecPath) {
    out = chunk_partial_scalar<T>(base, beg, end, greedy, k, -1, nullptr);
  } else if (end - beg == kSpan) {
    out = greedy ? span_partial_vec<T, true, true>(base, beg, end, k, -1, nullptr)
                 : span_partial_vec<T, false, true>(base, beg, end, k, -1, nullptr);
  } else {
    out = greedy ? span_partial_vec<T, true, false>(base, beg, end, k, -1, nullptr)
                 : span_partial_vec<T, false, false>(base, beg, end, k, -1, nullptr);
  }
  if (threadIdx.x == 0) {
    out.tag = p.epoch;
    st_partial_relaxed(w.partials + static_cast<size_t>(row) * S1 + span, out);
  }
}

// ------------------------------------------------------------ the walk

constexpr int kActContinue = 0, kActPass = 1, kActBonus = 2, kActResidual = 3;

// Level-1 blocks a CTA can keep staged in shared memory (both rows of the
// node under test): a residual pass or a draw at the same node then reads
// no global memory.  Staging is used for 16-bit rows with at most
// kStageBlocks blocks per CTA; other cases read the rows from global memory.
constexpr int kStageBlocks = 2;
template <typename T>
constexpr int tree_stage_bytes() {
  return 2 * kStageBlocks * kLevel1 * static_cast<int>(sizeof(T));
}
// Build-time override: -DSV_TREE_STAGE=0 reads the rows from global memory
// (L2 after the first pass) in every pass instead of staging them.
#ifndef SV_TREE_STAGE
#define SV_TREE_STAGE 1
#endif
template <typename T, bool kVecPath>
constexpr bool tree_stages() {
  return SV_TREE_STAGE && kVecPath && sizeof(T) == 2;
}

// The lazy walk (kLazy) reads no row statistics: when the walk reaches a
// node, the cluster reduces that node's target row (and its draft row, for
// a node with children in SAMPLED mode) with the same span reduction as
// tree_rowstats_kernel, one span per CTA at a time, and every CTA merges
// the spans' partials gathered through distributed shared memory in span
// order -- the numbers the eager walk merges, so the two take the same
// decisions.  Rows of nodes the walk never reaches are neither read nor
// checked.  Rows of at most kTreeLazyMaxS1 spans.
constexpr int kTreeLazyMaxS1 = kTreeLazyMaxSpans;
// groups of loads in flight per thread in the lazy walk's span reductions
// (a cp.async ring in dynamic shared memory)
#ifndef SV_TREE_LAZY_RING
#define SV_TREE_LAZY_RING 2
#endif
constexpr int kTreeLazyRing = SV_TREE_LAZY_RING;
constexpr int kTreeLazySlots = (2 * kTreeLazyMaxS1 + kTreeCluster - 1) / kTreeCluster;  // items per CTA

template <typename T, bool kVecPath, bool kLazy>
__global__ void __cluster_dims__(kTreeCluster, 1, 1)
    __launch_bounds__(kST, kLazy ? SV_TREE_LAZY_MINB : SV_TREE_MINB)
    tree_walk_kernel(TreeProblem p, Workspace w) {
  using E = Elem<T>;
  extern __shared__ __align__(16) unsigned char s_stage_raw[];
  __shared__ int s_staged;  // node whose rows are staged, -1 for none
  __shared__ int s_par[kMaxNodes], s_tok[kMaxNodes], s_first[kMaxNodes], s_next[kMaxNodes];
  __shared__ int s_gidx[kMaxNodes], s_path[kMaxNodes], s_rej[kMaxNodes];
  __shared__ float s_cq[kMaxNodes], s_sq[kMaxNodes], s_cp[kMaxNodes], s_sp[kMaxNodes];
  __shared__ float s_zc[kMaxNodes], s_yc[kMaxNodes];
  __shared__ float s_part[2];
  __shared__ BlockScratch scs[2];  // the draw's two staged blocks; scs[0] otherwise
  BlockScratch& sc = scs[0];
  __shared__ Job s_job;
  __shared__ unsigned s_err;
  __shared__ int s_node, s_depth, s_child, s_m, s_plen, s_act;
  __shared__ float s_rej_mass, s_c, s_d;  // s_c, s_d: c_m and D_m of the residual
  // after the node's last child is rejected: c_m before that rejection, and
  // whether D of the new residual is still unknown (no pass was run)
  __shared__ float s_cprev;
  __shared__ int s_tentative;
  __shared__ float s_cmass;  // the sum of this CTA's level-1 block masses in the draw
  // lazy walk: this CTA's span partials of a node visit (double-buffered by
  // visit parity) and the visit's partials gathered from the cluster
  __shared__ __align__(16) Partial s_own[2][kLazy ? kTreeLazySlots : 1];
  __shared__ __align__(16) Partial s_gather[kLazy ? 2 * kTreeLazyMaxS1 : 1];
  __shared__ int s_visit, s_statnode, s_bad;

  const int b = blockIdx.x / kTreeCluster;
  const unsigned rank = cluster_rank();
  const int M = p.M, V = p.V;
  const int i = threadIdx.x;  // node id
  const bool is_node = i <= M;
  const float temp = p.temperature[b];
  const int mode = temp_mode(temp);
  const bool sampled = mode == kModeSampled;
  const bool use_draft = sampled && p.mode == kTreeSampled;
  const float k = sampled ? scale_of(temp) : 0.f;

  // ---- per node: topology, token, row statistics, child logits
  int par = -1, tok = -1;
  if (i >= 1 && is_node) {
    par = p.parents[static_cast<size_t>(b) * M + i - 1];
    tok = p.tokens[static_cast<size_t>(b) * M + i - 1];
  }
  const int S1 = w.S1;
  const Partial* req_parts = w.partials + static_cast<size_t>(b) * 2 * (M + 1) * S1;
  const Partial* tparts = req_parts + static_cast<size_t>(i) * S1;
  const Partial* dparts = req_parts + static_cast<size_t>(M + 1 + i) * S1;
  // Every partial this thread may merge is requested now; which of them the
  // walk needs is known once the topology is (a draft row only for a node
  // with children), and those are then polled until they carry this call's
  // tag (the grid of the row statistics may still be running).
  const float4 empty = make_float4(-INFINITY, 0.f, __int_as_float(INT_MAX), 0.f);
  float4 tpre[kPre], dpre[kPre];
#pragma unroll
  for (int j = 0; j < kPre; ++j) {
    tpre[j] = (!kLazy && is_node && mode != kModeInvalid && j < S1) ? ld_partial_relaxed(tparts + j) : empty;
    dpre[j] = (!kLazy && is_node && use_draft && j < S1) ? ld_partial_relaxed(dparts + j) : empty;
  }
  __shared__ int s_late;
  if (i == 0) {
    s_err = mode == kModeInvalid ? kErrTemp : 0u;
    s_late = 0;
  }
  s_first[i] = kNoNode;
  s_next[i] = kNoNode;
  s_par[i] = par;
  s_tok[i] = tok;
  __syncthreads();
  const bool par_ok = i >= 1 && is_node && par >= 0 && par < i;
  const bool tok_ok = tok >= 0 && tok < V;
  if (i >= 1 && is_node) {
    if (!par_ok) atomicOr(&s_err, kErrTree);
    if (!tok_ok) atomicOr(&s_err, kErrToken);
  }
  if (par_ok) atomicMin(&s_first[par], i);
  __syncthreads();
  if (par_ok) {
    for (int j = i + 1; j <= M; ++j)
      if (s_par[j] == par) {
        s_next[i] = j;
        break;
      }
  }
  // child logits at the child's token, in its parent's rows
  float zc = 0.f, yc = 0.f;
  if (sampled && par_ok && tok_ok) {
    const size_t off = (static_cast<size_t>(b) * (M + 1) + par) * V + tok;
    zc = E::load1(static_cast<const T*>(p.target) + off);
    if (use_draft) yc = E::load1(static_cast<const T*>(p.draft) + off);
  }
  Poll pl{p.epoch, kPollLimit, false};
  const bool take_t = is_node && mode != kModeInvalid;
  const bool take_d = is_node && use_draft && s_first[i] != kNoNode;
  if (!kLazy) settle(tpre, tparts, take_t ? S1 : 0, dpre, dparts, take_d ? S1 : 0, pl);
  if (kLazy) {
    // statistics come node by node, below
  } else if (is_node && mode == kModeGreedy) {
    const RowMax g = merge_greedy_by(tpre, S1, TaggedLoad{tparts, S1, &pl});
    s_gidx[i] = g.idx;
    if (!g.ok) atomicOr(&s_err, kErrLogit);
  } else if (is_node && sampled) {
    const RowNorm q = merge_sampled_by(tpre, S1, TaggedLoad{tparts, S1, &pl});
    s_cq[i] = q.c;
    s_sq[i] = q.s;
    if (!q.ok) atomicOr(&s_err, kErrLogit);
    if (take_d) {
      const RowNorm pn = merge_sampled_by(dpre, S1, TaggedLoad{dparts, S1, &pl});
      s_cp[i] = pn.c;
      s_sp[i] = pn.s;
      if (!pn.ok) atomicOr(&s_err, kErrLogit);
    } else {
      s_cp[i] = 0.f;
      s_sp[i] = 1.f;
    }
  }
  s_zc[i] = zc;
  s_yc[i] = yc;
  if (pl.late) atomicOr(&s_late, 1);
  __syncthreads();
  // A wait that ran out in one CTA fails the request in all of them: that
  // CTA publishes it under the call's tag, and after a cluster barrier every
  // CTA reads it back, so the cluster takes the same branch below (a CTA
  // leaving alone would strand its peers' exchanges through its shared
  // memory).
  unsigned late_tag = 0;
  if (!kLazy) {
    if (i == 0 && s_late)
      asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(w.late + b), "r"(p.epoch) : "memory");
    cluster_sync();
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(late_tag) : "l"(w.late + b) : "memory");
  }

  int32_t* out_tok = p.out_tokens + static_cast<size_t>(b) * (M + 1);
  int32_t* out_path = p.out_path + static_cast<size_t>(b) * M;
  const unsigned bits = s_err | (!kLazy && late_tag == p.epoch ? kErrWait : 0u);
  if (bits) {
    // report the first failing check in the order temperature, topology,
    // tokens, wait, logits (a wait that ran out leaves the partials that the
    // logit check reads unread)
    const unsigned err = (bits & kErrTemp)    ? kErrTemp
                         : (bits & kErrTree)  ? kErrTree
                         : (bits & kErrToken) ? kErrToken
                         : (bits & kErrWait)  ? kErrWait
                                              : kErrLogit;
    if (rank == 0) {
      if (is_node) out_tok[i] = -1;
      if (i < M) out_path[i] = -1;
      if (i == 0) {
        p.out_accept[b] = -1;
        p.out_kv[b] = 0;
        atomicOr(w.err, err);
      }
    }
    return;  // identical in every CTA of the cluster
  }

  // ---- lazy walk: the statistics of one node's rows, reduced by the cluster
  // (span it of the node's target row, then of its draft row, by CTA
  // it % kTreeCluster), merged by thread 0 of every CTA into s_cq / s_sq /
  // s_cp / s_sp (sampled) or s_gidx (greedy); s_bad if a row is bad
  auto node_stats = [&](int node, bool greedy_row) {
    const bool with_draft = !greedy_row && use_draft && s_first[node] != kNoNode;
    const int nitems = with_draft ? 2 * S1 : S1;
    const int par = s_visit & 1;
    constexpr int kSpan = kSpanBytes / static_cast<int>(sizeof(T));
    for (int it = static_cast<int>(rank), li = 0; it < nitems; it += kTreeCluster, ++li) {
      const bool dr = it >= S1;
      const int span = dr ? it - S1 : it;
      const T* row = static_cast<const T*>(dr ? p.draft : p.target) + (static_cast<size_t>(b) * (M + 1) + node) * V;
      const int beg = span * kSpan, end = min(V, beg + kSpan);
      Partial out;
      uint4* ring = reinterpret_cast<uint4*>(s_stage_raw);
      if (!kVecPath)
        out = chunk_partial_scalar<T>(row, beg, end, greedy_row, k, -1, nullptr);
      else if (end - beg == kSpan)
        out = greedy_row ? span_partial_ring<T, true, true, kTreeLazyRing>(row, beg, end, k, -1, nullptr, ring)
                         : span_partial_ring<T, false, true, kTreeLazyRing>(row, beg, end, k, -1, nullptr, ring);
      else
        out = greedy_row ? span_partial_ring<T, true, false, kTreeLazyRing>(row, beg, end, k, -1, nullptr, ring)
                         : span_partial_ring<T, false, false, kTreeLazyRing>(row, beg, end, k, -1, nullptr, ring);
      if (i == 0) s_own[par][li] = out;
    }
    cluster_sync();  // every CTA's partials of this visit are in its shared memory
    if (i < nitems)
      *reinterpret_cast<float4*>(&s_gather[i]) =
          ld_dsmem16(&s_own[par][i / kTreeCluster], static_cast<unsigned>(i % kTreeCluster));
    __syncthreads();
    if (i == 0) {
      bool bad;
      if (greedy_row) {
        const RowMax g = merge_row_greedy_local(s_gather, S1);
        s_gidx[node] = g.idx;
        bad = !g.ok;
      } else {
        const RowNorm q = merge_row_local(s_gather, S1);
        s_cq[node] = q.c;
        s_sq[node] = q.s;
        bad = !q.ok;
        if (with_draft) {
          const RowNorm pn = merge_row_local(s_gather + S1, S1);
          s_cp[node] = pn.c;
          s_sp[node] = pn.s;
          bad = bad || !pn.ok;
        } else {
          s_cp[node] = 0.f;
          s_sp[node] = 1.f;
        }
      }
      s_bad = bad ? 1 : 0;
      s_visit += 1;
    }
    __syncthreads();
  };
  // a visited row is bad: the whole cluster fails the request (the same
  // merged numbers in every CTA), after a cluster barrier so that no CTA
  // leaves while a peer may still read its partial slots
  auto fail_logit = [&]() {
    cluster_sync();
    if (rank == 0) {
      if (is_node) out_tok[i] = -1;
      if (i < M) out_path[i] = -1;
      if (i == 0) {
        p.out_accept[b] = -1;
        p.out_kv[b] = 0;
        atomicOr(w.err, kErrLogit);
      }
    }
  };
  if (kLazy && i == 0) {
    s_visit = 0;
    s_statnode = -1;
  }

  if (kLazy && mode == kModeGreedy) {
    // every CTA walks: descend into the child whose token is the argmax of
    // the node's target row (emitted tokens kept in s_rej)
    if (i == 0) {
      s_node = 0;
      s_plen = 0;
    }
    __syncthreads();
    while (true) {
      node_stats(s_node, true);
      if (s_bad) {
        fail_logit();
        return;
      }
      if (i == 0) {
        const int node = s_node, g = s_gidx[node];
        int c = s_first[node];
        while (c != kNoNode && s_tok[c] != g) c = s_next[c];
        s_rej[s_plen] = g;
        if (c == kNoNode) {
          s_act = 1;
        } else {
          s_path[s_plen++] = c;
          s_node = c;
          s_act = 0;
        }
      }
      __syncthreads();
      if (s_act) break;
    }
    cluster_sync();  // no CTA leaves while a peer may still read its partial slots
    if (rank != 0) return;
    const int plen = s_plen;
    if (is_node) out_tok[i] = i <= plen ? s_rej[i] : -1;
    if (i < M) out_path[i] = i < plen ? s_path[i] : -1;
    if (i == 0) {
      p.out_accept[b] = plen;
      p.out_kv[b] = plen + 1;
    }
    return;
  }

  if (mode == kModeGreedy) {
    if (rank != 0) return;
    if (i == 0) {
      int node = 0, plen = 0;
      while (true) {
        const int g = s_gidx[node];
        int c = s_first[node];
        while (c != kNoNode && s_tok[c] != g) c = s_next[c];
        if (c == kNoNode) {
          out_tok[plen] = g;
          break;
        }
        out_tok[plen] = g;
        out_path[plen] = c;
        s_path[plen++] = c;
        node = c;
      }
      s_plen = plen;
      p.out_accept[b] = plen;
      p.out_kv[b] = plen + 1;
    }
    __syncthreads();
    const int plen = s_plen;
    if (is_node && i > plen) out_tok[i] = -1;
    if (i < M && i >= plen) out_path[i] = -1;
    return;
  }

  // ---- sampled walk: every CTA runs it; thread 0 decides
  if (i == 0) {
    s_node = 0;
    s_depth = 1;
    s_child = s_first[0];
    s_m = 0;
    s_plen = 0;
    s_rej_mass = 0.f;
    s_c = 0.f;
    s_d = 1.f;
    s_tentative = 0;
  }
  __syncthreads();
  const bool topk = p.mode == kTreeTopk;
  const T* zbase = static_cast<const T*>(p.target) + static_cast<size_t>(b) * (M + 1) * V;
  const T* ybase = use_draft ? static_cast<const T*>(p.draft) + static_cast<size_t>(b) * (M + 1) * V
                             : zbase;
  const int S3 = w.S3;
  // this CTA's level-1 blocks: the nbpc consecutive blocks from cfirst (the
  // layout of the chain sampler's blocks, so a one-child tree draws from the
  // same per-block masses in the same order)
  const int nbpc = (S3 + kTreeCluster - 1) / kTreeCluster;
  const int cfirst = static_cast<int>(rank) * nbpc;
  const int clast = min(S3, cfirst + nbpc);
  const bool staging = !kLazy && tree_stages<T, kVecPath>() && nbpc <= kStageBlocks;
  T* sz = reinterpret_cast<T*>(s_stage_raw);        // [kStageBlocks][kLevel1] of z
  T* sy = sz + kStageBlocks * kLevel1;              // the same for y
  if (i == 0) s_staged = -1;
  __syncthreads();
  // Issue this CTA's copies of the node's rows (z, and y when read) into the
  // staging buffer unless they are staged already: one group of copies per
  // level-1 block slot (kStageBlocks groups, empty ones included), so a
  // thread starts on its own vectors of block 0 while block 1's are still
  // arriving.  Before reading its vectors of slot bi a thread waits for its
  // own copies with cp_async_wait_pending(kStageBlocks - 1 - bi); other
  // threads' vectors are read only after a CTA barrier.  Thread 0 records
  // the node in s_staged after the caller's next CTA barrier (every thread
  // has read s_staged by then).
  auto stage_issue = [&](int node, bool with_y) {
    const bool fresh = s_staged != node;
    const T* z = zbase + static_cast<size_t>(node) * V;
    const T* y = ybase + static_cast<size_t>(node) * V;
    for (int bi = 0, c = cfirst; bi < kStageBlocks; ++bi, ++c) {
      if (fresh && c < clast) {
        const int cbeg = c * kLevel1, cend = min(V, cbeg + kLevel1);
        constexpr int kVec = Elem<T>::kVec;
        for (int v = 0; v < kSegTok / kVec; ++v) {  // the layout of staged_at
          const int e = i * kSegTok + v * kVec;
          const int at = bi * kLevel1 + (v * kST + i) * kVec;
          if (cbeg + e < cend) {
            cp_async16(sz + at, z + cbeg + e);
            if (with_y) cp_async16(sy + at, y + cbeg + e);
          }
        }
      }
      cp_async_commit();
    }
  };
  int pass = 0;
  while (true) {
    if (kLazy && s_statnode != s_node) {
      node_stats(s_node, false);  // the walk has just reached this node
      if (s_bad) {
        fail_logit();
        return;
      }
      if (i == 0) s_statnode = s_node;
      __syncthreads();
    }
    if (i == 0) {
      const int node = s_node, c = s_child, m = s_m;
      int act = kActContinue;
      if (c == kNoNode) {
        act = s_first[node] == kNoNode ? kActBonus : kActResidual;
      } else {
        const float zx = s_zc[c], yx = s_yc[c];
        const float cq = s_cq[node], sq = s_sq[node];
        const float u = philox_uniform(p.seed, b, s_depth, m == 0 ? 0u : static_cast<uint32_t>(m + 1));
        bool ok;
        if (!topk) {
          const float cp = s_cp[node], sp = s_sp[node];
          if (yx == -INFINITY) {
            ok = true;  // the drafter gives the child no mass
          } else if (m == 0) {
            // log2 q(x)/p(x), every term small when q and p are close
            const float lr = fmaf(zx - yx, k, -(cq - cp)) + log2f(sp / sq);
            ok = u < fminf(1.f, exp2f(lr));
          } else {
            const float qx = exp2f(fmaf(zx, k, -cq)) / sq;
            const float px = exp2f(fmaf(yx, k, -cp)) / sp;
            const float v = fmaxf(fmaf(-s_c, px, qx), 0.f) / s_d;  // r_m(x)
            ok = u < fminf(1.f, v / px);
          }
        } else {
          const int x = s_tok[c];
          bool seen = false;
          for (int j = 0; j < m; ++j) seen |= s_rej[j] == x;
          const float qx = exp2f(fmaf(zx, k, -cq)) / sq;
          const float rest = 1.f - s_rej_mass;  // q's mass left after the rejected tokens
          const float rx = seen ? 0.f : (rest > 0.f ? qx / rest : 1.f);
          ok = u < fminf(1.f, rx);
          if (!ok) {
            s_rej[m] = x;
            if (!seen) s_rej_mass += qx;
            s_m = m + 1;
            s_child = s_next[c];
          }
        }
        if (ok) {
          s_path[s_plen++] = c;
          s_node = c;
          s_depth += 1;
          s_child = s_first[c];
          s_m = 0;
          s_rej_mass = 0.f;
          s_c = 0.f;
          s_d = 1.f;
        } else if (!topk) {
          if (s_next[c] == kNoNode) {
            // The node's last child: the draw that follows is scale-free, so
            // it needs c_{m+1} = c_m + D_m but not D_{m+1}, and no pass runs.
            // Should (q - c_{m+1} p)_+ have no mass anywhere, the draw finds
            // out and falls back to r_m, as a pass would have left it.
            s_cprev = s_c;
            s_c = s_c + s_d;
            s_m = m + 1;
            s_child = kNoNode;
            s_tentative = 1;
            act = kActResidual;
          } else {
            act = kActPass;
          }
        }
      }
      s_act = act;
    }
    __syncthreads();
    const int act = s_act;
    if (act == kActContinue) continue;
    if (act != kActPass) break;
    // Residual pass: every CTA sums (r_m - p)_+ over its level-1 blocks.
    const int node = s_node;
    // S_{m+1} = sum_t (q - c_{m+1} p)_+ / D_m, c_{m+1} = c_m + D_m
    const float c_next = s_c + s_d;
    const NodeLaw law{NodeLaw::kSampled, k, s_cq[node], 1.f / s_sq[node], s_cp[node],
                      1.f / s_sp[node], c_next, 1.f / s_d, 0, s_rej};
    const T* z = zbase + static_cast<size_t>(node) * V;
    const T* y = ybase + static_cast<size_t>(node) * V;
    float acc = 0.f;
    auto lf = [&](float zt, float yt, int t) { return law.r(zt, yt, t); };
    if (staging) {
      stage_issue(node, true);
      int bi = 0;
      for (int c = cfirst; c < clast; ++c, ++bi) {
        float h0, h1;
        const int cbeg = c * kLevel1;
        cp_async_wait_pending(kStageBlocks - 1 - bi);  // this thread's copies of slot bi
        law_sums_staged<T>(law, sz + bi * kLevel1, sy + bi * kLevel1, true, cbeg, min(V, cbeg + kLevel1), h0,
                           h1);
        acc += h0 + h1;
      }
    } else {
      for (int c = cfirst; c < clast; ++c) {
        float h0, h1;
        seg_sums<T, kVecPath>(z, y, true, c * kLevel1 + i * kSegTok, min(V, (c + 1) * kLevel1), lf, h0,
                              h1);
        acc += h0 + h1;
      }
    }
    acc = cta_sum(acc, sc.red);
    if (i == 0) {
      s_part[pass & 1] = acc;
      if (staging) s_staged = node;
    }
    cluster_sync();
    if (i == 0) {
      float total = 0.f;
      for (unsigned r = 0; r < kTreeCluster; ++r) total += ld_dsmem(&s_part[pass & 1], r);
      if (total > 0.f) {  // else the residual step leaves r as it is
        s_c = c_next;
        s_d *= total;
      }
      s_m += 1;
      s_child = s_next[s_child];
    }
    ++pass;
    __syncthreads();
  }

  // ---- the drawn token: bonus from q at a leaf, else from the final r
  const int node = s_node;
  const int depth = s_depth;
  const bool bonus = s_act == kActBonus;
  if (i == 0) philox_uniforms4(p.seed, b, depth, 1, s_job.u);
  __syncthreads();
  const Job job = s_job;
  float* masses = w.chunk_sums + static_cast<size_t>(b) * S3;
  int* cands = w.blk_tok + static_cast<size_t>(b) * S3;
  // the blocks' masses and candidates reach rank 0 through distributed
  // shared memory (block c in slot c % nbpc of CTA c / nbpc) when they fit
  // the slots, else through the workspace
  constexpr int kPickSlots = 16;
  __shared__ float s_bmass[kPickSlots];
  __shared__ float s_bcand[kPickSlots];  // the candidate token's bits
  const bool dsm_pick = nbpc <= kPickSlots;
  while (true) {
    // a draw is scale-free: r_m is taken as (q - c_m p)_+ without the 1 / D_m
    const NodeLaw law{bonus ? NodeLaw::kQ : (topk ? NodeLaw::kTopk : NodeLaw::kSampled), k,
                      s_cq[node], 1.f / s_sq[node], s_cp[node], 1.f / s_sp[node], s_c, 1.f, s_m, s_rej};
    const bool need_y = law.kind == NodeLaw::kSampled && s_m > 0;
    const T* z = zbase + static_cast<size_t>(node) * V;
    const T* y = ybase + static_cast<size_t>(node) * V;
    auto rf = [&](float zt, float yt, int t) { return law.r(zt, yt, t); };
    if (staging) stage_issue(node, need_y);
    float cmass = 0.f;  // thread 0: the masses of this CTA's blocks
    if (staging) {
      // both staged blocks' sums, then their picks with one set of CTA barriers
      const int nb = max(0, clast - cfirst);
      float h0[kStageBlocks], h1[kStageBlocks], mass[kStageBlocks];
      int cand[kStageBlocks];
#pragma unroll
      for (int bi = 0; bi < kStageBlocks; ++bi) {
        h0[bi] = 0.f;
        h1[bi] = 0.f;
        cp_async_wait_pending(kStageBlocks - 1 - bi);  // this thread's copies of slot bi
        if (bi < nb) {
          const int cbeg = (cfirst + bi) * kLevel1;
          law_sums_staged<T>(law, sz + bi * kLevel1, sy + bi * kLevel1, need_y, cbeg, min(V, cbeg + kLevel1),
                             h0[bi], h1[bi]);
        }
      }
      blocks_pick<kStageBlocks>(
          h0, h1, cfirst * kLevel1, V, nb, job,
          [&](int bb, int t) {
            const int e = bb * kLevel1 + staged_at<T>(t - (cfirst + bb) * kLevel1);
            return law.r(staged_elem(sz + e), need_y ? staged_elem(sy + e) : 0.f, t);
          },
          scs, mass, cand);
      if (i == 0) {
        for (int bi = 0; bi < nb; ++bi) {
          cmass += mass[bi];
          if (dsm_pick) {
            s_bmass[bi] = mass[bi];
            s_bcand[bi] = __int_as_float(cand[bi]);
          } else {
            masses[cfirst + bi] = mass[bi];
            cands[cfirst + bi] = cand[bi];
          }
        }
      }
    } else {
      int bi = 0;
      for (int c = cfirst; c < clast; ++c, ++bi) {
        const int cbeg = c * kLevel1, cend = min(V, cbeg + kLevel1);
        float h0, h1, mass;
        seg_sums<T, kVecPath>(z, y, need_y, cbeg + i * kSegTok, cend, rf, h0, h1);
        const int cand = block_pick(
            h0, h1, cbeg, cend, job,
            [&](int t) { return law.r(E::load1(z + t), need_y ? E::load1(y + t) : 0.f, t); }, sc, &mass);
        if (i == 0) {
          cmass += mass;
          if (dsm_pick) {
            s_bmass[bi] = mass;
            s_bcand[bi] = __int_as_float(cand);
          } else {
            masses[c] = mass;
            cands[c] = cand;
          }
        }
      }
    }
    if (i == 0) s_cmass = cmass;
    if (!dsm_pick) __threadfence();
    cluster_sync();  // every block's mass and candidate are stored
    if (staging && i == 0) s_staged = node;
    if (!s_tentative) break;
    // no pass ran for the last rejection: fall back to r_m if the new
    // residual has no mass in any CTA (the same answer in every CTA)
    const float cm = i < kTreeCluster ? ld_dsmem(&s_cmass, static_cast<unsigned>(i)) : 0.f;
    const bool has_mass = __syncthreads_or(cm > 0.f) != 0;
    cluster_sync();  // every CTA has read the others' sums
    if (has_mass) break;
    if (i == 0) {
      s_c = s_cprev;
      s_tentative = 0;
    }
    __syncthreads();
  }
  if (dsm_pick) {
    if (rank == 0 && i < 32) {
      const int c1 = warp_pick(
          [&](int j) { return ld_dsmem(&s_bmass[j % nbpc], static_cast<unsigned>(j / nbpc)); },
          S3, job.u[0]);
      if (i == 0)
        s_child = c1 >= 0 ? __float_as_int(ld_dsmem(&s_bcand[c1 % nbpc], static_cast<unsigned>(c1 / nbpc)))
                          : 0;
    }
    cluster_sync();  // rank 0 has read the other CTAs' shared memory
    if (rank != 0) return;
  } else {
    if (rank != 0) return;
    if (i < 32) {
      const int c1 = warp_pick([&](int j) { return __ldcg(masses + j); }, S3, job.u[0]);
      if (i == 0) s_child = c1 >= 0 ? __ldcg(cands + c1) : 0;
    }
    __syncthreads();
  }
  const int plen = s_plen;
  if (is_node) {
    if (i < plen)
      out_tok[i] = s_tok[s_path[i]];
    else
      out_tok[i] = i == plen ? s_child : -1;
  }
  if (i < M) out_path[i] = i < plen ? s_path[i] : -1;
  if (i == 0) {
    p.out_accept[b] = plen;
    p.out_kv[b] = plen + 1;
  }
}

template <typename T, bool kVecPath>
cudaError_t launch_tree_t(const TreeProblem& p, const Workspace& w, cudaStream_t s, bool walk) {
  if (!walk) {
    const long long blocks = static_cast<long long>(p.B) * 2 * (p.M + 1) * w.S1;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    tree_rowstats_kernel<T, kVecPath><<<dim3(static_cast<unsigned>(blocks)), kThreads, 0, s>>>(p, w);
  } else {
    const long long blocks = static_cast<long long>(p.B) * kTreeCluster;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int smem = tree_stages<T, kVecPath>() ? tree_stage_bytes<T>() : 0;
    if (smem > 0) {
      const cudaError_t e = cudaFuncSetAttribute(tree_walk_kernel<T, kVecPath, false>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
    }
    // Programmatic dependent launch: the clusters may be scheduled once
    // every row-statistics CTA has started (all of them resident or done, so
    // a walk polling for partials never holds back a CTA it waits for).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kST);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tree_walk_kernel<T, kVecPath, false>, p, w);
  }
  return cudaGetLastError();
}

template <typename T, bool kVecPath>
cudaError_t launch_tree_lazy_t(const TreeProblem& p, const Workspace& w, cudaStream_t s) {
  const long long blocks = static_cast<long long>(p.B) * kTreeCluster;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL || w.S1 > kTreeLazyMaxS1) return cudaErrorInvalidConfiguration;
  const int smem = kVecPath ? span_ring_bytes<kTreeLazyRing>() : 0;
  tree_walk_kernel<T, kVecPath, true><<<dim3(static_cast<unsigned>(blocks)), kST, smem, s>>>(p, w);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tree_rowstats(int dtype, bool vec, const TreeProblem& p, const Workspace& w,
                                 cudaStream_t s) {
  if (dtype == 1)
    return vec ? launch_tree_t<__nv_bfloat16, true>(p, w, s, false)
               : launch_tree_t<__nv_bfloat16, false>(p, w, s, false);
  return vec ? launch_tree_t<float, true>(p, w, s, false) : launch_tree_t<float, false>(p, w, s, false);
}

cudaError_t launch_tree_lazy(int dtype, bool vec, const TreeProblem& p, const Workspace& w,
                             cudaStream_t s) {
  if (dtype == 1)
    return vec ? launch_tree_lazy_t<__nv_bfloat16, true>(p, w, s) : launch_tree_lazy_t<__nv_bfloat16, false>(p, w, s);
  return vec ? launch_tree_lazy_t<float, true>(p, w, s) : launch_tree_lazy_t<float, false>(p, w, s);
}

cudaError_t launch_tree_walk(int dtype, bool vec, const TreeProblem& p, const Workspace& w,
                             cudaStream_t s) {
  if (dtype == 1)
    return vec ? launch_tree_t<__nv_bfloat16, true>(p, w, s, true)
               : launch_tree_t<__nv_bfloat16, false>(p, w, s, true);
  return vec ? launch_tree_t<float, true>(p, w, s, true) : launch_tree_t<float, false>(p, w, s, true);
}

}  // namespace sv
