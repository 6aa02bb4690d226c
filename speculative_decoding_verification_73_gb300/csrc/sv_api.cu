// C ABI of libspecverify: context, argument checks, workspace and launches.
// The operation itself is documented in include/spec_verify.h.

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/spec_verify.h"
#include "sv_internal.cuh"

struct spec_verify_ctx {
  int max_B, max_N, max_V, dtype;
  int device;
  cudaStream_t stream;
  void* ws;  // one cudaMalloc holding the whole workspace
  sv::Workspace w;
  // profiling
  int profile_every;                // record every n-th call (0 = off)
  long long profile_seen;           // calls since profiling was turned on
  std::vector<cudaEvent_t> events;  // SV_NUM_KERNELS + 1 per recorded call
  int recorded;                     // calls whose events are in `events`
  double ms[SV_NUM_KERNELS];
  int calls;
  // sequence number of the last chain call: the tag of its row-statistics
  // partials (1, 2, ...; the partials are cleared again when it wraps)
  unsigned epoch;
  size_t part_bytes;  // bytes of the partials region
  size_t late_bytes;  // bytes of the tree walk's timeout tags
  size_t arr_bytes;   // bytes of the sampler's epoch-tagged arrival words
  int skip_rowstats;  // test hook: calls launch their walk kernel alone
  int late_cta;       // test hook: sampler CTA that acts as if its waits ran out
};

namespace {

constexpr int kMaxB = 1 << 20;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int flush_profile(spec_verify_ctx* ctx) {
  if (ctx->recorded == 0) return SV_OK;
  if (cudaStreamSynchronize(ctx->stream) != cudaSuccess) return SV_ECUDA;
  const int per = SV_NUM_KERNELS + 1;
  for (int c = 0; c < ctx->recorded; ++c) {
    for (int k = 0; k < SV_NUM_KERNELS; ++k) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, ctx->events[c * per + k], ctx->events[c * per + k + 1]) !=
          cudaSuccess)
        return SV_ECUDA;
      ctx->ms[k] += ms;
    }
  }
  ctx->calls += ctx->recorded;
  ctx->recorded = 0;
  return SV_OK;
}

cudaEvent_t* profile_slot(spec_verify_ctx* ctx) {
  const int per = SV_NUM_KERNELS + 1;
  constexpr int kMaxRecorded = 4096;
  if (ctx->recorded == kMaxRecorded && flush_profile(ctx) != SV_OK) return nullptr;
  const size_t need = static_cast<size_t>(ctx->recorded + 1) * per;
  while (ctx->events.size() < need) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    ctx->events.push_back(e);
  }
  return ctx->events.data() + static_cast<size_t>(ctx->recorded) * per;
}

// The next call's sequence number: the tag its row statistics carry.  When
// the count wraps, every tag in the workspace is cleared first, so no tag
// left by an earlier call can equal a later call's.
int next_epoch(spec_verify_ctx* ctx, unsigned* epoch) {
  if (++ctx->epoch == 0) {
    if (cudaMemsetAsync(ctx->w.partials, 0, ctx->part_bytes, ctx->stream) != cudaSuccess ||
        cudaMemsetAsync(ctx->w.late, 0, ctx->late_bytes, ctx->stream) != cudaSuccess ||
        cudaMemsetAsync(ctx->w.arrivals, 0, ctx->arr_bytes, ctx->stream) != cudaSuccess)
      return SV_ECUDA;
    ctx->epoch = 1;
  }
  *epoch = ctx->epoch;
  return SV_OK;
}

}  // namespace

extern "C" {

const char* spec_verify_strerror(int code) {
  switch (code) {
    case SV_OK: return "success";
    case SV_EINVAL: return "invalid argument (null pointer, size or dtype out of range)";
    case SV_EBADTEMP: return "a temperature is negative, NaN, infinite or subnormal";
    case SV_EBADTOKEN: return "a draft token is outside [0, V)";
    case SV_EBADLOGIT: return "a logit row holds NaN or +inf, or has no finite entry";
    case SV_ECUDA: return "a CUDA runtime call failed";
    case SV_EBADTREE: return "a draft-tree node's parent is outside [0, node - 1]";
    case SV_EBADKV:
      return "a KV commit would pass the cache length, read outside the window, or keep "
             "positions that do not rise";
    case SV_ETIMEOUT: return "a bounded device wait ran out (a kernel stopped early)";
    case SV_ESCRATCH:
      return "the problem needs more working memory than spec_verify_noalloc's static array "
             "(SV_NOALLOC_SCRATCH_BYTES) holds";
    default: return "unknown error code";
  }
}

int spec_verify_launches_per_call(void) { return SV_NUM_KERNELS; }

int spec_verify_init(spec_verify_ctx** out, int max_B, int max_N, int max_V, sv_dtype dtype,
                     void* cuda_stream) {
  if (out == nullptr) return SV_EINVAL;
  *out = nullptr;
  if (max_B < 1 || max_B > kMaxB || max_N < 0 || max_N > SV_MAX_N || max_V < 1 ||
      max_V > SV_MAX_V || (dtype != SV_F32 && dtype != SV_BF16))
    return SV_EINVAL;
  spec_verify_ctx* ctx = new (std::nothrow) spec_verify_ctx();
  if (ctx == nullptr) return SV_ECUDA;
  ctx->max_B = max_B;
  ctx->max_N = max_N;
  ctx->max_V = max_V;
  ctx->dtype = dtype;
  ctx->stream = static_cast<cudaStream_t>(cuda_stream);
  ctx->late_cta = -1;
  if (cudaGetDevice(&ctx->device) != cudaSuccess) {
    delete ctx;
    return SV_ECUDA;
  }
  const int s1 = ceil_div(max_V, sv::row_chunk_elems(dtype));
  const int s3 = ceil_div(max_V, sv::sample_chunk_elems(dtype));
  const size_t rows = static_cast<size_t>(max_B) * (2 * static_cast<size_t>(max_N) + 1);
  // partials also serve a tree of up to max_N draft nodes: 2 (max_N + 1) rows
  const size_t part_rows = static_cast<size_t>(max_B) * (2 * static_cast<size_t>(max_N) + 2);
  size_t off = 0;
  const size_t o_part = off;
  off = align_up(off + part_rows * s1 * sizeof(sv::Partial), 256);
  const size_t o_tok = off;
  off = align_up(off + rows * sizeof(float), 256);
  const size_t o_sums = off;
  off = align_up(off + static_cast<size_t>(max_B) * s3 * sizeof(float), 256);
  const size_t o_btok = off;
  off = align_up(off + static_cast<size_t>(max_B) * s3 * sizeof(int), 256);
  const size_t o_err = off;
  off = align_up(off + sizeof(unsigned), 256);
  const size_t o_arr = off;
  off = align_up(off + static_cast<size_t>(max_B) * sizeof(unsigned long long), 256);
  const size_t o_late = off;
  off = align_up(off + static_cast<size_t>(max_B) * sizeof(unsigned), 256);
  // the error word, arrival counters and tree-walk timeout tags start at zero
  const size_t zero_bytes = off - o_err;
  const size_t o_acc = off;
  off = align_up(off + static_cast<size_t>(max_B) * (max_N > 0 ? max_N : 1) * sizeof(float), 256);
  const size_t o_lz = off;
  off = align_up(off + rows * sizeof(float), 256);
  if (cudaMalloc(&ctx->ws, off) != cudaSuccess) {
    delete ctx;
    return SV_ECUDA;
  }
  char* base = static_cast<char*>(ctx->ws);
  ctx->w.partials = reinterpret_cast<sv::Partial*>(base + o_part);
  ctx->w.tok_logit = reinterpret_cast<float*>(base + o_tok);
  ctx->w.chunk_sums = reinterpret_cast<float*>(base + o_sums);
  ctx->w.blk_tok = reinterpret_cast<int*>(base + o_btok);
  ctx->w.err = reinterpret_cast<unsigned*>(base + o_err);
  ctx->w.arrivals = reinterpret_cast<unsigned long long*>(base + o_arr);
  ctx->arr_bytes = static_cast<size_t>(max_B) * sizeof(unsigned long long);
  ctx->w.late = reinterpret_cast<unsigned*>(base + o_late);
  ctx->late_bytes = static_cast<size_t>(max_B) * sizeof(unsigned);
  ctx->w.dbg_accept = reinterpret_cast<float*>(base + o_acc);
  ctx->w.dbg_logz = reinterpret_cast<float*>(base + o_lz);
  // tags start at 0, which no chain call uses
  ctx->part_bytes = part_rows * s1 * sizeof(sv::Partial);
  ctx->epoch = 0;
  if (cudaMemsetAsync(base + o_err, 0, zero_bytes, ctx->stream) != cudaSuccess ||
      cudaMemsetAsync(base + o_part, 0, ctx->part_bytes, ctx->stream) != cudaSuccess ||
      cudaStreamSynchronize(ctx->stream) != cudaSuccess) {
    cudaFree(ctx->ws);
    delete ctx;
    return SV_ECUDA;
  }
  *out = ctx;
  return SV_OK;
}

int spec_verify(spec_verify_ctx* ctx, int B, int N, int V, const void* target_logits,
                const void* draft_logits, const int32_t* draft_tokens, const float* temperature,
                uint64_t seed, int32_t* out_tokens, int32_t* out_accept_len,
                int32_t* out_kv_len) {
  if (ctx == nullptr) return SV_EINVAL;
  if (B < 0 || B > ctx->max_B || N < 0 || N > ctx->max_N || V < 1 || V > ctx->max_V)
    return SV_EINVAL;
  if (B == 0) return SV_OK;
  if (target_logits == nullptr || temperature == nullptr || out_tokens == nullptr ||
      out_accept_len == nullptr || out_kv_len == nullptr)
    return SV_EINVAL;
  if (N > 0 && (draft_logits == nullptr || draft_tokens == nullptr)) return SV_EINVAL;

  const size_t esize = ctx->dtype == SV_BF16 ? 2 : 4;
  const bool vec = (static_cast<size_t>(V) * esize) % 16 == 0 && aligned16(target_logits) &&
                   (N == 0 || aligned16(draft_logits));
  sv::Problem p;
  p.B = B;
  p.N = N;
  p.V = V;
  p.target = target_logits;
  p.draft = draft_logits;
  p.tokens = draft_tokens;
  p.temperature = temperature;
  p.seed = seed;
  p.out_tokens = out_tokens;
  p.out_accept = out_accept_len;
  p.out_kv = out_kv_len;
  sv::Workspace w = ctx->w;
  w.S1 = ceil_div(V, sv::row_chunk_elems(ctx->dtype));
  w.S3 = ceil_div(V, sv::sample_chunk_elems(ctx->dtype));
  p.debug_late_cta = ctx->late_cta;
  // A fresh tag per call: the sampler of this call takes a partial only once
  // it carries this tag, never one left by an earlier call.
  if (next_epoch(ctx, &p.epoch) != SV_OK) return SV_ECUDA;

  cudaEvent_t* ev = nullptr;
  if (ctx->profile_every > 0 && (ctx->profile_seen++ % ctx->profile_every) == 0) {
    ev = profile_slot(ctx);
    if (ev == nullptr) return SV_ECUDA;
    if (cudaEventRecord(ev[0], ctx->stream) != cudaSuccess) return SV_ECUDA;
  }
  if (!ctx->skip_rowstats && sv::launch_rowstats(ctx->dtype, vec, p, w, ctx->stream) != cudaSuccess)
    return SV_ECUDA;
  if (ev && cudaEventRecord(ev[1], ctx->stream) != cudaSuccess) return SV_ECUDA;
  if (sv::launch_sample(ctx->dtype, vec, p, w, ctx->stream) != cudaSuccess) return SV_ECUDA;
  if (ev) {
    if (cudaEventRecord(ev[2], ctx->stream) != cudaSuccess) return SV_ECUDA;
    ctx->recorded += 1;
  }
  return SV_OK;
}

namespace {

// spec_verify_tree and spec_verify_tree_lazy: the same checks and problem;
// the eager form streams every row first, the lazy one only the rows its
// walk reaches (rows of at most 32 spans).
int tree_call(spec_verify_ctx* ctx, bool lazy, int B, int M, int V, int mode, const void* target_logits,
              const void* draft_logits, const int32_t* parents, const int32_t* draft_tokens,
              const float* temperature, uint64_t seed, int32_t* out_tokens, int32_t* out_path,
              int32_t* out_accept_len, int32_t* out_kv_len) {
  if (ctx == nullptr) return SV_EINVAL;
  if (B < 0 || B > ctx->max_B || M < 0 || M > ctx->max_N || V < 1 || V > ctx->max_V ||
      (mode != SV_TREE_SAMPLED && mode != SV_TREE_TOPK))
    return SV_EINVAL;
  if (lazy && ceil_div(V, sv::row_chunk_elems(ctx->dtype)) > sv::kTreeLazyMaxSpans) return SV_EINVAL;
  if (B == 0) return SV_OK;
  if (target_logits == nullptr || temperature == nullptr || out_tokens == nullptr ||
      out_accept_len == nullptr || out_kv_len == nullptr)
    return SV_EINVAL;
  if (M > 0 && (parents == nullptr || draft_tokens == nullptr || out_path == nullptr))
    return SV_EINVAL;
  const bool use_draft = mode == SV_TREE_SAMPLED && M > 0;
  if (use_draft && draft_logits == nullptr) return SV_EINVAL;

  const size_t esize = ctx->dtype == SV_BF16 ? 2 : 4;
  const bool vec = (static_cast<size_t>(V) * esize) % 16 == 0 && aligned16(target_logits) &&
                   (!use_draft || aligned16(draft_logits));
  sv::TreeProblem p;
  p.B = B;
  p.M = M;
  p.V = V;
  p.mode = mode;
  p.target = target_logits;
  p.draft = use_draft ? draft_logits : target_logits;
  p.parents = parents;
  p.tokens = draft_tokens;
  p.temperature = temperature;
  p.seed = seed;
  p.out_tokens = out_tokens;
  p.out_path = out_path;
  p.out_accept = out_accept_len;
  p.out_kv = out_kv_len;
  p.epoch = 0;
  sv::Workspace w = ctx->w;
  w.S1 = ceil_div(V, sv::row_chunk_elems(ctx->dtype));
  w.S3 = ceil_div(V, sv::sample_chunk_elems(ctx->dtype));
  // the eager walk polls the tags of this call's partials
  if (!lazy && next_epoch(ctx, &p.epoch) != SV_OK) return SV_ECUDA;

  cudaEvent_t* ev = nullptr;
  if (ctx->profile_every > 0 && (ctx->profile_seen++ % ctx->profile_every) == 0) {
    ev = profile_slot(ctx);
    if (ev == nullptr) return SV_ECUDA;
    if (cudaEventRecord(ev[0], ctx->stream) != cudaSuccess) return SV_ECUDA;
  }
  if (lazy) {
    if (sv::launch_tree_lazy(ctx->dtype, vec, p, w, ctx->stream) != cudaSuccess) return SV_ECUDA;
    if (ev) {  // one kernel: its time is reported as kernel 0, kernel 1 gets ~0
      if (cudaEventRecord(ev[1], ctx->stream) != cudaSuccess ||
          cudaEventRecord(ev[2], ctx->stream) != cudaSuccess)
        return SV_ECUDA;
      ctx->recorded += 1;
    }
    return SV_OK;
  }
  if (!ctx->skip_rowstats && sv::launch_tree_rowstats(ctx->dtype, vec, p, w, ctx->stream) != cudaSuccess)
    return SV_ECUDA;
  if (ev && cudaEventRecord(ev[1], ctx->stream) != cudaSuccess) return SV_ECUDA;
  if (sv::launch_tree_walk(ctx->dtype, vec, p, w, ctx->stream) != cudaSuccess) return SV_ECUDA;
  if (ev) {
    if (cudaEventRecord(ev[2], ctx->stream) != cudaSuccess) return SV_ECUDA;
    ctx->recorded += 1;
  }
  return SV_OK;
}

}  // namespace

int spec_verify_tree(spec_verify_ctx* ctx, int B, int M, int V, int mode,
                     const void* target_logits, const void* draft_logits, const int32_t* parents,
                     const int32_t* draft_tokens, const float* temperature, uint64_t seed,
                     int32_t* out_tokens, int32_t* out_path, int32_t* out_accept_len,
                     int32_t* out_kv_len) {
  return tree_call(ctx, false, B, M, V, mode, target_logits, draft_logits, parents, draft_tokens, temperature,
                   seed, out_tokens, out_path, out_accept_len, out_kv_len);
}

int spec_verify_tree_lazy(spec_verify_ctx* ctx, int B, int M, int V, int mode,
                          const void* target_logits, const void* draft_logits, const int32_t* parents,
                          const int32_t* draft_tokens, const float* temperature, uint64_t seed,
                          int32_t* out_tokens, int32_t* out_path, int32_t* out_accept_len,
                          int32_t* out_kv_len) {
  return tree_call(ctx, true, B, M, V, mode, target_logits, draft_logits, parents, draft_tokens, temperature,
                   seed, out_tokens, out_path, out_accept_len, out_kv_len);
}

int spec_verify_kv_commit(spec_verify_ctx* ctx, int mode, int L, int B, int S, int W,
                          size_t entry_bytes, const void* scratch, void* cache, int32_t* seq_len,
                          const int32_t* kv_len, const int32_t* path, int path_stride) {
  if (ctx == nullptr || (mode != SV_KV_SCRATCH && mode != SV_KV_INPLACE) || L < 0 || B < 0 ||
      S < 1 || entry_bytes == 0 || entry_bytes % 16 != 0)
    return SV_EINVAL;
  if (mode == SV_KV_SCRATCH && (W < 1 || scratch == nullptr || !aligned16(scratch)))
    return SV_EINVAL;
  if (path != nullptr && path_stride < 0) return SV_EINVAL;
  if (L == 0 || B == 0) return SV_OK;
  if (cache == nullptr || !aligned16(cache) || seq_len == nullptr || kv_len == nullptr)
    return SV_EINVAL;
  sv::KvProblem p;
  p.mode = mode;
  p.L = L;
  p.B = B;
  p.S = S;
  p.W = mode == SV_KV_SCRATCH ? W : 0;
  p.E = entry_bytes;
  p.scratch = scratch;
  p.cache = cache;
  p.seq_len = seq_len;
  p.kv_len = kv_len;
  p.path = path;
  p.path_stride = path_stride;
  p.err = ctx->w.err;
  return sv::launch_kv_commit(p, ctx->stream) == cudaSuccess ? SV_OK : SV_ECUDA;
}

int spec_verify_lazy(spec_verify_ctx* ctx, int B, int N, int V, const void* target_logits,
                     const void* draft_logits, const int32_t* draft_tokens,
                     const float* temperature, uint64_t seed, int32_t* out_tokens,
                     int32_t* out_accept_len, int32_t* out_kv_len) {
  if (ctx == nullptr) return SV_EINVAL;
  if (B < 0 || B > ctx->max_B || N < 0 || N > ctx->max_N || V < 1 || V > ctx->max_V)
    return SV_EINVAL;
  if (B == 0) return SV_OK;
  if (target_logits == nullptr || temperature == nullptr || out_tokens == nullptr ||
      out_accept_len == nullptr || out_kv_len == nullptr)
    return SV_EINVAL;
  if (N > 0 && (draft_logits == nullptr || draft_tokens == nullptr)) return SV_EINVAL;
  const size_t esize = ctx->dtype == SV_BF16 ? 2 : 4;
  const bool vec = (static_cast<size_t>(V) * esize) % 16 == 0 && aligned16(target_logits) &&
                   (N == 0 || aligned16(draft_logits));
  sv::Problem p;
  p.B = B;
  p.N = N;
  p.V = V;
  p.target = target_logits;
  p.draft = draft_logits;
  p.tokens = draft_tokens;
  p.temperature = temperature;
  p.seed = seed;
  p.out_tokens = out_tokens;
  p.out_accept = out_accept_len;
  p.out_kv = out_kv_len;
  p.epoch = 0;  // the lazy kernel reads its own partials after a CTA barrier
  sv::Workspace w = ctx->w;
  w.S1 = ceil_div(V, sv::row_chunk_elems(ctx->dtype));
  w.S3 = ceil_div(V, sv::sample_chunk_elems(ctx->dtype));
  cudaEvent_t* ev = nullptr;
  if (ctx->profile_every > 0 && (ctx->profile_seen++ % ctx->profile_every) == 0) {
    ev = profile_slot(ctx);
    if (ev == nullptr) return SV_ECUDA;
    if (cudaEventRecord(ev[0], ctx->stream) != cudaSuccess) return SV_ECUDA;
  }
  if (sv::launch_lazy(ctx->dtype, vec, p, w, ctx->stream) != cudaSuccess) return SV_ECUDA;
  if (ev) {  // one kernel: its time is reported as kernel 0, kernel 1 gets ~0
    if (cudaEventRecord(ev[1], ctx->stream) != cudaSuccess ||
        cudaEventRecord(ev[2], ctx->stream) != cudaSuccess)
      return SV_ECUDA;
    ctx->recorded += 1;
  }
  return SV_OK;
}

int spec_verify_fc_norm(spec_verify_ctx* ctx, int T, int d, int d_out, int norm, float eps,
                        const void* h_early, const void* h_mid, const void* h_late,
                        const float* gamma, const float* beta, const void* weight,
                        const float* bias, void* out, void* xbuf) {
  if (ctx == nullptr || T < 0 || d < 64 || d % 64 != 0 || d_out < 1 ||
      (norm != SV_NORM_NONE && norm != SV_NORM_LAYER && norm != SV_NORM_RMS) || !(eps >= 0.f) ||
      eps > 3.0e38f)
    return SV_EINVAL;
  if (static_cast<long long>(d) * 3 > (1LL << 30) || d_out > (1 << 28)) return SV_EINVAL;
  if (T == 0) return SV_OK;
  if (h_early == nullptr || h_mid == nullptr || h_late == nullptr || weight == nullptr ||
      out == nullptr || xbuf == nullptr || !aligned16(h_early) || !aligned16(h_mid) ||
      !aligned16(h_late) || !aligned16(weight) || !aligned16(xbuf))
    return SV_EINVAL;
  if (norm != SV_NORM_NONE && gamma == nullptr) return SV_EINVAL;
  sv::FcNormProblem p;
  p.T = T;
  p.d = d;
  p.d_out = d_out;
  p.norm = norm;
  p.eps = eps;
  p.h[0] = static_cast<const __nv_bfloat16*>(h_early);
  p.h[1] = static_cast<const __nv_bfloat16*>(h_mid);
  p.h[2] = static_cast<const __nv_bfloat16*>(h_late);
  p.gamma = gamma;
  p.beta = norm == SV_NORM_LAYER ? beta : nullptr;
  p.w = static_cast<const __nv_bfloat16*>(weight);
  p.bias = bias;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.out_vec = aligned16(out) && d_out % 8 == 0;
  p.gb_vec = (norm == SV_NORM_NONE || aligned16(gamma)) && (p.beta == nullptr || aligned16(p.beta));
  p.x = static_cast<__nv_bfloat16*>(xbuf);
  p.err = ctx->w.err;
  return sv::launch_fcnorm(p, ctx->stream) == cudaSuccess ? SV_OK : SV_ECUDA;
}

int spec_verify_get_error(spec_verify_ctx* ctx, uint32_t* bits) {
  if (ctx == nullptr) return SV_EINVAL;
  unsigned word = 0;
  if (cudaMemcpyAsync(&word, ctx->w.err, sizeof(word), cudaMemcpyDeviceToHost, ctx->stream) !=
          cudaSuccess ||
      cudaMemsetAsync(ctx->w.err, 0, sizeof(unsigned), ctx->stream) != cudaSuccess ||
      cudaStreamSynchronize(ctx->stream) != cudaSuccess)
    return SV_ECUDA;
  if (bits) *bits = word;
  if (word & SV_ERRBIT_TEMP) return SV_EBADTEMP;
  if (word & SV_ERRBIT_TREE) return SV_EBADTREE;
  if (word & SV_ERRBIT_TOKEN) return SV_EBADTOKEN;
  if (word & SV_ERRBIT_LOGIT) return SV_EBADLOGIT;
  if (word & SV_ERRBIT_KV) return SV_EBADKV;
  if (word & SV_ERRBIT_WAIT) return SV_ETIMEOUT;
  return SV_OK;
}

int spec_verify_debug_stats(spec_verify_ctx* ctx, int B, int N, float* accept_prob,
                            float* log_z) {
  if (ctx == nullptr || B < 1 || B > ctx->max_B || N < 0 || N > ctx->max_N) return SV_EINVAL;
  if (N > 0 && accept_prob != nullptr &&
      cudaMemcpyAsync(accept_prob, ctx->w.dbg_accept, sizeof(float) * B * N,
                      cudaMemcpyDeviceToDevice, ctx->stream) != cudaSuccess)
    return SV_ECUDA;
  if (log_z != nullptr &&
      cudaMemcpyAsync(log_z, ctx->w.dbg_logz, sizeof(float) * B * (2 * N + 1),
                      cudaMemcpyDeviceToDevice, ctx->stream) != cudaSuccess)
    return SV_ECUDA;
  return SV_OK;
}

int spec_verify_profile(spec_verify_ctx* ctx, int every) {
  if (ctx == nullptr || every < 0) return SV_EINVAL;
  if (every == 0 && ctx->profile_every > 0 && flush_profile(ctx) != SV_OK) return SV_ECUDA;
  ctx->profile_every = every;
  ctx->profile_seen = 0;
  return SV_OK;
}

int spec_verify_profile_read(spec_verify_ctx* ctx, double* ms_per_kernel, int* calls) {
  if (ctx == nullptr) return SV_EINVAL;
  if (flush_profile(ctx) != SV_OK) return SV_ECUDA;
  for (int k = 0; k < SV_NUM_KERNELS; ++k) {
    if (ms_per_kernel) ms_per_kernel[k] = ctx->ms[k];
    ctx->ms[k] = 0.0;
  }
  if (calls) *calls = ctx->calls;
  ctx->calls = 0;
  return SV_OK;
}

int spec_verify_destroy(spec_verify_ctx* ctx) {
  if (ctx == nullptr) return SV_OK;
  int rc = SV_OK;
  if (cudaStreamSynchronize(ctx->stream) != cudaSuccess) rc = SV_ECUDA;
  for (cudaEvent_t e : ctx->events) cudaEventDestroy(e);
  if (cudaFree(ctx->ws) != cudaSuccess) rc = SV_ECUDA;
  delete ctx;
  return rc;
}

int spec_verify_debug_skip_row_stats(spec_verify_ctx* ctx, int on) {
  if (ctx == nullptr) return SV_EINVAL;
  ctx->skip_rowstats = on != 0;
  return SV_OK;
}

int spec_verify_debug_late_cta(spec_verify_ctx* ctx, int cta) {
  if (ctx == nullptr || cta < -1) return SV_EINVAL;
  ctx->late_cta = cta;
  return SV_OK;
}

int spec_verify_debug_seek_calls(spec_verify_ctx* ctx, uint32_t calls) {
  if (ctx == nullptr) return SV_EINVAL;
  ctx->epoch = calls;
  return SV_OK;
}

/* Test hook: Philox4x32-10 words for n counters (c0, c1, c2, 0) under a
 * 64-bit seed, computed by the same device function the walk uses.
 * ctr3: device [n, 3] uint32; out4: device [n, 4] uint32. */
int spec_verify_debug_philox(uint64_t seed, const uint32_t* ctr3, uint32_t* out4, int n,
                             void* cuda_stream) {
  if (n < 0 || (n > 0 && (ctr3 == nullptr || out4 == nullptr))) return SV_EINVAL;
  return sv::launch_philox_probe(seed, ctr3, out4, n, static_cast<cudaStream_t>(cuda_stream)) ==
                 cudaSuccess
             ? SV_OK
             : SV_ECUDA;
}

int spec_verify_debug_read_stream(const void* buf, size_t bytes, uint64_t* out_sum, void* cuda_stream) {
  if (out_sum == nullptr || bytes % 16 != 0 || (bytes > 0 && (buf == nullptr || !aligned16(buf))))
    return SV_EINVAL;
  return sv::launch_read_stream(buf, bytes, reinterpret_cast<unsigned long long*>(out_sum),
                                static_cast<cudaStream_t>(cuda_stream)) == cudaSuccess
             ? SV_OK
             : SV_ECUDA;
}

}  // extern "C"
