// Internal declarations shared by the kernels and the C-ABI layer of
// libspecverify.  Nothing here is part of the public interface.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace sv {

constexpr int kThreads = 256;           // threads per CTA, every kernel
// Tuning constants of the row-statistics kernel; each can be overridden at
// build time with -D<name>=<value> (the build script's `defines`).
#ifndef SV_SPAN_BYTES
#define SV_SPAN_BYTES 65536
#endif
#ifndef SV_GROUP
#define SV_GROUP 2
#endif
#ifndef SV_SPAN_MINB
#define SV_SPAN_MINB 8
#endif
constexpr int kSpanBytes = SV_SPAN_BYTES;      // bytes of a row one CTA reduces
constexpr int kGroup = SV_GROUP;               // 16-byte loads per thread per group
constexpr int kSpanMinBlocks = SV_SPAN_MINB;   // resident CTAs per SM the kernel is built for
constexpr int kLevel1 = 8192;           // tokens per level-1 block of the grouped inverse CDF
constexpr int kLevel2 = 256;            // tokens per level-2 block
constexpr int kLevel3 = 16;             // tokens per level-3 block
constexpr int kSampleThreads = 256;     // sampler: threads per CTA (one CTA per level-1 block)
// The walk runs on a sampler CTA, one thread per row of a request, so
// N + 1 <= kSampleThreads (the API caps N at 255).

constexpr int kModeInvalid = 0;
constexpr int kModeGreedy = 1;
constexpr int kModeSampled = 2;

constexpr unsigned kErrTemp = 1u;
constexpr unsigned kErrToken = 2u;
constexpr unsigned kErrLogit = 4u;
constexpr unsigned kErrTree = 8u;
constexpr unsigned kErrKv = 16u;
constexpr unsigned kErrWait = 32u;

// FC-norm: how each target hidden state is normalised before the FC.
constexpr int kNormNone = 0;   // EAGLE-3
constexpr int kNormLayer = 1;  // LayerNorm (EAGLE 3.1)
constexpr int kNormRms = 2;    // RMSNorm

// How the verify window's KV entries were written.
constexpr int kKvScratch = 0;  // to a scratch window [L, B, W, E]
constexpr int kKvInplace = 1;  // into the cache right after each sequence's length

// How the children of a draft-tree node were drafted.
constexpr int kTreeSampled = 0;  // independent draws from the node's draft row
constexpr int kTreeTopk = 1;     // fixed candidates (point masses)

// Statistics of one chunk of one logit row (16 bytes, 16-byte aligned).
//   sampled row: a = c = fl(M * k) with M the chunk maximum and k = log2(e)/T,
//                s = sum over the chunk of 2^(x*k - c)   (NaN marks a bad chunk)
//                idx = bits of the float logit at the row's draft token when
//                the chunk holds it (chain kernel), else 0
//   greedy row : a = chunk maximum M, s = 0 (NaN if a NaN was seen),
//                idx = lowest index holding M
//   tag        : the call's sequence number (never 0) in the chain's and the
//                tree's row statistics; the lazy kernel writes 0.  The whole
//                partial is stored with one 128-bit access and the chain
//                sampler / tree walk polls for its tag, so it can start on a
//                request whose rows are done while the rest of the grid
//                still runs.
struct Partial {
  float a;
  float s;
  int idx;
  unsigned tag;
};

constexpr int kJobNone = 0;
constexpr int kJobResidual = 1;
constexpr int kJobBonus = 2;
constexpr int kJobLate = 3;  // a sampled request whose wait ran out in this CTA
constexpr int kJobFailed = 4;  // a sampled request failed by its inputs (token, logit)

// What the walk leaves for the sampler (in shared memory of each CTA).
//   q_t = 2^(z_t*k - cq) * inv_sq,  p_t = 2^(y_t*k - cp) * inv_sp
struct Job {
  int kind;     // kJob*
  int row;      // 0-based row of the correction (first rejected) or bonus row
  float u[4];   // uniforms of the sampling draw, one per level
  float k;      // log2(e) / T
  float cq, inv_sq;
  float cp, inv_sp;
};

struct Problem {
  int B, N, V;
  const void* target;        // [B, N+1, V]
  const void* draft;         // [B, N, V]
  const int32_t* tokens;     // [B, N]
  const float* temperature;  // [B]
  unsigned long long seed;
  int32_t* out_tokens;       // [B, N+1]
  int32_t* out_accept;       // [B]
  int32_t* out_kv;           // [B]
  unsigned epoch;            // tag of this call's row-statistics partials (never 0)
  int debug_late_cta = -1;   // test hook: the sampler CTA (index within its request)
                             // that acts as if its waits ran out; -1 = none
};

struct TreeProblem {
  int B, M, V, mode;         // mode: kTreeSampled | kTreeTopk
  const void* target;        // [B, M+1, V]: row r after node r
  const void* draft;         // [B, M+1, V]: row r drafted node r's children
  const int32_t* parents;    // [B, M]: parent of node i+1, in [0, i]
  const int32_t* tokens;     // [B, M]
  const float* temperature;  // [B]
  unsigned long long seed;
  int32_t* out_tokens;       // [B, M+1]
  int32_t* out_path;         // [B, M]
  int32_t* out_accept;       // [B]
  int32_t* out_kv;           // [B]
  unsigned epoch;            // tag of this call's row-statistics partials (never 0)
};

struct KvProblem {
  int mode, L, B, S, W;
  size_t E;                  // bytes per (layer, sequence, position); multiple of 16
  const void* scratch;       // [L, B, W, E] (scratch mode)
  void* cache;               // [L, B, S, E]
  int32_t* seq_len;          // [B], in / out
  const int32_t* kv_len;     // [B]
  const int32_t* path;       // [B, path_stride] accepted node ids, or nullptr (chain)
  int path_stride;
  unsigned* err;
};

struct FcNormProblem {
  int T, d, d_out, norm;
  float eps;
  const __nv_bfloat16* h[3];   // [T, d] each: early, middle, late layer
  const float* gamma;          // [3, d]
  const float* beta;           // [3, d] or nullptr
  const __nv_bfloat16* w;      // [d_out, 3d]
  const float* bias;           // [d_out] or nullptr
  __nv_bfloat16* out;          // [T, d_out]
  bool out_vec;                // rows of out 16-byte aligned
  bool gb_vec;                 // gamma and beta (when given) 16-byte aligned
  __nv_bfloat16* x;            // [T, 3d]: the normalised, concatenated input (scratch)
  unsigned* err;
};

struct Workspace {
  Partial* partials;     // [B][2N+1][S1]: target rows 0..N, then draft rows 0..N-1
                         // (tree: [B][2(M+1)][S1], target rows then draft rows 0..M)
  float* tok_logit;      // [B][2N+1]: logit at the row's draft token (sampled rows)
  float* chunk_sums;     // [B, S3]: residual mass of each level-1 block
  int* blk_tok;          // [B, S3]: the token each level-1 block would give
  unsigned* err;         // [1], OR of kErr* bits (starts at zero)
  unsigned long long* arrivals;  // [B]: sampler arrivals per request, (late arrivals << 32) |
                                 // count; zero between calls (the last CTA clears it)
  unsigned* late;        // [B]: tree walk: the call's tag once a wait of the request ran out
  float* dbg_accept;     // [B, N]
  float* dbg_logz;       // [B, 2N+1]
  int S1;                // spans per row for this call's V
  int S3;                // level-1 blocks per row for this call's V
};

// dtype codes match SV_F32 / SV_BF16; vec selects 16-byte loads (aligned rows).
cudaError_t launch_rowstats(int dtype, bool vec, const Problem& p, const Workspace& w,
                            cudaStream_t s);
cudaError_t launch_sample(int dtype, bool vec, const Problem& p, const Workspace& w,
                          cudaStream_t s);
cudaError_t launch_tree_rowstats(int dtype, bool vec, const TreeProblem& p, const Workspace& w,
                                 cudaStream_t s);
cudaError_t launch_tree_walk(int dtype, bool vec, const TreeProblem& p, const Workspace& w,
                             cudaStream_t s);
// The lazy tree walk alone (no row-statistics grid): rows of at most
// kTreeLazyMaxSpans spans.
constexpr int kTreeLazyMaxSpans = 32;
cudaError_t launch_tree_lazy(int dtype, bool vec, const TreeProblem& p, const Workspace& w,
                             cudaStream_t s);
cudaError_t launch_kv_commit(const KvProblem& p, cudaStream_t s);
cudaError_t launch_fcnorm(const FcNormProblem& p, cudaStream_t s);
cudaError_t launch_lazy(int dtype, bool vec, const Problem& p, const Workspace& w, cudaStream_t s);
cudaError_t launch_read_stream(const void* buf, size_t bytes, unsigned long long* out, cudaStream_t s);
cudaError_t launch_philox_probe(unsigned long long seed, const uint32_t* ctr3, uint32_t* out4,
                                int n, cudaStream_t s);

inline int row_chunk_elems(int dtype) { return kSpanBytes / (dtype == 1 ? 2 : 4); }

inline int sample_chunk_elems(int) { return kLevel1; }

}  // namespace sv
