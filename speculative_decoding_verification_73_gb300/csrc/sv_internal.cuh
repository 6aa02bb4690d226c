// Internal declarations shared by the kernels and the C-ABI layer of
// libspecverify.  Nothing here is part of the public interface.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

constexpr int kThreads = 256;           // threads per CTA, every kernel
// Tuning constants of the row-statistics kernels; each can be overridden at
// build time with -D<name>=<value> (the build script's `defines`).
#ifndef SV_SPAN_BYTES
#define SV_SPAN_BYTES 65536
#endif
#ifndef SV_GROUP
#define SV_GROUP 4
#endif
#ifndef SV_SPAN_MINB
#define SV_SPAN_MINB 5
#endif
#ifndef SV_STREAM_CTAS
#define SV_STREAM_CTAS 2
#endif
#ifndef SV_STREAM_STAGES
#define SV_STREAM_STAGES 5
#endif
#ifndef SV_STREAM_RANGES
#define SV_STREAM_RANGES 1
#endif
#ifndef SV_LAYOUT
#define SV_LAYOUT 0
#endif
constexpr int kSpanBytes = SV_SPAN_BYTES;      // span kernel: bytes of a row one CTA reduces
constexpr int kGroup = SV_GROUP;               // 16-byte loads per thread per group
constexpr int kSpanMinBlocks = SV_SPAN_MINB;   // span kernel: resident CTAs per SM it is built for
constexpr int kStreamMaxB = 2048;              // stream kernel keeps per-request row counts in smem
constexpr int kStreamCtasPerSm = SV_STREAM_CTAS;   // stream kernel: resident CTAs per SM
constexpr int kStreamStages = SV_STREAM_STAGES;    // stream kernel: cp.async groups per warp
constexpr int kStreamRanges = SV_STREAM_RANGES;    // stream kernel: byte ranges per warp
constexpr int kLayoutChoice = SV_LAYOUT;       // 0 automatic, 1 span only, 2 stream when possible
constexpr int kLevel1 = 8192;           // tokens per level-1 block of the grouped inverse CDF
constexpr int kLevel2 = 256;            // tokens per level-2 block
constexpr int kLevel3 = 16;             // tokens per level-3 block
constexpr int kSampleCluster = 8;       // sampler: CTAs (one cluster) per request
// The walk runs on a CTA of kThreads threads, one thread per row of a
// request, so N + 1 <= kThreads.

constexpr int kModeInvalid = 0;
constexpr int kModeGreedy = 1;
constexpr int kModeSampled = 2;

constexpr unsigned kErrTemp = 1u;
constexpr unsigned kErrToken = 2u;
constexpr unsigned kErrLogit = 4u;

// Statistics of one chunk of one logit row (16 bytes).
//   sampled row: a = c = fl(M * k) with M the chunk maximum and k = log2(e)/T,
//                s = sum over the chunk of 2^(x*k - c)   (NaN marks a bad chunk)
//   greedy row : a = chunk maximum M, s = 0 (NaN if a NaN was seen),
//                idx = lowest index holding M
struct Partial {
  float a;
  float s;
  int idx;
  int pad;
};

constexpr int kJobNone = 0;
constexpr int kJobResidual = 1;
constexpr int kJobBonus = 2;

// What the walk leaves for the sampler (in shared memory of each CTA).
//   q_t = 2^(z_t*k - cq) * inv_sq
//   log2(q_t / p_t) = (z_t - y_t)*k - (dhi + dlo)
struct Job {
  int kind;     // kJob*
  int row;      // 0-based row of the correction (first rejected) or bonus row
  float u[4];   // uniforms of the sampling draw, one per level
  float k;      // log2(e) / T
  float cq, inv_sq;
  float dhi, dlo;
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
};

constexpr int kLayoutSpan = 0;    // partials[b][2N+1][S1]
constexpr int kLayoutStream = 1;  // partials[range][2], see sv_rowstats.cu

struct Workspace {
  Partial* partials;     // row-statistics partials, laid out as `layout` says
  unsigned* row_prefix;  // [B+1] stream layout: active rows before request b
  float* tok_logit;      // [B][2N+1] stream layout: logit at the row's draft token
  float* chunk_sums;     // [B, S3]: residual mass of each level-1 block
  unsigned* err;         // [1], OR of kErr* bits
  float* dbg_accept;     // [B, N]
  float* dbg_logz;       // [B, 2N+1]
  int layout;            // kLayout*
  int S1;                // span layout: spans per row for this call's V
  int stream_warps;      // stream layout: warps of the row-statistics launch
  int S3;                // level-1 blocks per row for this call's V
};

// Byte ranges of the stream layout.  The active rows (target rows 0..N of
// every valid request, draft rows 0..N-1 of sampled ones; request-major) are
// concatenated into one byte stream of total = rows * row_bytes bytes, cut
// into ranges of range_bytes (a multiple of 16, at most one row) so that
// every warp of the launch gets kStreamRanges ranges, spread over the stream
// (warp w takes ranges w, w + warps, ...), or more when rows are small.
// Range rho covers [rho * range_bytes, ...) and touches at most two rows;
// its partial for the first row it touches is partials[2 rho], for the
// second partials[2 rho + 1].
__host__ __device__ inline unsigned long long stream_range_bytes(unsigned long long total,
                                                                 unsigned long long row_bytes,
                                                                 unsigned long long warps) {
  const unsigned long long parts = warps * static_cast<unsigned long long>(kStreamRanges);
  unsigned long long r = ((total + parts - 1) / parts + 15) / 16 * 16;
  if (r > row_bytes) r = row_bytes;
  return r < 16 ? 16 : r;
}

// dtype codes match SV_F32 / SV_BF16; vec selects 16-byte loads (aligned rows).
// The layout and stream_warps fields of w must match what the launch uses:
// stream layout iff vec && B <= kStreamMaxB, with stream_warps = grid * 8.
cudaError_t launch_rowstats(int dtype, bool vec, const Problem& p, const Workspace& w,
                            cudaStream_t s);
cudaError_t prepare_rowstats();  // once per device, before the first launch
cudaError_t launch_sample(int dtype, bool vec, const Problem& p, const Workspace& w,
                          cudaStream_t s);
cudaError_t launch_philox_probe(unsigned long long seed, const uint32_t* ctr3, uint32_t* out4,
                                int n, cudaStream_t s);

inline int row_chunk_elems(int dtype) { return kSpanBytes / (dtype == 1 ? 2 : 4); }
inline int sample_chunk_elems(int) { return kLevel1; }

}  // namespace sv
