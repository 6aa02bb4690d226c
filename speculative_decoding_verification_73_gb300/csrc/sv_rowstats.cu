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
// one CTA-wide merge per span) and writes partials[row][span] tagged with
// the call's sequence number, in one 128-bit store: the sampler polls the
// tags of its own request, so it can start on a request whose rows are done
// while later rows are still streaming.  The CTA whose span holds the row's
// draft token puts that token's logit in the same partial, so the walk
// never reads the logits again.  Rows that are not 16-byte aligned
// take a scalar two-pass path over the same spans.  Small per-thread state
// and groups of two loads keep eight CTAs resident per SM, which measured
// best (more warps in flight, fewer registers per byte in flight).

#include <climits>
#include <cuda_bf16.h>

#include "sv_device.cuh"
#include "sv_span.cuh"

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
  __shared__ float s_tok;  // the logit at d, set by the thread whose vector holds it
  float* tok = &s_tok;
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
  if (threadIdx.x == 0) {
    // the reductions above end in CTA barriers, so s_tok is visible here
    if (!greedy) out.idx = (d >= beg && d < end) ? __float_as_int(s_tok) : 0;
    out.tag = p.epoch;
    st_partial_relaxed(w.partials + static_cast<size_t>(row) * S1 + span, out);
  }
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
