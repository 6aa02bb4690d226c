// KV-cache commit after verification ("Speculative Decoding and EAGLE-3"
// lesson, section "KV cache rollback", and exercise 4): keep the window
// entries of the verified input token and the accepted drafts, drop the
// rest, and advance each sequence's logical length by out_kv_len.
//
// Cache [L, B, S, E bytes], window [L, B, W, E].  Kept window positions:
// 0, then 1, 2, ... (chain) or the accepted node ids out_path[b, :] (tree),
// out_kv_len[b] of them.  SCRATCH: kept position i is copied from the
// scratch window to cache position seq_len + i.  IN-PLACE: the window was
// written at cache positions seq_len + w; kept position i moves from
// seq_len + pos_i to seq_len + i (pos_i >= i because kept positions rise, so
// a thread that walks i upwards never reads an entry it has already
// overwritten); entries already in place are not touched.  A sequence whose
// commit would pass S, read outside the window, or whose kept positions do
// not rise is left unchanged and flagged.
//
// kv_commit_kernel: a grid of at most kKvCtasPerSm CTAs per SM (40
// registers, six resident per SM) takes the (layer, sequence) entries in
// turn; one thread per 16-byte column copies the kept positions four at a
// time (four loads in flight per thread) -- a plain bandwidth-bound copy
// with coalesced 16-byte accesses (consecutive threads, consecutive
// columns).  kv_advance_kernel
// then moves the lengths: a second grid, launched with programmatic
// dependent launch so that it is resident while the copy drains, whose
// griddepcontrol.wait returns only once the copy grid has completed and its
// writes are visible -- so no CTA of the copy can read a length already
// advanced.  The copy is itself a programmatic dependent of the grid before
// it and waits for that grid the same way.  (Measured per commit of 32
// layers x 64 sequences x 4 KB: 13.44 us as built; eight entries per batch
// at 74 registers, 3 CTAs per SM: 14.73 us; four per batch at 32 registers:
// 14.58 us; a CTA per sequence and group of four layers 18.1 us; one launch
// whose last CTA advances the lengths 16.9 us; one launch counting per
// sequence, the entry completing the count advancing the length, 21.6 us;
// one launch with a cluster of 8 CTAs per sequence, rank 0 handing the
// length to the others through distributed shared memory, 15.65 us.)

#include <cstdint>

#include "sv_device.cuh"

namespace sv {
namespace {

constexpr int kKvThreads = 256;
// Kept entries copied per batch (loads in flight per thread), and resident
// CTAs per SM the copy kernel is built for; build-time overrides
// -DSV_KV_BATCH=<n>, -DSV_KV_MINB=<n>.
#ifndef SV_KV_BATCH
#define SV_KV_BATCH 4
#endif
#ifndef SV_KV_MINB
#define SV_KV_MINB 6
#endif
constexpr int kKvBatch = SV_KV_BATCH;
// CTAs per SM of the copy grid (more items than that are taken in turn);
// build-time override -DSV_KV_CTAS_PER_SM=<n>.
#ifndef SV_KV_CTAS_PER_SM
#define SV_KV_CTAS_PER_SM 12
#endif
constexpr int kKvCtasPerSm = SV_KV_CTAS_PER_SM;

// Window position of kept entry i, or -1 past the path.
__device__ __forceinline__ int kept_pos(const KvProblem& p, int b, int i) {
  if (i == 0) return 0;
  if (p.path == nullptr) return i;
  return p.path[static_cast<size_t>(b) * p.path_stride + (i - 1)];
}

// Whether sequence b's commit is valid (the same answer in every thread).
__device__ __forceinline__ bool commit_ok(const KvProblem& p, int b, int n, int start) {
  if (start < 0 || static_cast<long long>(start) + n > p.S) return false;
  if (p.path != nullptr && n - 1 > p.path_stride) return false;
  const int width = p.mode == kKvScratch ? p.W : p.S - start;
  int prev = -1;
  for (int i = 0; i < n; ++i) {
    const int w = kept_pos(p, b, i);
    if (w <= prev || w >= width) return false;
    prev = w;
  }
  return true;
}

// Copy the kept window entries of one (layer, sequence, column slice) item.
template <bool kScratch>
__device__ __forceinline__ void commit_item(const KvProblem& p, long long item, long long slices,
                                            long long cols) {
  const long long lb = item / slices;
  const long long col = (item - lb * slices) * kKvThreads + threadIdx.x;
  const int l = static_cast<int>(lb / p.B);
  const int b = static_cast<int>(lb - static_cast<long long>(l) * p.B);
  const int n = p.kv_len[b];
  if (n <= 0) return;
  const int start = p.seq_len[b];
  if (!commit_ok(p, b, n, start)) {
    if (l == 0 && col == 0) atomicOr(p.err, kErrKv);
    return;
  }
  if (col >= cols) return;
  const size_t E = p.E;
  unsigned char* cache = static_cast<unsigned char*>(p.cache) +
                         (static_cast<size_t>(l) * p.B + b) * p.S * E + static_cast<size_t>(start) * E +
                         static_cast<size_t>(col) * 16;
  const unsigned char* src = kScratch
                                 ? static_cast<const unsigned char*>(p.scratch) +
                                       (static_cast<size_t>(l) * p.B + b) * p.W * E + static_cast<size_t>(col) * 16
                                 : cache;
  // kKvBatch kept entries at a time: all their loads in flight before any
  // store.  In place this is still safe: a batch reads positions
  // pos_i >= i, above every position written so far or by this batch.
  for (int i0 = 0; i0 < n; i0 += kKvBatch) {
    uint4 v[kKvBatch];
    int w[kKvBatch];
#pragma unroll
    for (int k = 0; k < kKvBatch; ++k) {
      const int i = i0 + k;
      w[k] = i < n ? kept_pos(p, b, i) : i;
      if (i < n && (kScratch || w[k] != i))
        v[k] = kScratch ? ld_stream16(src + static_cast<size_t>(w[k]) * E)
                        : *reinterpret_cast<const uint4*>(src + static_cast<size_t>(w[k]) * E);
    }
#pragma unroll
    for (int k = 0; k < kKvBatch; ++k) {
      const int i = i0 + k;
      if (i < n && (kScratch || w[k] != i))  // entries already in place are not touched
        *reinterpret_cast<uint4*>(cache + static_cast<size_t>(i) * E) = v[k];
    }
  }
}

// The copy grid: at most kKvCtasPerSm CTAs per SM, each taking the
// (layer, sequence, column slice) items in turn.
template <bool kScratch>
__global__ void __launch_bounds__(kKvThreads, SV_KV_MINB) kv_commit_kernel(KvProblem p) {
  // Launched as a programmatic dependent of whatever precedes it: wait for
  // that grid (it may be the verify step writing kv_len, or the previous
  // commit's length update) before reading anything.
  wait_for_prerequisite();
  allow_dependents();  // the length update may be scheduled behind the last wave
  const long long cols = static_cast<long long>(p.E / 16);
  const long long slices = (cols + kKvThreads - 1) / kKvThreads;
  const long long items = static_cast<long long>(p.L) * p.B * slices;
  for (long long it = blockIdx.x; it < items; it += gridDim.x) commit_item<kScratch>(p, it, slices, cols);
}

__global__ void kv_advance_kernel(KvProblem p) {
  allow_dependents();       // a following commit may be scheduled early (it waits too)
  wait_for_prerequisite();  // the copy grid has completed
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= p.B) return;
  const int n = p.kv_len[b];
  if (n <= 0) return;
  const int start = p.seq_len[b];
  if (commit_ok(p, b, n, start)) p.seq_len[b] = start + n;
}

}  // namespace

cudaError_t launch_kv_commit(const KvProblem& p, cudaStream_t s) {
  if (p.B <= 0 || p.L <= 0) return cudaSuccess;
  const long long cols = static_cast<long long>(p.E / 16);
  const long long items = static_cast<long long>(p.L) * p.B * ((cols + kKvThreads - 1) / kKvThreads);
  int dev = 0, sms = 0;
  cudaError_t e0;
  if ((e0 = cudaGetDevice(&dev)) != cudaSuccess ||
      (e0 = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e0;
  const long long cap = static_cast<long long>(sms) * kKvCtasPerSm;
  const long long blocks = items < cap ? items : cap;
  // Both launches are programmatic dependents of the grid before them; each
  // kernel waits for that grid before it reads what the grid writes.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kKvThreads);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (blocks > 0) {
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    const cudaError_t e = p.mode == kKvScratch ? cudaLaunchKernelEx(&cfg, kv_commit_kernel<true>, p)
                                               : cudaLaunchKernelEx(&cfg, kv_commit_kernel<false>, p);
    if (e != cudaSuccess) return e;
  }
  cfg.gridDim = dim3(static_cast<unsigned>((p.B + kKvThreads - 1) / kKvThreads));
  return cudaLaunchKernelEx(&cfg, kv_advance_kernel, p);
}

}  // namespace sv
