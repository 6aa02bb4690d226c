// spec_verify_noalloc: the verify step without a context and without any
// device allocation by the library.
//
// Who needs it: callers that may not allocate device memory on the verify
// path.  A serving runtime that carves all of HBM into its own pools (KV
// cache blocks, activations) up front leaves nothing for a library's
// cudaMalloc, and a cudaMalloc or cudaFree in the middle of a decode loop
// also synchronises the device.  Such callers cannot keep a spec_verify_ctx,
// whose creation allocates the workspace.
//
// How: the working memory of one call (row-statistics partials, token
// logits, the sampler's per-block masses, candidates and arrival counters,
// the error word and the debug statistics) lives in g_scratch, a file-scope
// device array of SV_NOALLOC_SCRATCH_BYTES that exists in every device's
// copy of the module.  Host code cannot use the array's name as a device
// pointer, so the first call on each device (with that device current) asks
// the runtime for its address with cudaGetSymbolAddress and caches it; later
// calls on that device reuse the cached pointer.  Problems whose working memory does
// not fit are refused with SV_ESCRATCH before anything is enqueued.
//
// Sharing: every call on a device uses the same array.  The row-statistics
// partials (whose tags the sampler polls), the error word and the arrival
// counters have to start at zero; each call clears that front part of the
// array on its stream before its kernels run, in one memset.  Two calls whose kernels overlap in
// time (different streams without ordering between them, or host threads
// racing on one stream) corrupt each other's scratch and results.

#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/spec_verify.h"
#include "sv_internal.cuh"

namespace {

constexpr size_t kScratchBytes = SV_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Byte offsets of the workspace parts inside g_scratch for one problem; the
// same order and 256-byte alignment as the context workspace.
struct Carve {
  size_t part, tok, sums, btok, err, arr, acc, logz, end;
};

Carve carve(size_t B, size_t N, int s1, int s3) {
  const size_t rows = B * (2 * N + 1);
  Carve c;
  size_t off = 0;
  c.part = off;
  off = align_up(off + rows * s1 * sizeof(sv::Partial), 256);
  c.tok = off;
  off = align_up(off + rows * sizeof(float), 256);
  c.sums = off;
  off = align_up(off + B * s3 * sizeof(float), 256);
  c.btok = off;
  off = align_up(off + B * s3 * sizeof(int), 256);
  c.err = off;
  off = align_up(off + sizeof(unsigned), 256);
  c.arr = off;
  off = align_up(off + B * sizeof(unsigned long long), 256);
  c.acc = off;
  off = align_up(off + B * (N > 0 ? N : 1) * sizeof(float), 256);
  c.logz = off;
  off = align_up(off + rows * sizeof(float), 256);
  c.end = off;
  return c;
}

// Device address of g_scratch on the current device, looked up once per
// device; nullptr when the runtime call fails.
void* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" {

int spec_verify_noalloc(int B, int N, int V, sv_dtype dtype, const void* target_logits,
                        const void* draft_logits, const int32_t* draft_tokens,
                        const float* temperature, uint64_t seed, int32_t* out_tokens,
                        int32_t* out_accept_len, int32_t* out_kv_len, void* cuda_stream) {
  if (B < 0 || N < 0 || N > SV_MAX_N || V < 1 || V > SV_MAX_V ||
      (dtype != SV_F32 && dtype != SV_BF16))
    return SV_EINVAL;
  if (B == 0) return SV_OK;
  if (target_logits == nullptr || temperature == nullptr || out_tokens == nullptr ||
      out_accept_len == nullptr || out_kv_len == nullptr)
    return SV_EINVAL;
  if (N > 0 && (draft_logits == nullptr || draft_tokens == nullptr)) return SV_EINVAL;

  sv::Workspace w;
  w.S1 = ceil_div(V, sv::row_chunk_elems(dtype));
  w.S3 = ceil_div(V, sv::sample_chunk_elems(dtype));
  const Carve c = carve(static_cast<size_t>(B), static_cast<size_t>(N), w.S1, w.S3);
  if (c.end > kScratchBytes) return SV_ESCRATCH;
  char* base = static_cast<char*>(scratch_on_current_device());
  if (base == nullptr) return SV_ECUDA;
  w.partials = reinterpret_cast<sv::Partial*>(base + c.part);
  w.tok_logit = reinterpret_cast<float*>(base + c.tok);
  w.chunk_sums = reinterpret_cast<float*>(base + c.sums);
  w.blk_tok = reinterpret_cast<int*>(base + c.btok);
  w.err = reinterpret_cast<unsigned*>(base + c.err);
  w.arrivals = reinterpret_cast<unsigned long long*>(base + c.arr);
  w.late = nullptr;  // tree walks only
  w.dbg_accept = reinterpret_cast<float*>(base + c.acc);
  w.dbg_logz = reinterpret_cast<float*>(base + c.logz);

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
  p.epoch = 1;  // the partials were cleared just before (below)
  const size_t esize = dtype == SV_BF16 ? 2 : 4;
  const bool vec = (static_cast<size_t>(V) * esize) % 16 == 0 && aligned16(target_logits) &&
                   (N == 0 || aligned16(draft_logits));
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  // The partials (tags 0: not yet written by this call), token logits,
  // block sums, the error word and the arrival counters start at zero.  The
  // parts move with the problem's shape, so whatever an earlier call left
  // there could otherwise pass for a tag of this call.
  if (cudaMemsetAsync(base, 0, c.acc, s) != cudaSuccess) return SV_ECUDA;
  if (sv::launch_rowstats(dtype, vec, p, w, s) != cudaSuccess) return SV_ECUDA;
  if (sv::launch_sample(dtype, vec, p, w, s) != cudaSuccess) return SV_ECUDA;
  return SV_OK;
}

}  // extern "C"
