// Test hooks: Philox4x32-10 words computed by the device function the walk
// and the sampler use, for checking against an independent implementation;
// and a plain streaming read of a buffer (the achievable read bandwidth the
// row statistics are compared with), folding what it reads into a checksum
// so that no load can be dropped.

#include "sv_device.cuh"

namespace sv {
namespace {

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

// Sum of the buffer's 64-bit words (mod 2^64): every thread reads 16-byte
// vectors i, i + stride, ... with non-allocating loads, four in flight; the
// CTA adds up its threads' totals and adds the result to *out once (one
// atomic per CTA, so the atomics on the one word stay few).
__global__ void __launch_bounds__(256) read_stream_kernel(const uint4* __restrict__ src, size_t n16,
                                                          unsigned long long* out) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  unsigned long long acc = 0;
  auto fold = [](const uint4& v) {
    return (static_cast<unsigned long long>(v.y) << 32 | v.x) + (static_cast<unsigned long long>(v.w) << 32 | v.z);
  };
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = ld_stream16(src + i), b = ld_stream16(src + i + stride);
    const uint4 c = ld_stream16(src + i + 2 * stride), d = ld_stream16(src + i + 3 * stride);
    acc += fold(a) + fold(b) + fold(c) + fold(d);
  }
  for (; i < n16; i += stride) acc += fold(ld_stream16(src + i));
#pragma unroll
  for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
  __shared__ unsigned long long s_warp[256 / 32];
  if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long t = 0;
#pragma unroll
    for (int w = 0; w < 256 / 32; ++w) t += s_warp[w];
    atomicAdd(out, t);
  }
}

}  // namespace

cudaError_t launch_read_stream(const void* buf, size_t bytes, unsigned long long* out, cudaStream_t s) {
  if (bytes == 0) return cudaSuccess;
  cudaError_t e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  read_stream_kernel<<<sms * 8, 256, 0, s>>>(static_cast<const uint4*>(buf), bytes / 16, out);
  return cudaGetLastError();
}

cudaError_t launch_philox_probe(unsigned long long seed, const uint32_t* ctr3, uint32_t* out4,
                                int n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  philox_probe_kernel<<<(n + 255) / 256, 256, 0, s>>>(seed, ctr3, out4, n);
  return cudaGetLastError();
}

}  // namespace sv
