// Test hook: Philox4x32-10 words computed by the device function the walk
// and the sampler use, for checking against an independent implementation.

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

}  // namespace

cudaError_t launch_philox_probe(unsigned long long seed, const uint32_t* ctr3, uint32_t* out4,
                                int n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  philox_probe_kernel<<<(n + 255) / 256, 256, 0, s>>>(seed, ctr3, out4, n);
  return cudaGetLastError();
}

}  // namespace sv
