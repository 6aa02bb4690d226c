// Device-side helpers of libspecverify: element access, streaming loads,
// block reductions, the temperature rule and Philox4x32-10.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "sv_internal.cuh"

namespace sv {

constexpr unsigned kFull = 0xffffffffu;

// ------------------------------------------------- dependent launches
// Programmatic dependent launch (PTX griddepcontrol).  A kernel launched
// with the programmatic-serialisation attribute may start while the kernel
// before it in the stream is still running; allow_dependents() lets such a
// dependent grid be scheduled as soon as every CTA of this grid has made
// the call or exited.  The dependent then synchronises with this grid by
// itself: the chain sampler polls the tags of the partials it reads, and
// the KV length update calls wait_for_prerequisite(), which returns once
// the grid before it has completed and its writes are visible.
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }
__device__ __forceinline__ void wait_for_prerequisite() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// A Partial moved as one 128-bit scalar at gpu scope (PTX .b128 with
// .relaxed.gpu): a reader in another grid that is running at the same time
// sees either the whole old or the whole new 16 bytes, never a mix, so the
// tag in the last word vouches for the three words before it.  Returned as
// float4 (a, s, idx bits, tag bits).
__device__ __forceinline__ void st_partial_relaxed(Partial* at, const Partial& v) {
  const uint64_t lo = static_cast<uint64_t>(__float_as_uint(v.s)) << 32 | __float_as_uint(v.a);
  const uint64_t hi = static_cast<uint64_t>(v.tag) << 32 | static_cast<uint32_t>(v.idx);
  asm volatile(
      "{\n\t.reg .b128 t;\n\tmov.b128 t, {%1, %2};\n\tst.relaxed.gpu.global.b128 [%0], t;\n\t}" ::"l"(at),
      "l"(lo), "l"(hi)
      : "memory");
}
__device__ __forceinline__ float4 ld_partial_relaxed(const Partial* at) {
  uint64_t lo, hi;
  asm volatile(
      "{\n\t.reg .b128 t;\n\tld.relaxed.gpu.global.b128 t, [%2];\n\tmov.b128 {%0, %1}, t;\n\t}"
      : "=l"(lo), "=l"(hi)
      : "l"(at)
      : "memory");
  return make_float4(__uint_as_float(static_cast<uint32_t>(lo)), __uint_as_float(static_cast<uint32_t>(lo >> 32)),
                     __uint_as_float(static_cast<uint32_t>(hi)), __uint_as_float(static_cast<uint32_t>(hi >> 32)));
}

// ---------------------------------------------------------------- numbers

// 2^x on the SFU (PTX ex2.approx.ftz.f32): results below 2^-126 flush to 0,
// 2^-inf = 0, NaN stays NaN.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max that propagates NaN (PTX max.NaN.f32).
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Temperature rule: 0 is greedy, a finite value >= 2^-126 is sampled,
// anything else (negative, NaN, inf, subnormal) is invalid.
__device__ __forceinline__ int temp_mode(float t) {
  if (t == 0.0f) return kModeGreedy;
  if (t >= 1.17549435e-38f && t <= 3.40282347e38f) return kModeSampled;
  return kModeInvalid;
}

// k = log2(e) / T, correctly rounded; every kernel derives it the same way.
__device__ __forceinline__ float scale_of(float t) { return __fdiv_rn(1.44269504088896341f, t); }

// Packed pairs of floats in one 64-bit register and the paired float
// instructions of this architecture (PTX fma/mul/add .f32x2).
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// ---------------------------------------------------------------- loads

// 16-byte copy global -> shared that holds no register while in flight
// (cached in L2 only); the issuing thread waits for its own copies with
// cp_async_wait_all.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Groups of copies: commit closes the group of this thread's copies issued
// since the last commit; wait_pending(n) returns once at most n of this
// thread's groups are still in flight (n a constant after unrolling).
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int kN>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(kN) : "memory");
}
__device__ __forceinline__ void cp_async_wait_pending(int n) {
  switch (n) {
    case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
  }
}


// 16-byte read-only load that does not allocate in L1 (each byte of a row
// is read once by the row-statistics pass).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int kVec = 4;                       // elements per 16 bytes
  static constexpr uint32_t kNegInfWord = 0xff800000u; // one -inf per word
  static __device__ __forceinline__ float get(const uint4& v, int e) {
    return __uint_as_float(word(v, e));
  }
  static __device__ __forceinline__ float vmax_nan(const uint4& v) {
    return fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                    fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
  static __device__ __forceinline__ float load1(const float* p) { return __ldg(p); }
  static constexpr int kPairs = 2;  // float pairs per 16 bytes
  // pair i of the 16 bytes: elements 2i, 2i+1
  static __device__ __forceinline__ uint64_t pair(const uint4& v, int i) {
    return i == 0 ? f2pack(__uint_as_float(v.x), __uint_as_float(v.y))
                  : f2pack(__uint_as_float(v.z), __uint_as_float(v.w));
  }
};

template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kVec = 8;
  static constexpr uint32_t kNegInfWord = 0xff80ff80u; // two bf16 -inf
  // Element e of the 16 bytes: element 2i is the low half of word i.
  static __device__ __forceinline__ float get(const uint4& v, int e) {
    const uint32_t w = word(v, e >> 1);
    return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
  }
  static __device__ __forceinline__ float vmax_nan(const uint4& v) {
    const uint32_t m = bmax2_nan(bmax2_nan(v.x, v.y), bmax2_nan(v.z, v.w));
    return fmax_nan(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
  }
  static __device__ __forceinline__ float load1(const __nv_bfloat16* p) {
    const unsigned short bits = __ldg(reinterpret_cast<const unsigned short*>(p));
    return __uint_as_float(static_cast<uint32_t>(bits) << 16);
  }
  static constexpr int kPairs = 4;
  static __device__ __forceinline__ uint64_t pair(const uint4& v, int i) {
    const uint32_t w = word(v, i);
    return f2pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
};

// ---------------------------------------------------------------- reductions
// Each takes its own shared scratch of kThreads/32 slots so that back-to-back
// reductions need no trailing barrier; every thread gets the result.

__device__ __forceinline__ float block_max_nan(float v, float* scratch) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmax_nan(v, __shfl_xor_sync(kFull, v, o));
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  v = scratch[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) v = fmax_nan(v, scratch[w]);
  return v;
}

__device__ __forceinline__ float block_sum(float v, float* scratch) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  v = scratch[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) v += scratch[w];
  return v;
}

__device__ __forceinline__ int block_min_int(int v, int* scratch) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(kFull, v, o));
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  v = scratch[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) v = min(v, scratch[w]);
  return v;
}

__device__ __forceinline__ int block_max_int(int v, int* scratch) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(kFull, v, o));
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  v = scratch[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) v = max(v, scratch[w]);
  return v;
}

// Exclusive prefix sum over the CTA in thread order (fp32); *total gets the
// CTA-wide sum.  scratch holds kThreads/32 floats.
__device__ __forceinline__ float block_exclusive_scan(float v, float* scratch, float* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  float before = 0.f, all = 0.f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const float t = scratch[w];
    if (w < warp) before += t;
    all += t;
  }
  *total = all;
  return before + incl - v;
}

// Exclusive prefix sum of unsigned counts over the CTA in thread order;
// *total gets the CTA-wide sum.  scratch holds kThreads/32 words.
__device__ __forceinline__ unsigned block_exclusive_scan_u32(unsigned v, unsigned* scratch,
                                                             unsigned* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  unsigned before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const unsigned t = scratch[w];
    if (w < warp) before += t;
    all += t;
  }
  *total = all;
  return before + incl - v;
}

// ---------------------------------------------------------------- Philox
// Philox4x32-10 as defined by Salmon, Moraes, Dror and Shaw, "Parallel
// Random Numbers: As Easy as 1, 2, 3" (SC'11): per round the products
// M0*x0 and M1*x2 are split into high and low words, the output is
// (hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0), and the key advances by the
// Weyl increments between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 x, uint2 key) {
  constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
  constexpr uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      key.x += kW0;
      key.y += kW1;
    }
    const uint32_t hi0 = __umulhi(kM0, x.x), lo0 = kM0 * x.x;
    const uint32_t hi1 = __umulhi(kM1, x.z), lo1 = kM1 * x.z;
    x = make_uint4(hi1 ^ x.y ^ key.x, lo1, hi0 ^ x.w ^ key.y, lo0);
  }
  return x;
}

__device__ __forceinline__ float word_uniform(uint32_t w) {
  return static_cast<float>(w >> 8) * 5.9604644775390625e-8f;  // 2^-24
}

// The four uniforms of (request b, 1-based position j, draw), one per word.
__device__ __forceinline__ void philox_uniforms4(unsigned long long seed, uint32_t b, uint32_t j,
                                                 uint32_t draw, float u[4]) {
  const uint2 key = make_uint2(static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  const uint4 r = philox4x32_10(make_uint4(b, j, draw, 0u), key);
  u[0] = word_uniform(r.x);
  u[1] = word_uniform(r.y);
  u[2] = word_uniform(r.z);
  u[3] = word_uniform(r.w);
}

// The uniform of (request b, 1-based position j, draw): (word0 >> 8) * 2^-24,
// exact in float32.
__device__ __forceinline__ float philox_uniform(unsigned long long seed, uint32_t b, uint32_t j,
                                                uint32_t draw) {
  const uint2 key = make_uint2(static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  const uint4 r = philox4x32_10(make_uint4(b, j, draw, 0u), key);
  return static_cast<float>(r.x >> 8) * 5.9604644775390625e-8f;  // 2^-24
}

}  // namespace sv
