// The drafter's input fusion with FC normalisation (EAGLE-3 / EAGLE 3.1):
//   out = [norm(h_early); norm(h_mid); norm(h_late)] . W^T + bias
// (EAGLE-3 / EAGLE 3.1 page, "FC normalisation: the key change of EAGLE
// 3.1": LayerNorm on each of the three target hidden states before the FC;
// the EAGLE 3.1 news page speaks of RMSNorm; no norm is EAGLE-3).
//
// Two kernels.  fcnorm_prep: one warp per (token, segment) computes the
// row's mean and 1/sqrt(var + eps) (LayerNorm; mean 0 and 1/sqrt(mean
// square + eps) for RMSNorm) in fp32 and writes the normalised row, rounded
// to bf16, into its third of the concatenated input X [T, 3d] (three passes
// over a row that stays in L1/L2).  fc_gemm: a tcgen05 GEMM out = X W^T +
// bias.  Each CTA owns a 256 x 256 output tile (two 128-row halves sharing
// the B tile) and walks K in steps of 64 through three shared-memory stages
// filled by cp.async in the canonical K-major layout (8 x 16-byte core
// matrices, no swizzle), loads issued two steps ahead; one thread issues,
// per step and half, four tcgen05.mma.kind::f16 (M = 128, K = 16 each) into
// that half's fp32 accumulator of 256 TMEM columns and commits them to the
// stage's mbarrier, which frees the stage for the loads of a later step.  The
// epilogue reads the accumulator with tcgen05.ld, adds the bias and stores
// bf16.  Every mbarrier wait is bounded; one that runs out sets an error bit
// and the kernel still frees its TMEM.  (A first version normalised the A
// tile on the fly inside the GEMM, with each step's loads issued only after
// the previous step's MMAs: 150 TFLOP/s on T = d = d_out = 4096; writing X
// costs one more pass over the hidden states and lets the GEMM pipeline.)

#include <cstdint>
#include <cuda_bf16.h>

#include "sv_device.cuh"

namespace sv {
namespace {

// kMW 128-row halves of the output tile per CTA, each its own MMA (M = 128)
// and accumulator, all sharing the stage's B tile: kMW = 2 moves 64 KB per
// K step for twice the MMAs of kMW = 1 (48 KB).
#ifndef SV_FC_MW
#define SV_FC_MW 2
#endif
constexpr int kMW = SV_FC_MW;
constexpr int kBM = 128 * kMW, kBN = 256, kBK = 64;
constexpr int kKG = kBK / 8;                       // core matrices along K per tile
constexpr int kStages = kMW == 2 ? 3 : 4;          // 3 x 64 KB or 4 x 48 KB of shared memory
#ifndef SV_FC_AHEAD
#define SV_FC_AHEAD 2  // 3 measured slower with kMW = 1: 246 against 281 TFLOP/s
#endif
constexpr int kAhead = SV_FC_AHEAD;                // steps of loads in flight ahead of the MMAs
constexpr int kFcThreads = 256;
constexpr int kABytes = kBM * kBK * 2;             // 16 KB per 128 rows
constexpr int kBBytes = kBN * kBK * 2;             // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kHalfABytes = 128 / 8 * kKG * 128;   // offset of rows 128.. in the A tile
constexpr int kTmemCols = kBN * kMW;               // fp32 accumulators: 128 lanes x 256 columns each
static_assert(kMW == 1 || kMW == 2, "one or two 128-row halves");
static_assert(kAhead + 1 <= kStages, "a stage is refilled only after the MMAs that read it");
constexpr uint32_t kWaitLimit = 1u << 26;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Shared-memory matrix descriptor: start address, leading (K-direction) and
// stride (M/N-direction) byte offsets between core matrices, descriptor
// version 1, no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((addr & 0x3FFFF) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, M x N.
__device__ __forceinline__ uint32_t mma_idesc(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t it = 0; it < kWaitLimit; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}

// --------------------------------------------------------------- normalisation

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__global__ void fcnorm_prep_kernel(FcNormProblem p) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= p.T * 3) return;
  const int t = warp / 3, s = warp - t * 3;
  const int d = p.d;
  const __nv_bfloat16* h = (s == 0 ? p.h[0] : s == 1 ? p.h[1] : p.h[2]) + static_cast<size_t>(t) * d;
  __nv_bfloat16* x = p.x + static_cast<size_t>(t) * 3 * d + static_cast<size_t>(s) * d;
  float mu = 0.f, rstd = 1.f;
  if (p.norm != kNormNone) {
    if (p.norm == kNormLayer) {
      float sum = 0.f;
      for (int f = lane * 8; f < d; f += 256) {
        const uint4 v = *reinterpret_cast<const uint4*>(h + f);
#pragma unroll
        for (int e = 0; e < 8; ++e) sum += Elem<__nv_bfloat16>::get(v, e);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
      mu = sum / static_cast<float>(d);
    }
    float sq = 0.f;
    for (int f = lane * 8; f < d; f += 256) {
      const uint4 v = *reinterpret_cast<const uint4*>(h + f);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float y = Elem<__nv_bfloat16>::get(v, e) - mu;
        sq = fmaf(y, y, sq);
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) sq += __shfl_xor_sync(kFull, sq, o);
    rstd = rsqrtf(sq / static_cast<float>(d) + p.eps);
  }
  const float* g = p.gamma + static_cast<size_t>(s) * d;
  const float* bt = p.beta != nullptr ? p.beta + static_cast<size_t>(s) * d : nullptr;
  for (int f = lane * 8; f < d; f += 256) {
    const uint4 v = *reinterpret_cast<const uint4*>(h + f);
    uint4 o = v;
    if (p.norm != kNormNone) {
      float y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float z = (Elem<__nv_bfloat16>::get(v, e) - mu) * rstd * __ldg(g + f + e);
        if (bt != nullptr) z += __ldg(bt + f + e);
        y[e] = z;
      }
      o = make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]),
                     pack_bf16(y[6], y[7]));
    }
    *reinterpret_cast<uint4*>(x + f) = o;
  }
}

// --------------------------------------------------------------- the GEMM

// 16-byte cp.async that writes zeros instead of reading when !valid.
__device__ __forceinline__ void cp_async16_or_zero(void* smem_dst, const void* gmem_src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "l"(gmem_src), "r"(valid ? 16 : 0)
               : "memory");
}

// Loads of K step kt into a stage: X rows m0.., W rows n0.., 8 chunks of 16
// bytes each.  Chunk q goes to row (q / 64) * 8 + q % 8 and column chunk
// (q / 8) % 8: eight consecutive threads fill one 16-byte column of eight
// rows (eight distinct bank groups of a core matrix: no shared-memory bank
// conflict), and a warp reads 64 contiguous bytes from each of eight rows.
__device__ __forceinline__ int chunk_row(int q) { return (q >> 6) * 8 + (q & 7); }
__device__ __forceinline__ int chunk_col(int q) { return (q >> 3) & 7; }

__device__ __forceinline__ void load_stage(const FcNormProblem& p, unsigned char* stage, int m0, int n0,
                                           int kt) {
  const int K = 3 * p.d;
  const int k0 = kt * kBK;
  unsigned char* sA = stage;
  unsigned char* sB = stage + kABytes;
  for (int q = threadIdx.x; q < kBM * kKG; q += kFcThreads) {
    const int m = chunk_row(q), c = chunk_col(q);
    const bool in = m0 + m < p.T;
    const __nv_bfloat16* src = p.x + static_cast<size_t>(in ? m0 + m : 0) * K + k0 + c * 8;
    cp_async16_or_zero(sA + (m >> 3) * (kKG * 128) + c * 128 + (m & 7) * 16, src, in);
  }
  for (int q = threadIdx.x; q < kBN * kKG; q += kFcThreads) {
    const int n = chunk_row(q), c = chunk_col(q);
    const bool in = n0 + n < p.d_out;
    const __nv_bfloat16* src = p.w + static_cast<size_t>(in ? n0 + n : 0) * K + k0 + c * 8;
    cp_async16_or_zero(sB + (n >> 3) * (kKG * 128) + c * 128 + (n & 7) * 16, src, in);
  }
}

__global__ void __launch_bounds__(kFcThreads, 1) fc_gemm_kernel(FcNormProblem p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ __align__(8) uint64_t s_bar[kStages];
  __shared__ uint32_t s_tmem;
  __shared__ int s_fail;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int n0 = blockIdx.x * kBN, m0 = blockIdx.y * kBM;
  const int nk = 3 * p.d / kBK;

  if (tid == 0) {
    s_fail = 0;
    for (int s = 0; s < kStages; ++s)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&s_bar[s])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&s_tmem)),
                 "n"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
#pragma unroll
  for (int a = 0; a < kAhead; ++a) {
    if (a < nk) load_stage(p, smem + a * kStageBytes, m0, n0, a);
    cp_async_commit();
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = s_tmem;
  const uint32_t idesc = mma_idesc(128, kBN);

  bool ok = true;
  int committed = -1;  // last k step whose MMAs were committed
  for (int kt = 0; kt < nk; ++kt) {
    // refill the stage of step kt + kAhead, last read by the MMAs of step
    // kt + kAhead - kStages (<= kt - 1, committed in an earlier iteration):
    // wait for them first
    const int nxt = kt + kAhead;
    const int prev = nxt - kStages;
    if (prev >= 0 && nxt < nk) {
      if (!mbar_wait(smem_u32(&s_bar[prev % kStages]), static_cast<uint32_t>((prev / kStages) & 1)))
        s_fail = 1;
    }
    if (nxt < nk) load_stage(p, smem + (nxt % kStages) * kStageBytes, m0, n0, nxt);
    cp_async_commit();
    cp_async_wait_group<kAhead>();  // this thread's loads of step kt have landed
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor core
    __syncthreads();
    if (s_fail) {
      ok = false;
      break;
    }
    if (tid == 0) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const unsigned char* sA = smem + (kt % kStages) * kStageBytes;
      const unsigned char* sB = sA + kABytes;
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        const uint64_t db = smem_desc(smem_u32(sB) + kk * 256, 128, kKG * 128);
        const uint32_t acc = (kt > 0 || kk > 0) ? 1u : 0u;
#pragma unroll
        for (int h = 0; h < kMW; ++h) {  // half h: A rows 128h.., accumulator columns 256h..
          const uint64_t da = smem_desc(smem_u32(sA) + h * kHalfABytes + kk * 256, 128, kKG * 128);
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem + h * kBN),
              "l"(da), "l"(db), "r"(idesc), "r"(acc)
              : "memory");
        }
      }
      asm volatile(
          "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
              smem_u32(&s_bar[kt % kStages]))
          : "memory");
    }
    committed = kt;
  }
  cp_async_wait_group<0>();

  // the last commit covers every MMA issued before it
  if (ok && nk > 0) {
    const int last = nk - 1;
    if (!mbar_wait(smem_u32(&s_bar[last % kStages]), static_cast<uint32_t>((last / kStages) & 1)))
      ok = false;
  }
  ok = __syncthreads_and(ok);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  for (int h = 0; h < kMW && ok && nk > 0; ++h) {
    // warp w reads TMEM lanes 32 (w % 4) .. + 31 (its rows of half h) and
    // column half w / 4 of that half's accumulator
    const int lane_base = (warp & 3) * 32;
    const int m = h * 128 + lane_base + (tid & 31);
    const int t = m0 + m;
    const int cbase = (warp >> 2) * (kBN / 2);
    for (int c = 0; c < kBN / 2; c += 16) {
      uint32_t r[16];
      const uint32_t addr = tmem + (static_cast<uint32_t>(lane_base) << 16) + h * kBN + cbase + c;
      asm volatile(
          "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
          "%15}, [%16];"
          : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
            "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
            "=r"(r[14]), "=r"(r[15])
          : "r"(addr));
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      const int n = n0 + cbase + c;
      if (t < p.T) {
        float y[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          y[j] = __uint_as_float(r[j]) + (p.bias != nullptr && n + j < p.d_out ? __ldg(p.bias + n + j) : 0.f);
        __nv_bfloat16* out = p.out + static_cast<size_t>(t) * p.d_out + n;
        if (n + 16 <= p.d_out && p.out_vec) {
          uint4* o = reinterpret_cast<uint4*>(out);
          o[0] = make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]),
                            pack_bf16(y[6], y[7]));
          o[1] = make_uint4(pack_bf16(y[8], y[9]), pack_bf16(y[10], y[11]), pack_bf16(y[12], y[13]),
                            pack_bf16(y[14], y[15]));
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (n + j < p.d_out) out[j] = __float2bfloat16_rn(y[j]);
        }
      }
    }
  }
  if (!ok && tid == 0) {
    atomicOr(p.err, kErrWait);
    // give the tensor core a last bounded chance to finish before the
    // accumulator's columns are freed
    if (committed >= 0)
      mbar_wait(smem_u32(&s_bar[committed % kStages]),
                static_cast<uint32_t>((committed / kStages) & 1));
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols)
                 : "memory");
}

}  // namespace

cudaError_t launch_fcnorm(const FcNormProblem& p, cudaStream_t s) {
  if (p.T <= 0 || p.d_out <= 0) return cudaSuccess;
  const int warps = p.T * 3;
  fcnorm_prep_kernel<<<(warps * 32 + 255) / 256, 256, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int smem = kStages * kStageBytes;
  e = cudaFuncSetAttribute(fc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((p.d_out + kBN - 1) / kBN, (p.T + kBM - 1) / kBM);
  fc_gemm_kernel<<<grid, kFcThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace sv
