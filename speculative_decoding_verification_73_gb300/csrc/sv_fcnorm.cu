// The drafter's input fusion with FC normalisation (EAGLE-3 / EAGLE 3.1):
//   out = [norm(h_early); norm(h_mid); norm(h_late)] . W^T + bias
// (EAGLE-3 / EAGLE 3.1 page, "FC normalisation: the key change of EAGLE
// 3.1": LayerNorm on each of the three target hidden states before the FC;
// the EAGLE 3.1 news page speaks of RMSNorm; no norm is EAGLE-3).
//
// Two kernels.  fcnorm_stats: one warp per (token, segment) computes the
// row's mean and 1/sqrt(var + eps) (LayerNorm; mean 0 and 1/sqrt(mean
// square + eps) for RMSNorm) in fp32, two passes over the row.
// fcnorm_gemm: a tcgen05 GEMM.  Each CTA owns a 128 x 256 output tile; per
// 64-wide K step its 256 threads build the A tile (128 tokens x 64 inputs)
// by normalising h on the fly -- (h - mean) * rstd * gamma + beta, rounded
// to bf16 -- straight into shared memory in the canonical K-major layout
// (8 x 16-byte core matrices, no swizzle), while the W tile (256 outputs x
// 64 inputs) arrives with cp.async.  One thread issues four
// tcgen05.mma.kind::f16 (K = 16 each) into an fp32 accumulator of 256 TMEM
// columns and commits them to the stage's mbarrier; three stages let the
// loads of the next steps overlap the tensor core.  The epilogue reads the
// accumulator with tcgen05.ld, adds the bias and stores bf16.  Every wait on
// an mbarrier is bounded; a wait that runs out sets an error bit and the
// kernel still frees its TMEM.

#include <cstdint>
#include <cuda_bf16.h>

#include "sv_device.cuh"

namespace sv {
namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kKG = kBK / 8;                       // core matrices along K per tile
constexpr int kStages = 3;
constexpr int kFcThreads = 256;
constexpr int kABytes = kBM * kBK * 2;             // 16 KB
constexpr int kBBytes = kBN * kBK * 2;             // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;     // 48 KB
constexpr int kTmemCols = kBN;                     // fp32 accumulator 128 lanes x 256 columns
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

// --------------------------------------------------------------- statistics

__global__ void fcnorm_stats_kernel(FcNormProblem p) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= p.T * 3) return;
  const int t = warp / 3, s = warp - t * 3;
  const __nv_bfloat16* h = (s == 0 ? p.h[0] : s == 1 ? p.h[1] : p.h[2]) + static_cast<size_t>(t) * p.d;
  float mu = 0.f, rstd = 1.f;
  if (p.norm != kNormNone) {
    float sum = 0.f;
    if (p.norm == kNormLayer) {
      for (int f = lane * 8; f < p.d; f += 256) {
        const uint4 v = *reinterpret_cast<const uint4*>(h + f);
#pragma unroll
        for (int e = 0; e < 8; ++e) sum += Elem<__nv_bfloat16>::get(v, e);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
      mu = sum / static_cast<float>(p.d);
    }
    float sq = 0.f;
    for (int f = lane * 8; f < p.d; f += 256) {
      const uint4 v = *reinterpret_cast<const uint4*>(h + f);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float x = Elem<__nv_bfloat16>::get(v, e) - mu;
        sq = fmaf(x, x, sq);
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) sq += __shfl_xor_sync(kFull, sq, o);
    rstd = rsqrtf(sq / static_cast<float>(p.d) + p.eps);
  }
  if (lane == 0) {
    p.stats[(static_cast<size_t>(t) * 3 + s) * 2] = mu;
    p.stats[(static_cast<size_t>(t) * 3 + s) * 2 + 1] = rstd;
  }
}

// --------------------------------------------------------------- the GEMM

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__global__ void __launch_bounds__(kFcThreads, 1) fcnorm_gemm_kernel(FcNormProblem p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ float s_mu[3][kBM], s_rs[3][kBM];
  __shared__ __align__(8) uint64_t s_bar[kStages];
  __shared__ uint32_t s_tmem;
  __shared__ int s_fail;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int n0 = blockIdx.x * kBN, m0 = blockIdx.y * kBM;
  const int d = p.d, K = 3 * d, nk = K / kBK;

  for (int i = tid; i < 3 * kBM; i += kFcThreads) {
    const int s = i / kBM, r = i - s * kBM;
    const int t = m0 + r;
    s_mu[s][r] = t < p.T ? p.stats[(static_cast<size_t>(t) * 3 + s) * 2] : 0.f;
    s_rs[s][r] = t < p.T ? p.stats[(static_cast<size_t>(t) * 3 + s) * 2 + 1] : 0.f;
  }
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
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = s_tmem;
  const uint32_t idesc = mma_idesc(kBM, kBN);

  bool ok = true;
  int committed = -1;  // last k step whose MMAs were committed
  for (int kt = 0; kt < nk && ok; ++kt) {
    const int st = kt % kStages;
    unsigned char* sA = smem + st * kStageBytes;
    unsigned char* sB = sA + kABytes;
    if (kt >= kStages) {  // the MMAs that read this stage kStages steps ago are done
      if (!mbar_wait(smem_u32(&s_bar[st]), static_cast<uint32_t>((kt / kStages - 1) & 1))) {
        if (tid == 0) s_fail = 1;
      }
      __syncthreads();
      if (s_fail) {
        ok = false;
        break;
      }
    }
    const int k0 = kt * kBK;
    // W tile: 256 rows x 8 chunks of 16 bytes, rows past d_out zero
    for (int q = tid; q < kBN * kKG; q += kFcThreads) {
      const int n = q % kBN, c = q / kBN;
      unsigned char* dst = sB + (n >> 3) * (kKG * 128) + c * 128 + (n & 7) * 16;
      if (n0 + n < p.d_out)
        cp_async16(dst, p.w + static_cast<size_t>(n0 + n) * K + k0 + c * 8);
      else
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
    // A tile: normalised hidden states, 128 tokens x 8 chunks
    const int seg = k0 / d, f0 = k0 - seg * d;
    const __nv_bfloat16* hs = seg == 0 ? p.h[0] : seg == 1 ? p.h[1] : p.h[2];
    for (int q = tid; q < kBM * kKG; q += kFcThreads) {
      const int m = q % kBM, c = q / kBM;
      unsigned char* dst = sA + (m >> 3) * (kKG * 128) + c * 128 + (m & 7) * 16;
      const int t = m0 + m;
      uint4 out = make_uint4(0, 0, 0, 0);
      if (t < p.T) {
        const int f = f0 + c * 8;
        const uint4 v = *reinterpret_cast<const uint4*>(hs + static_cast<size_t>(t) * d + f);
        if (p.norm == kNormNone) {
          out = v;
        } else {
          const float mu = s_mu[seg][m], rs = s_rs[seg][m];
          const float* g = p.gamma + seg * d + f;
          const float* bt = p.beta != nullptr ? p.beta + seg * d + f : nullptr;
          float x[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float y = (Elem<__nv_bfloat16>::get(v, e) - mu) * rs * __ldg(g + e);
            if (bt != nullptr) y += __ldg(bt + e);
            x[e] = y;
          }
          out = make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                           pack_bf16(x[6], x[7]));
        }
      }
      *reinterpret_cast<uint4*>(dst) = out;
    }
    cp_async_wait_all();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor core
    __syncthreads();
    if (tid == 0) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        const uint64_t da = smem_desc(smem_u32(sA) + kk * 256, 128, kKG * 128);
        const uint64_t db = smem_desc(smem_u32(sB) + kk * 256, 128, kKG * 128);
        const uint32_t acc = (kt > 0 || kk > 0) ? 1u : 0u;
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
            "l"(da), "l"(db), "r"(idesc), "r"(acc)
            : "memory");
      }
      asm volatile(
          "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
              smem_u32(&s_bar[st]))
          : "memory");
    }
    committed = kt;
  }

  // the last commit covers every MMA issued before it
  if (ok && nk > 0) {
    const int last = nk - 1;
    if (!mbar_wait(smem_u32(&s_bar[last % kStages]), static_cast<uint32_t>((last / kStages) & 1)))
      ok = false;
  }
  ok = __syncthreads_and(ok);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (ok && nk > 0) {
    // warp w reads TMEM lanes 32 (w % 4) .. + 31 (its rows) and column half w / 4
    const int lane_base = (warp & 3) * 32;
    const int m = lane_base + (tid & 31);
    const int t = m0 + m;
    const int cbase = (warp >> 2) * (kBN / 2);
    for (int c = 0; c < kBN / 2; c += 16) {
      uint32_t r[16];
      const uint32_t addr = tmem + (static_cast<uint32_t>(lane_base) << 16) + cbase + c;
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

int fcnorm_smem_bytes() { return kStages * kStageBytes; }

cudaError_t launch_fcnorm(const FcNormProblem& p, cudaStream_t s) {
  if (p.T <= 0 || p.d_out <= 0) return cudaSuccess;
  const int warps = p.T * 3;
  fcnorm_stats_kernel<<<(warps * 32 + 255) / 256, 256, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int smem = kStages * kStageBytes;
  e = cudaFuncSetAttribute(fcnorm_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((p.d_out + kBN - 1) / kBN, (p.T + kBM - 1) / kBM);
  fcnorm_gemm_kernel<<<grid, kFcThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace sv
