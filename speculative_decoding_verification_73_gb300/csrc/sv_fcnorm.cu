// The drafter's input fusion with FC normalisation (EAGLE-3 / EAGLE 3.1):
//   out = [norm(h_early); norm(h_mid); norm(h_late)] . W^T + bias
// (EAGLE-3 / EAGLE 3.1 page, "FC normalisation: the key change of EAGLE
// 3.1": LayerNorm on each of the three target hidden states before the FC;
// the EAGLE 3.1 news page speaks of RMSNorm; no norm is EAGLE-3).
//
// fcnorm_prep (LayerNorm / RMSNorm): for each (token, segment) row the
// row's mean and 1/sqrt(var + eps) (LayerNorm; mean 0 and
// 1/sqrt(mean square + eps) for RMSNorm) in fp32, and the normalised row,
// rounded to bf16, written into its third of the concatenated input
// X [T, 3d] -- a CTA per four tokens of one segment (one warp per row past
// 4096 elements).  fc_gemm: a persistent tcgen05
// GEMM out = X W^T + bias -- with no normalisation it reads the three
// hidden states themselves, K step kb from the state kb / (d / 64), and
// nothing runs before it -- one CTA per SM walking 128 x bn output tiles
// (bn <= 256), with its warps split by role:
//   * warp 0 (one lane) loads: for each K step of 64 it waits until the
//     stage is free, then fetches the 128 x 64 input tile and the bn x 64
//     tile of W with two TMA tensor copies (cp.async.bulk.tensor, 128-byte
//     swizzle) completing on the stage's "full" barrier;
//   * warp 1 (one lane) multiplies: for each K step it waits for the stage,
//     issues four tcgen05.mma.kind::f16 (M = 128, N = 256, K = 16) into one
//     of two fp32 accumulators of 256 TMEM columns, and commits them to the
//     stage's "empty" barrier (the stage is refilled once they are done);
//     after the tile's last step it commits to the accumulator's "full"
//     barrier;
//   * warps 2-5 drain: they wait for an accumulator, read it with tcgen05.ld
//     (each warp its quarter of the 128 lanes, one output row per thread),
//     add the bias, store bf16 rows and release the accumulator, while the
//     MMAs of the next tile already fill the other one.
// So loads, MMAs and the epilogue overlap without any CTA-wide barrier in the
// loop.  Tiles go m-block by m-block (all n-blocks of the first 128 rows,
// then the next), so the CTAs working at one time share their X tiles and
// W stays in L2.  Every barrier wait is bounded; one that runs out sets
// SV_ERRBIT_WAIT, stops the CTA's loop, waits (bounded) for the copies and
// MMAs it started, and frees its TMEM.

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "sv_device.cuh"
#include "sv_mbar.cuh"

namespace sv {
namespace {

constexpr int kBM = 128, kBNMax = 256, kBK = 64;  // output tile (kBM x bn, bn <= 256), K step
constexpr int kMaxStages = 8;  // the ring holds as many stages as fit (see gemm_stages)
constexpr int kABytes = kBM * kBK * 2;          // 16 KB
// One stage: the 128 x 64 input tile, then the bn x 64 W tile, rounded up
// to the 1024-byte swizzle atom (44 KB for bn = 224, 48 KB for 256).
__host__ __device__ constexpr int stage_bytes(int bn) { return (kABytes + bn * kBK * 2 + 1023) / 1024 * 1024; }
constexpr int kAccCols = kBNMax;                // fp32 accumulator slot: 128 lanes x 256 columns
constexpr int kTmemCols = 2 * kAccCols;         // two accumulators
constexpr int kFcThreads = 192;                 // loads, MMAs, four epilogue warps
constexpr int kEpiThreads = 128;
// Where the GEMM's input tiles come from.
constexpr int kGemmX = 0;       // X [T, 3d], written by the normalisation grid before
constexpr int kGemmDirect = 1;  // the three hidden states themselves (no normalisation)

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, M x N.
__device__ __forceinline__ uint32_t mma_idesc(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// --------------------------------------------------------------- normalisation

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}


// Rows of d <= 4096 elements with 16-byte aligned gamma / beta: one CTA
// normalises kPrepRows consecutive tokens of one segment.  Warp w holds, in
// lane l, the 16-byte vectors 64 w + 32 i + l (i < 2) of each of those rows,
// so every element is read from global memory once; each warp sums its part
// of every row, the parts meet in shared memory (added in warp order, the
// same in every warp), then the same for the squared deviations.  Since a
// warp holds the same columns of all the CTA's rows, it loads each gamma /
// beta vector once and applies it to every row: the loads of gamma / beta
// (four times the bytes of the row vector they scale) kept the kernel bound
// by L1 when every warp had its own row.
// Tokens of one segment per CTA (build-time override -DSV_PREP_ROWS=<n>):
// four at 64 registers (4 CTAs per SM) measured 314.8 us per LayerNorm call
// at T = d = d_out = 4096, two at 40 registers (6 per SM) 316.1 us, two at
// 58 registers (4 per SM) 319.7 us.
#ifndef SV_PREP_ROWS
#define SV_PREP_ROWS 4
#endif
constexpr int kPrepRows = SV_PREP_ROWS;
constexpr int kPrepVec = 2;    // vectors per lane and row: 8 warps x 32 lanes x 2 x 8 = 4096 columns
constexpr int kPrepMaxD = 8 * 32 * kPrepVec * 8;

// The CTA's total of one per-warp partial each, in warp order.
__device__ __forceinline__ float warps_total(const float* s_part) {
  float t = s_part[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) t += s_part[w];
  return t;
}

// The same statistics and output for any row length, three passes over the
// row (the later ones from L1 / L2).
__device__ __forceinline__ void prep_row_loop(const FcNormProblem& p, const __nv_bfloat16* h,
                                              __nv_bfloat16* x, const float* g, const float* bt, int lane) {
  const int d = p.d;
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

// Resident CTAs per SM the normalisation kernel of short rows is built for.
#ifndef SV_PREP_MINB
#define SV_PREP_MINB 4
#endif

__global__ void __launch_bounds__(256, SV_PREP_MINB) fcnorm_prep_rows_kernel(FcNormProblem p) {
  allow_dependents();  // the GEMM's CTAs may be scheduled as this grid drains
  __shared__ float s_part[kPrepRows][8];
  const int wl = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int groups = (p.T + kPrepRows - 1) / kPrepRows;
  const int sg = blockIdx.x / groups;  // segment: h_early, h_mid, h_late
  const int t0 = (blockIdx.x - sg * groups) * kPrepRows;
  const int d = p.d, nvec = d / 8;
  const __nv_bfloat16* h = sg == 0 ? p.h[0] : sg == 1 ? p.h[1] : p.h[2];
  uint4 v[kPrepRows][kPrepVec];
#pragma unroll
  for (int r = 0; r < kPrepRows; ++r) {
#pragma unroll
    for (int i = 0; i < kPrepVec; ++i) {
      const int q = 64 * wl + 32 * i + lane;
      const int t = t0 + r;
      v[r][i] = (t < p.T && q < nvec) ? *reinterpret_cast<const uint4*>(h + static_cast<size_t>(t) * d + 8 * q)
                                      : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  // the arithmetic in pairs of floats (paired float instructions)
  using E = Elem<__nv_bfloat16>;
  float mu[kPrepRows], rstd[kPrepRows];
#pragma unroll
  for (int r = 0; r < kPrepRows; ++r) {
    mu[r] = 0.f;
    rstd[r] = 1.f;
  }
  if (p.norm != kNormNone) {
    if (p.norm == kNormLayer) {
#pragma unroll
      for (int r = 0; r < kPrepRows; ++r) {
        uint64_t s2 = f2pack(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < kPrepVec; ++i) {
#pragma unroll
          for (int e = 0; e < E::kPairs; ++e) s2 = f2add(s2, E::pair(v[r][i], e));  // zeros past the row
        }
        float lo, hi;
        f2unpack(s2, lo, hi);
        float sum = lo + hi;
#pragma unroll
        for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
        if (lane == 0) s_part[r][wl] = sum;
      }
      __syncthreads();
#pragma unroll
      for (int r = 0; r < kPrepRows; ++r) mu[r] = warps_total(s_part[r]) / static_cast<float>(d);
      __syncthreads();  // every warp has read s_part
    }
#pragma unroll
    for (int r = 0; r < kPrepRows; ++r) {
      const uint64_t nmu2 = f2pack(-mu[r], -mu[r]);
      uint64_t q2 = f2pack(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < kPrepVec; ++i) {
        if (64 * wl + 32 * i + lane < nvec) {
#pragma unroll
          for (int e = 0; e < E::kPairs; ++e) {
            const uint64_t y2 = f2add(E::pair(v[r][i], e), nmu2);
            q2 = f2fma(y2, y2, q2);
          }
        }
      }
      float lo, hi;
      f2unpack(q2, lo, hi);
      float sq = lo + hi;
#pragma unroll
      for (int o = 16; o; o >>= 1) sq += __shfl_xor_sync(kFull, sq, o);
      if (lane == 0) s_part[r][wl] = sq;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kPrepRows; ++r)
      rstd[r] = rsqrtf(warps_total(s_part[r]) / static_cast<float>(d) + p.eps);
  }
  const float* g = p.norm != kNormNone ? p.gamma + static_cast<size_t>(sg) * d : nullptr;
  const float* bt = p.beta != nullptr ? p.beta + static_cast<size_t>(sg) * d : nullptr;
  __nv_bfloat16* x = p.x + static_cast<size_t>(sg) * d;
#pragma unroll
  for (int i = 0; i < kPrepVec; ++i) {
    const int q = 64 * wl + 32 * i + lane;
    if (q >= nvec) continue;
    // gamma and beta of the vector's 8 columns, as 4 pairs each
    uint64_t g2[4], b2[4];
    if (p.norm != kNormNone) {
      const int f = 8 * q;
      const float4 g0 = __ldg(reinterpret_cast<const float4*>(g + f));
      const float4 g1 = __ldg(reinterpret_cast<const float4*>(g + f + 4));
      float4 b0 = make_float4(0.f, 0.f, 0.f, 0.f), b1 = b0;
      if (bt != nullptr) {
        b0 = __ldg(reinterpret_cast<const float4*>(bt + f));
        b1 = __ldg(reinterpret_cast<const float4*>(bt + f + 4));
      }
      g2[0] = f2pack(g0.x, g0.y);
      g2[1] = f2pack(g0.z, g0.w);
      g2[2] = f2pack(g1.x, g1.y);
      g2[3] = f2pack(g1.z, g1.w);
      b2[0] = f2pack(b0.x, b0.y);
      b2[1] = f2pack(b0.z, b0.w);
      b2[2] = f2pack(b1.x, b1.y);
      b2[3] = f2pack(b1.z, b1.w);
    }
#pragma unroll
    for (int r = 0; r < kPrepRows; ++r) {
      const int t = t0 + r;
      if (t >= p.T) continue;
      uint4 o = v[r][i];
      if (p.norm != kNormNone) {
        // y = (x - mu) (rstd gamma) + beta
        const uint64_t nmu2 = f2pack(-mu[r], -mu[r]), rs2 = f2pack(rstd[r], rstd[r]);
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < E::kPairs; ++e) {
          const uint64_t y2 = f2fma(f2add(E::pair(v[r][i], e), nmu2), f2mul(rs2, g2[e]), b2[e]);
          float lo, hi;
          f2unpack(y2, lo, hi);
          w[e] = pack_bf16(lo, hi);
        }
        o = make_uint4(w[0], w[1], w[2], w[3]);
      }
      *reinterpret_cast<uint4*>(x + static_cast<size_t>(t) * 3 * d + 8 * q) = o;
    }
  }
}

// Any other row: one warp per row, three passes.
__global__ void __launch_bounds__(256) fcnorm_prep_kernel(FcNormProblem p) {
  allow_dependents();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= p.T * 3) return;
  const int t = warp / 3, s = warp - t * 3;
  const int d = p.d;
  const __nv_bfloat16* h = (s == 0 ? p.h[0] : s == 1 ? p.h[1] : p.h[2]) + static_cast<size_t>(t) * d;
  __nv_bfloat16* x = p.x + static_cast<size_t>(t) * 3 * d + static_cast<size_t>(s) * d;
  const float* g = p.norm != kNormNone ? p.gamma + static_cast<size_t>(s) * d : nullptr;
  const float* bt = p.beta != nullptr ? p.beta + static_cast<size_t>(s) * d : nullptr;
  prep_row_loop(p, h, x, g, bt, lane);
}

// --------------------------------------------------------------- the GEMM

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes in atoms of 8 rows (1024 bytes apart
// along M/N), descriptor version 1, swizzle mode 2 (128 bytes).  The K
// offset inside the 128-byte row is added to the start address.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  uint64_t d = static_cast<uint64_t>((addr & 0x3FFFF) >> 4);
  d |= static_cast<uint64_t>(1) << 16;              // leading offset (unused with this swizzle)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;      // stride offset: 8 rows of 128 bytes
  d |= static_cast<uint64_t>(1) << 46;              // descriptor version
  d |= static_cast<uint64_t>(2) << 61;              // 128-byte swizzle
  return d;
}

// 2-D TMA tensor copy of the box at (x, y) (x = K element offset, a multiple
// of 64; y = row) into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tile_of(int t, int n_tiles_n, int bn, int& m0, int& n0) {
  const int mb = t / n_tiles_n;
  m0 = mb * kBM;
  n0 = (t - mb * n_tiles_n) * bn;
}

struct GemmShared {
  uint64_t full[kMaxStages], empty[kMaxStages];  // stage loaded / stage free
  uint64_t acc_full[2], acc_empty[2];       // accumulator ready / drained
  uint32_t tmem;
  int abort;
};

// map_a0..2: the input tiles -- X (kGemmX: map_a0 only, K = 3d) or the
// three hidden states [T, d] (K step kb of segment kb / (d / 64)).
template <int kMode>
__global__ void __launch_bounds__(kFcThreads, 1)
    fc_gemm_kernel(FcNormProblem p, const __grid_constant__ CUtensorMap map_a0,
                   const __grid_constant__ CUtensorMap map_a1, const __grid_constant__ CUtensorMap map_a2,
                   const __grid_constant__ CUtensorMap map_w, int bn, int stages) {
  const int sbytes = stage_bytes(bn);
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // stages 1024-byte aligned (the swizzle atom); the runtime guarantees 16
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ GemmShared sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = 3 * p.d;
  const int nk = K / kBK;
  const int n_tiles_n = (p.d_out + bn - 1) / bn;
  const int n_tiles = ((p.T + kBM - 1) / kBM) * n_tiles_n;

  const int kps = p.d / kBK;  // K steps per hidden state
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh.acc_full[a], 1);
      mbar_init(&sh.acc_empty[a], kEpiThreads);
    }
    sh.abort = 0;
    mbar_init_fence();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sh.tmem)),
                 "n"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = sh.tmem;
  volatile int* abort = &sh.abort;

  if (warp == 0) {
    // ---------------- loads
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_a0)) : "memory");
      if (kMode != kGemmX) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_a1)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_a2)) : "memory");
      }
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_w)) : "memory");
      // kGemmX: X is written by the normalisation grid before this one (this
      // grid is its programmatic dependent): wait for it before the first
      // load.  (kGemmDirect is launched plainly: this returns at once.)
      wait_for_prerequisite();
      uint32_t it = 0;
      for (int t = blockIdx.x; t < n_tiles && !*abort; t += gridDim.x) {
        int m0, n0;
        tile_of(t, n_tiles_n, bn, m0, n0);
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = static_cast<int>(it % stages);
          const uint32_t ph = (it / stages) & 1u;
          if (!mbar_wait(smem_u32(&sh.empty[s]), ph ^ 1u)) {
            *abort = 1;
            break;
          }
          unsigned char* st = smem + s * sbytes;
          const int seg = kMode == kGemmX ? 0 : kb / kps;
          const int xa = kMode == kGemmX ? kb * kBK : (kb - seg * kps) * kBK;
          const CUtensorMap* ma = seg == 0 ? &map_a0 : seg == 1 ? &map_a1 : &map_a2;
          mbar_expect_tx(&sh.full[s], kABytes + bn * kBK * 2);
          tma_load_2d(st, ma, xa, m0, &sh.full[s]);
          tma_load_2d(st + kABytes, &map_w, kb * kBK, n0, &sh.full[s]);
        }
      }
      // copies into this CTA's shared memory must have landed before it
      // can leave: wait (bounded) for the last use of every stage
      for (uint32_t q = it > stages ? it - stages : 0; q < it; ++q)
        mbar_wait(smem_u32(&sh.full[q % stages]), (q / stages) & 1u);
    }
  } else if (warp == 1) {
    // ---------------- MMAs
    if (lane == 0) {
      const uint32_t idesc = mma_idesc(kBM, bn);
      uint32_t it = 0, lt = 0;
      bool issued = false;
      uint64_t* last_commit = nullptr;
      uint32_t last_phase = 0;
      for (int t = blockIdx.x; t < n_tiles && !*abort; t += gridDim.x, ++lt) {
        const uint32_t a = lt & 1u, aph = (lt >> 1) & 1u;
        if (!mbar_wait(smem_u32(&sh.acc_empty[a]), aph ^ 1u)) {
          *abort = 1;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t acc = tmem + a * kAccCols;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = static_cast<int>(it % stages);
          const uint32_t ph = (it / stages) & 1u;
          if (!mbar_wait(smem_u32(&sh.full[s]), ph)) {
            *abort = 1;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t sa = smem_u32(smem + s * sbytes);
          const uint64_t da = sw128_desc(sa), db = sw128_desc(sa + kABytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // K slice kk: 16 elements = 32 bytes further along the swizzled row
            const uint32_t accumulate = (kb > 0 || kk > 0) ? 1u : 0u;
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(acc),
                "l"(da + 2 * kk), "l"(db + 2 * kk), "r"(idesc), "r"(accumulate)
                : "memory");
          }
          asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                           smem_u32(&sh.empty[s]))
                       : "memory");
          issued = true;
          last_commit = &sh.empty[s];
          last_phase = ph;
        }
        if (*abort) break;
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         smem_u32(&sh.acc_full[a]))
                     : "memory");
      }
      // the tensor core must be done with TMEM and the stages before they go
      if (issued && *abort) mbar_wait(smem_u32(last_commit), last_phase);
    }
  } else {
    // ---------------- epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    uint32_t lt = 0;
    for (int t = blockIdx.x; t < n_tiles && !*abort; t += gridDim.x, ++lt) {
      const uint32_t a = lt & 1u, aph = (lt >> 1) & 1u;
      if (!mbar_wait(smem_u32(&sh.acc_full[a]), aph)) {
        *abort = 1;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      int m0, n0;
      tile_of(t, n_tiles_n, bn, m0, n0);
      const int tok = m0 + row;
      const uint32_t base = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + a * kAccCols;
#pragma unroll 1
      for (int c = 0; c < bn; c += 32) {
        uint32_t r[32];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
            "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
              "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
              "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
              "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
            : "r"(base + c));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        const int n = n0 + c;
        if (tok < p.T && n < p.d_out) {
          float y[32];
#pragma unroll
          for (int j = 0; j < 32; ++j)
            y[j] = __uint_as_float(r[j]) + (p.bias != nullptr && n + j < p.d_out ? __ldg(p.bias + n + j) : 0.f);
          __nv_bfloat16* out = p.out + static_cast<size_t>(tok) * p.d_out + n;
          if (n + 32 <= p.d_out && p.out_vec) {
            uint4* o = reinterpret_cast<uint4*>(out);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              o[q] = make_uint4(pack_bf16(y[8 * q], y[8 * q + 1]), pack_bf16(y[8 * q + 2], y[8 * q + 3]),
                                pack_bf16(y[8 * q + 4], y[8 * q + 5]), pack_bf16(y[8 * q + 6], y[8 * q + 7]));
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (n + j < p.d_out) out[j] = __float2bfloat16_rn(y[j]);
          }
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      mbar_arrive(&sh.acc_empty[a]);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && sh.abort) atomicOr(p.err, kErrWait);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
}

// cuTensorMapEncodeTiled, fetched from the driver once.
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_tiled() {
  static EncodeTiled fn = nullptr;
  if (fn == nullptr) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(f);
  }
  return fn;
}

// A bf16 matrix [rows, K] (row stride K elements, 16-byte aligned) read in
// boxes of 64 x box_rows with the 128-byte swizzle; rows past the end read 0.
bool make_map(CUtensorMap* map, const void* base, int K, int rows, int box_rows) {
  EncodeTiled enc = encode_tiled();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t elem[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output tile width: of 256, 224, 192, 160 and 128 columns (multiples of
// 32 for the epilogue, at most the 256 columns of an accumulator slot) the
// one whose busiest CTA does the least work, ceil(tiles / SMs) x width (the
// widest on a tie): 4096 x 4096 on 152 SMs takes 224 (608 tiles, four full
// rounds) rather than 256 (512 tiles, the last of four rounds a third full).
int tile_width(int T, int d_out, int sms) {
  const int mt = (T + kBM - 1) / kBM;
  int best = kBNMax;
  long long best_cost = -1;
  for (int bn = kBNMax; bn >= 128; bn -= 32) {
    const long long tiles = static_cast<long long>(mt) * ((d_out + bn - 1) / bn);
    const long long cost = (tiles + sms - 1) / sms * bn;
    if (best_cost < 0 || cost < best_cost) {
      best = bn;
      best_cost = cost;
    }
  }
  return best;
}

// Stages of the ring for tile width bn: as many as fit in max_smem bytes of
// shared memory with the 1024 bytes of alignment room and the barriers
// (at most kMaxStages; build-time cap -DSV_FC_STAGES=<n>).
#ifndef SV_FC_STAGES
#define SV_FC_STAGES kMaxStages
#endif
int gemm_stages(int bn, int max_smem) {
  const int room = max_smem - 1024 - static_cast<int>(sizeof(GemmShared));
  const int n = room / stage_bytes(bn);
  const int cap = SV_FC_STAGES < kMaxStages ? SV_FC_STAGES : kMaxStages;
  return n < cap ? n : cap;
}

// Build-time switch -DSV_FC_DIRECT=0: SV_NORM_NONE also goes through X.
#ifndef SV_FC_DIRECT
#define SV_FC_DIRECT 1
#endif

template <int kMode>
cudaError_t launch_gemm(const FcNormProblem& p, const CUtensorMap& a0, const CUtensorMap& a1,
                        const CUtensorMap& a2, const CUtensorMap& w, int bn, int sms, bool dependent,
                        cudaStream_t s) {
  int dev = 0, max_smem = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
    return e;
  // as many stages as fit beside the barriers: five of 44 KB for bn = 224
  const int stages = gemm_stages(bn, max_smem);
  if (stages < 2) return cudaErrorInvalidValue;
  const int smem = stages * stage_bytes(bn) + 1024;  // + room to align the stages to 1024 bytes
  e = cudaFuncSetAttribute(fc_gemm_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int n_tiles = ((p.T + kBM - 1) / kBM) * ((p.d_out + bn - 1) / bn);
  const int grid = n_tiles < sms ? n_tiles : sms;
  // A programmatic dependent of the normalisation grid: its prologue (barrier
  // set-up, TMEM allocation) overlaps that grid's tail; its loads wait.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kFcThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, fc_gemm_kernel<kMode>, p, a0, a1, a2, w, bn, stages);
}

}  // namespace

// SV_NORM_NONE: kGemmDirect, the GEMM alone, reading the hidden states.
// LayerNorm / RMSNorm: the normalisation grid writes X, then kGemmX.
cudaError_t launch_fcnorm(const FcNormProblem& p, cudaStream_t s) {
  if (p.T <= 0 || p.d_out <= 0) return cudaSuccess;
  const int rows = p.T * 3;
  const bool direct = SV_FC_DIRECT && p.norm == kNormNone;
  cudaError_t e;
  if (!direct) {
    if (p.d <= kPrepMaxD && p.gb_vec)
      fcnorm_prep_rows_kernel<<<3 * ((p.T + kPrepRows - 1) / kPrepRows), 256, 0, s>>>(p);
    else
      fcnorm_prep_kernel<<<(rows * 32 + 255) / 256, 256, 0, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const int bn = tile_width(p.T, p.d_out, sms);
  CUtensorMap a0, a1, a2, w;
  if (!make_map(&w, p.w, 3 * p.d, p.d_out, bn)) return cudaErrorInvalidValue;
  if (!direct) {
    if (!make_map(&a0, p.x, 3 * p.d, p.T, kBM)) return cudaErrorInvalidValue;
    return launch_gemm<kGemmX>(p, a0, a0, a0, w, bn, sms, true, s);
  }
  if (!make_map(&a0, p.h[0], p.d, p.T, kBM) || !make_map(&a1, p.h[1], p.d, p.T, kBM) ||
      !make_map(&a2, p.h[2], p.d, p.T, kBM))
    return cudaErrorInvalidValue;
  return launch_gemm<kGemmDirect>(p, a0, a1, a2, w, bn, sms, false, s);
}

}  // namespace sv
