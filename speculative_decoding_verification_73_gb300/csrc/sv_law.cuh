// Cluster helpers, per-token target distributions and block sums shared by
// the kernels that walk a request with a whole thread-block cluster (the
// draft-tree walk and the lazy chain).
#pragma once

#include <cuda_bf16.h>

#include "sv_device.cuh"
#include "sv_pick.cuh"

namespace sv {
namespace {

// ------------------------------------------------------------ cluster helpers

__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Barrier over every thread of every CTA of the cluster; orders the memory
// accesses before it (release) with those after it (acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// The float at `local`'s place in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ float ld_dsmem(const float* local, unsigned rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(local))), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

// 16 bytes at `local`'s place in the shared memory of cluster CTA `rank`
// (16-byte aligned).
__device__ __forceinline__ float4 ld_dsmem16(const void* local, unsigned rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(local))), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(remote)
               : "memory");
  return v;
}

// ------------------------------------------------------------ distributions

// The distribution a node's token is drawn from, or that its next child is
// tested against, as a per-token function of the two logits.
//   kQ:       q_t = 2^(z_t k - cq) / sq
//   kSampled: after m rejections the residual r_m is a single clipped line in
//             (q, p): r_0 = q and r_{m+1} = (r_m - p)_+ / S_{m+1} give
//             r_m = (q - c_m p)_+ / D_m with c_{m+1} = c_m + D_m, D_{m+1} =
//             D_m S_{m+1} (c_0 = 0, D_0 = 1; a step whose sum S is 0 leaves r
//             unchanged).  The law evaluates (q - c p)_+ * scale.
//   kTopk:    q with the m rejected tokens removed (unnormalised)
struct NodeLaw {
  static constexpr int kQ = 0, kSampled = 1, kTopk = 2;
  int kind;
  float k, cq, inv_sq, cp, inv_sp;
  float c, scale;  // kSampled
  int m;           // kTopk: rejected tokens in rej[0, m)
  const int* rej;
  __device__ __forceinline__ float q(float zt) const { return ex2(fmaf(zt, k, -cq)) * inv_sq; }
  __device__ __forceinline__ float p(float yt) const { return ex2(fmaf(yt, k, -cp)) * inv_sp; }
  __device__ __forceinline__ float r(float zt, float yt, int t) const {
    float v = q(zt);
    if (kind == kSampled) {
      v = fmaxf(fmaf(-c, p(yt), v), 0.f) * scale;
    } else if (kind == kTopk) {
      for (int j = 0; j < m; ++j)
        if (rej[j] == t) v = 0.f;
    }
    return v;
  }
};

// Sums of f(z_t, y_t, t) over this thread's 32 tokens [t0, t0 + 32) of a
// level-1 block (0 past cend): h0 over the first 16, h1 over the last 16.
// One element of a row staged in shared memory, as float.
__device__ __forceinline__ float staged_elem(const float* p) { return *p; }
__device__ __forceinline__ float staged_elem(const __nv_bfloat16* p) {
  return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(p)) << 16);
}

// kSmem: z and y point into rows staged in shared memory (plain loads).
template <typename T, bool kVecPath, typename F, bool kSmem = false>
__device__ __forceinline__ void seg_sums(const T* z, const T* y, bool need_y, int t0, int cend, F f,
                                         float& h0, float& h1) {
  using E = Elem<T>;
  h0 = 0.f;
  h1 = 0.f;
  if (kVecPath) {
    constexpr int kVec = E::kVec;
    constexpr int kVecs = kSegTok / kVec;
    uint4 zv[kVecs], yv[kVecs];
#pragma unroll
    for (int i = 0; i < kVecs; ++i) {
      const int e0 = t0 + i * kVec;
      const bool in = e0 < cend;
      const uint4* zp = reinterpret_cast<const uint4*>(z + e0);
      const uint4* yp = reinterpret_cast<const uint4*>(y + e0);
      zv[i] = in ? (kSmem ? *zp : __ldg(zp)) : make_uint4(0, 0, 0, 0);
      yv[i] = (in && need_y) ? (kSmem ? *yp : __ldg(yp)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kVecs; ++i) {
      float part = 0.f;
#pragma unroll
      for (int e = 0; e < kVec; ++e) {
        const int t = t0 + i * kVec + e;
        if (t < cend) part += f(E::get(zv[i], e), need_y ? E::get(yv[i], e) : 0.f, t);
      }
      if (i < kVecs / 2)
        h0 += part;
      else
        h1 += part;
    }
  } else {
    for (int i = 0; i < kSegTok; ++i) {
      const int t = t0 + i;
      const float v = t < cend ? f(E::load1(z + t), need_y ? E::load1(y + t) : 0.f, t) : 0.f;
      if (i < kLevel3)
        h0 += v;
      else
        h1 += v;
    }
  }
}

// seg_sums over a level-1 block staged in shared memory in the layout of
// staged_at (bz, by: the block's staged rows; cbeg, cend: its tokens).  The
// same values summed in the same order as seg_sums, so the sums are equal
// bit for bit.
template <typename T, typename F>
__device__ __forceinline__ void seg_sums_staged(const T* bz, const T* by, bool need_y, int cbeg, int cend,
                                                F f, float& h0, float& h1) {
  using E = Elem<T>;
  constexpr int kVec = E::kVec;
  constexpr int kVecs = kSegTok / kVec;
  h0 = 0.f;
  h1 = 0.f;
  const int t0 = cbeg + static_cast<int>(threadIdx.x) * kSegTok;
  uint4 zv[kVecs], yv[kVecs];
#pragma unroll
  for (int i = 0; i < kVecs; ++i) {
    const bool in = t0 + i * kVec < cend;
    const int at = (i * kST + static_cast<int>(threadIdx.x)) * kVec;
    zv[i] = in ? *reinterpret_cast<const uint4*>(bz + at) : make_uint4(0, 0, 0, 0);
    yv[i] = (in && need_y) ? *reinterpret_cast<const uint4*>(by + at) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int i = 0; i < kVecs; ++i) {
    float part = 0.f;
#pragma unroll
    for (int e = 0; e < kVec; ++e) {
      const int t = t0 + i * kVec + e;
      if (t < cend) part += f(E::get(zv[i], e), need_y ? E::get(yv[i], e) : 0.f, t);
    }
    if (i < kVecs / 2)
      h0 += part;
    else
      h1 += part;
  }
}

// The sums of law.r over this thread's 32 staged tokens of a block, as
// seg_sums_staged gives them, with the q / p / residual of kQ and kSampled
// evaluated two tokens at a time by the paired float instructions (each
// lane performs the scalar law's operations, so every token's value and the
// sums are the same bit for bit); kTopk takes the scalar law.
template <typename T>
__device__ __forceinline__ void law_sums_staged(const NodeLaw& law, const T* bz, const T* by, bool need_y,
                                                int cbeg, int cend, float& h0, float& h1) {
  if (law.kind == NodeLaw::kTopk) {
    seg_sums_staged<T>(bz, by, need_y, cbeg, cend, [&](float zt, float yt, int t) { return law.r(zt, yt, t); },
                       h0, h1);
    return;
  }
  using E = Elem<T>;
  constexpr int kVec = E::kVec;
  constexpr int kVecs = kSegTok / kVec;
  h0 = 0.f;
  h1 = 0.f;
  const bool sampled = law.kind == NodeLaw::kSampled;
  const uint64_t k2 = f2pack(law.k, law.k);
  const uint64_t nq2 = f2pack(-law.cq, -law.cq), iq2 = f2pack(law.inv_sq, law.inv_sq);
  const uint64_t np2 = f2pack(-law.cp, -law.cp), ip2 = f2pack(law.inv_sp, law.inv_sp);
  const uint64_t nc2 = f2pack(-law.c, -law.c);
  const int t0 = cbeg + static_cast<int>(threadIdx.x) * kSegTok;
  uint4 zv[kVecs], yv[kVecs];
#pragma unroll
  for (int i = 0; i < kVecs; ++i) {
    const bool in = t0 + i * kVec < cend;
    const int at = (i * kST + static_cast<int>(threadIdx.x)) * kVec;
    zv[i] = in ? *reinterpret_cast<const uint4*>(bz + at) : make_uint4(0, 0, 0, 0);
    yv[i] = (in && need_y) ? *reinterpret_cast<const uint4*>(by + at) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int i = 0; i < kVecs; ++i) {
    float rv[kVec];
#pragma unroll
    for (int e = 0; e < E::kPairs; ++e) {
      float a0, a1;
      f2unpack(f2fma(E::pair(zv[i], e), k2, nq2), a0, a1);
      uint64_t v2 = f2mul(f2pack(ex2(a0), ex2(a1)), iq2);  // q
      if (sampled) {
        float b0, b1;
        f2unpack(f2fma(E::pair(yv[i], e), k2, np2), b0, b1);
        const uint64_t p2 = f2mul(f2pack(ex2(b0), ex2(b1)), ip2);
        float w0, w1;
        f2unpack(f2fma(nc2, p2, v2), w0, w1);  // q - c p
        v2 = f2pack(fmaxf(w0, 0.f) * law.scale, fmaxf(w1, 0.f) * law.scale);
      }
      f2unpack(v2, rv[2 * e], rv[2 * e + 1]);
    }
    float part = 0.f;
#pragma unroll
    for (int e = 0; e < kVec; ++e)
      if (t0 + i * kVec + e < cend) part += rv[e];
    if (i < kVecs / 2)
      h0 += part;
    else
      h1 += part;
  }
}

}  // namespace
}  // namespace sv
