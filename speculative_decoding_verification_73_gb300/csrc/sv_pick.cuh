// Pieces of the grouped inverse CDF shared by the chain sampler and the tree
// walk: CTA sums, the warp-wide inverse CDF over a list of masses, and the
// levels 2-4 choice inside one level-1 block of 8192 tokens.
#pragma once

#include "sv_device.cuh"

namespace sv {
namespace {

constexpr int kST = kSampleThreads;      // threads per sampler CTA
constexpr int kSegTok = kLevel1 / kST;   // tokens per thread in a level-1 block (32)
constexpr int kL2 = kLevel1 / kLevel2;   // level-2 blocks per level-1 block (32)
constexpr int kL3 = kLevel1 / kLevel3;   // level-3 blocks per level-1 block (512)
constexpr int kL3PerL2 = kLevel2 / kLevel3;  // 16
static_assert(kSegTok == 2 * kLevel3, "two level-3 blocks per thread");

// Staged layout of a level-1 block in shared memory: thread t owns tokens
// [32t, 32t + 32), and its i-th 16-byte vector sits at element
// (i * kST + t) * kVec, so the vector accesses of a warp (copies in, reads
// out) cover 512 consecutive bytes and meet no bank conflict.  staged_at
// maps a token offset in the block to its element.
template <typename T>
__device__ __forceinline__ int staged_at(int e) {
  constexpr int kVec = Elem<T>::kVec;
  const int th = e / kSegTok, r = e - th * kSegTok;
  return ((r / kVec) * kST + th) * kVec + (r % kVec);
}

__device__ __forceinline__ float cta_sum(float v, float* scratch) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  v = 0.f;
#pragma unroll
  for (int w = 0; w < kST / 32; ++w) v += scratch[w];
  __syncthreads();
  return v;
}

// Inverse CDF over n masses, evaluated by one whole warp (all lanes get the
// result): the smallest c with running sum C_c > u * C_{n-1}; if none, the
// last c with mass > 0; -1 if every mass is 0.  Masses are read through
// `get(i)`, once each when n <= 32; longer lists are scanned in tiles of 32
// twice (total, then the crossing) with identical arithmetic.
template <typename Get>
__device__ int warp_pick(Get get, int n, float u) {
  const int lane = threadIdx.x & 31;
  if (n <= 32) {
    const float m = lane < n ? get(lane) : 0.f;
    float incl = m;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned pos = __ballot_sync(kFull, m > 0.f);
    if (!pos) return -1;
    const float target = u * __shfl_sync(kFull, incl, 31);
    const unsigned hit = __ballot_sync(kFull, lane < n && incl > target);
    return hit ? __ffs(hit) - 1 : 31 - __clz(pos);
  }
  float carry = 0.f;
  int last_pos = -1;
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    const float m = i < n ? get(i) : 0.f;
    float incl = m;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned pos = __ballot_sync(kFull, m > 0.f);
    if (pos) last_pos = base + 31 - __clz(pos);
    carry += __shfl_sync(kFull, incl, 31);
  }
  if (last_pos < 0) return -1;
  const float target = u * carry;
  carry = 0.f;
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    const float m = i < n ? get(i) : 0.f;
    float incl = m;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned hit = __ballot_sync(kFull, i < n && carry + incl > target);
    if (hit) return base + __ffs(hit) - 1;
    carry += __shfl_sync(kFull, incl, 31);
  }
  return last_pos;
}

struct BlockScratch {
  float red[kST / 32];
  float l2[kL2];      // level-2 masses of the block
  float l3[kL3];      // level-3 masses of the block
  float l4[kLevel3];  // token masses of the chosen level-3 block
  int pick;
  int tok;
};

// From each thread's two level-3 masses of the level-1 block
// [cbeg, cbeg + kLevel1): the level-2 and level-1 masses (*mass), and the
// token the grouped inverse CDF picks inside the block at levels 2-4
// (u[1..3]), or -1 when the block has no mass.  r_at(t) re-evaluates r at
// token t (cbeg <= t < cend) for level 4 with the same arithmetic.  Called
// by the whole CTA.
template <typename RAt>
__device__ int block_pick(float h0, float h1, int cbeg, int cend, const Job& job, RAt r_at,
                          BlockScratch& sc, float* mass) {
  sc.l3[2 * threadIdx.x] = h0;
  sc.l3[2 * threadIdx.x + 1] = h1;
  float m2 = h0 + h1;  // level-2 mass: the 8 consecutive threads of a 256-token block
#pragma unroll
  for (int o = 1; o < kL3PerL2 / 2; o <<= 1) m2 += __shfl_xor_sync(kFull, m2, o);
  if ((threadIdx.x & (kL3PerL2 / 2 - 1)) == 0) sc.l2[threadIdx.x / (kL3PerL2 / 2)] = m2;
  *mass = cta_sum(h0 + h1, sc.red);  // its barriers also publish l2 and l3
  if (threadIdx.x < 32) {
    const int g2 = warp_pick([&](int i) { return sc.l2[i]; }, kL2, job.u[1]);
    int pick = -1;
    if (g2 >= 0) {
      const int g3 = warp_pick([&](int i) { return sc.l3[g2 * kL3PerL2 + i]; }, kL3PerL2, job.u[2]);
      pick = g2 * kL3PerL2 + max(g3, 0);
    }
    if (threadIdx.x == 0) sc.pick = pick;
  }
  __syncthreads();
  const int blk3 = sc.pick;
  if (blk3 < 0) return -1;  // CTA-uniform
  const int t0 = cbeg + blk3 * kLevel3;
  if (threadIdx.x < kLevel3) {
    const int t = t0 + threadIdx.x;
    sc.l4[threadIdx.x] = t < cend ? r_at(t) : 0.f;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int g4 = max(warp_pick([&](int i) { return sc.l4[i]; }, kLevel3, job.u[3]), 0);
    if (threadIdx.x == 0) sc.tok = t0 + g4;
  }
  __syncthreads();
  return sc.tok;
}

// block_pick for the kNB consecutive level-1 blocks starting at token c0
// (the first nb of them real, the last one cut at V): the same masses and
// tokens, bit for bit, as kNB calls of block_pick, with one set of CTA
// barriers for all the blocks.  Warp b picks levels 2-4 of block b, so kNB
// <= kST / 32.  r_at(b, t) re-evaluates r at token t of block b.
template <int kNB, typename RAt>
__device__ void blocks_pick(const float (&h0)[kNB], const float (&h1)[kNB], int c0, int V, int nb,
                            const Job& job, RAt r_at, BlockScratch (&sc)[kNB], float (&mass)[kNB],
                            int (&tok)[kNB]) {
  static_assert(kNB <= kST / 32, "one warp per block");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float tot[kNB];
#pragma unroll
  for (int b = 0; b < kNB; ++b) {
    sc[b].l3[2 * threadIdx.x] = h0[b];
    sc[b].l3[2 * threadIdx.x + 1] = h1[b];
    float m2 = h0[b] + h1[b];
#pragma unroll
    for (int o = 1; o < kL3PerL2 / 2; o <<= 1) m2 += __shfl_xor_sync(kFull, m2, o);
    if ((threadIdx.x & (kL3PerL2 / 2 - 1)) == 0) sc[b].l2[threadIdx.x / (kL3PerL2 / 2)] = m2;
    // CTA sum of h0 + h1 in cta_sum's order
    float v = h0[b] + h1[b];
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    if (lane == 0) sc[b].red[warp] = v;
  }
  __syncthreads();  // publishes l2, l3 and the warp sums
#pragma unroll
  for (int b = 0; b < kNB; ++b) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kST / 32; ++w) v += sc[b].red[w];
    tot[b] = v;
  }
  if (warp < nb) {  // warp-uniform
    const int b = warp;
    const int g2 = warp_pick([&](int i) { return sc[b].l2[i]; }, kL2, job.u[1]);
    int pick = -1;
    if (g2 >= 0) {
      const int g3 = warp_pick([&](int i) { return sc[b].l3[g2 * kL3PerL2 + i]; }, kL3PerL2, job.u[2]);
      pick = g2 * kL3PerL2 + max(g3, 0);
    }
    if (lane == 0) sc[b].pick = pick;
  }
  __syncthreads();
  if (warp < nb && lane < kLevel3) {
    const int b = warp;
    const int blk3 = sc[b].pick;
    if (blk3 >= 0) {
      const int cbeg = c0 + b * kLevel1;
      const int t = cbeg + blk3 * kLevel3 + lane;
      sc[b].l4[lane] = t < min(V, cbeg + kLevel1) ? r_at(b, t) : 0.f;
    }
  }
  __syncthreads();
  if (warp < nb) {
    const int b = warp;
    const int blk3 = sc[b].pick;
    int tk = -1;
    if (blk3 >= 0) {
      const int g4 = max(warp_pick([&](int i) { return sc[b].l4[i]; }, kLevel3, job.u[3]), 0);
      tk = c0 + b * kLevel1 + blk3 * kLevel3 + g4;
    }
    if (lane == 0) sc[b].tok = tk;
  }
  __syncthreads();
#pragma unroll
  for (int b = 0; b < kNB; ++b) {
    mass[b] = tot[b];
    tok[b] = b < nb ? sc[b].tok : -1;
  }
}

}  // namespace
}  // namespace sv
