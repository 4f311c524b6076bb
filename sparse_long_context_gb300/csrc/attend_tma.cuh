// Device pieces shared by the tensor-map fed kernels (the split-K attend
// kernel and the fused Quest decode step): the shared-memory stage layout,
// the tensor-core work on one 16-token group of K and V, and the combine of
// a row's splits inside a thread-block cluster.
//
// A stage holds 16 rows (tokens, or pages of metadata) of D bf16 channels,
// copied by one 3-D tensor-map box (64 channels x 16 rows x D/64 halves)
// with the 128-byte swizzle: half b of row t sits at b * 2048 + t * 128, and
// 16-byte chunk c of that half at chunk c ^ (t % 8), so that ldmatrix reads
// of 8 rows at one chunk hit 8 different bank groups.
#pragma once

#include <cooperative_groups.h>

#include "attend_common.cuh"
#include "mma.cuh"
#include "tma.cuh"

namespace sls {

constexpr int kTmaConsumers = 4;      // consumer warps per CTA
constexpr int kTmaStages = 8;         // ring stages (a multiple of the consumer warps)
constexpr int kMaxClusterSplits = 16;  // splits of a row that may combine inside one cluster
static_assert(kTmaStages % kTmaConsumers == 0, "a stage must always be consumed by the same warp");

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
struct TmaLayout {
  static constexpr int GROUP = 16 * D * 2;          // bytes of K (or V) of a 16-token group
  static constexpr int STAGE = 2 * GROUP;           // K then V
  static constexpr int BOX = 16 * 128;              // one 64-channel half: 16 rows of 128 bytes
  static constexpr size_t RING = (size_t)kTmaStages * STAGE;
  static constexpr size_t MERGE = (size_t)kTmaConsumers * 8 * D * sizeof(float);  // warps' accumulators
  static constexpr size_t SMEM = (RING > MERGE ? RING : MERGE) + 1024;  // + alignment slack
};

// The 16-token group's softmax and P.V once its raw scores are known: sc
// holds the QK sums of lane (r, m) (head r; n-tile nt, chain c: tokens
// 8 nt + 2m, +1), mul turns them into base-2 logits, and the group's V sits
// at shared address `vstage` in the swizzled layout.  Tokens at or past
// `lim` are masked (score -inf, V zero).
template <int D>
__device__ __forceinline__ void tma_softmax_pv(const float (&sc)[2][2][4], uint32_t vstage, int lim,
                                               float (&o)[D / 16][4], float& m_run, float& l_run, float mul,
                                               int lane) {
  using L = TmaLayout<D>;
  constexpr int KS = D / 16;
  const int m = lane & 3;
  const int j = lane >> 3, i = lane & 7;
  const int tok = 8 * (j >> 1) + i;
  auto row_addr = [&](uint32_t half_base, int c16) -> uint32_t {
    const int bx = c16 >> 3, c = c16 & 7;
    return half_base + bx * L::BOX + tok * 128 + ((c ^ i) << 4);
  };
  // lane (r, m): head r, tokens 2m, 2m+1 (n-tile 0) and 8+2m, 9+2m (n-tile 1)
  const int t0 = 2 * m;
  float s4[4];
  s4[0] = t0 < lim ? (sc[0][0][0] + sc[0][1][0]) * mul : kNegInf;
  s4[1] = t0 + 1 < lim ? (sc[0][0][1] + sc[0][1][1]) * mul : kNegInf;
  s4[2] = t0 + 8 < lim ? (sc[1][0][0] + sc[1][1][0]) * mul : kNegInf;
  s4[3] = t0 + 9 < lim ? (sc[1][0][1] + sc[1][1][1]) * mul : kNegInf;
  float gm = fmaxf(fmaxf(s4[0], s4[1]), fmaxf(s4[2], s4[3]));
  gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 1));
  gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 2));
  const float mn = fmaxf(m_run, gm);
  const bool live = mn != kNegInf;
  const float alpha = live ? ex2_approx(m_run - mn) : 1.f;
  m_run = mn;
  float p[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) p[k] = live ? ex2_approx(s4[k] - mn) : 0.f;
  l_run = fmaf(l_run, alpha, (p[0] + p[1]) + (p[2] + p[3]));
  const uint32_t pb0 = pack_bf16(p[0], p[1]), pb1 = pack_bf16(p[2], p[3]);
  // accumulator columns are heads 2m and 2m+1
  const float a_lo = __shfl_sync(0xffffffffu, alpha, 8 * m);
  const float a_hi = __shfl_sync(0xffffffffu, alpha, 8 * m + 4);
  if (!__all_sync(0xffffffffu, a_lo == 1.f && a_hi == 1.f)) {
#pragma unroll
    for (int t = 0; t < KS; ++t) {
      o[t][0] *= a_lo; o[t][1] *= a_hi; o[t][2] *= a_lo; o[t][3] *= a_hi;
    }
  }
  // V values of tokens past the context may be anything (even NaN): zero them
  const uint32_t mlo = (t0 < lim ? 0x0000ffffu : 0u) | (t0 + 1 < lim ? 0xffff0000u : 0u);
  const uint32_t mhi = (t0 + 8 < lim ? 0x0000ffffu : 0u) | (t0 + 9 < lim ? 0xffff0000u : 0u);
#pragma unroll
  for (int t = 0; t < KS; ++t) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4_t(row_addr(vstage, 2 * t + (j & 1)), a0, a1, a2, a3);
    if (lim < 16) {
      a0 &= mlo; a1 &= mlo; a2 &= mhi; a3 &= mhi;
    }
    mma_bf16(o[t], a0, a1, a2, a3, pb0, pb1);
  }
}

// One group from the stage at shared address `stage` (K, then V at +GROUP).
// Lane (r, m) supplies ldmatrix row addresses for matrix j = lane / 8, row
// i = lane % 8: token 8 * (j / 2) + i and 8-channel chunk 2 * step + (j % 2),
// which makes the four matrices the two n-tiles' (or the k-halves')
// fragments in the order the mma wants.
template <int D>
__device__ __forceinline__ void tma_group(uint32_t stage, int lim, const uint32_t (&qa)[D / 16][2],
                                          float (&o)[D / 16][4], float& m_run, float& l_run, float sl2,
                                          int lane) {
  using L = TmaLayout<D>;
  constexpr int KS = D / 16;
  const int j = lane >> 3, i = lane & 7;
  const int tok = 8 * (j >> 1) + i;
  // 128-byte swizzle: 16-byte chunk c of the row of token t sits at chunk c ^ (t % 8)
  auto row_addr = [&](uint32_t half_base, int c16) -> uint32_t {
    const int bx = c16 >> 3, c = c16 & 7;
    return half_base + bx * L::BOX + tok * 128 + ((c ^ i) << 4);
  };
  float sc[2][2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int c = 0; c < 2; ++c) sc[nt][c][0] = sc[nt][c][1] = sc[nt][c][2] = sc[nt][c][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    uint32_t b00, b01, b10, b11;
    ldsm_x4(row_addr(stage, 2 * ks + (j & 1)), b00, b01, b10, b11);
    mma_bf16(sc[0][ks & 1], qa[ks][0], 0u, qa[ks][1], 0u, b00, b01);
    mma_bf16(sc[1][ks & 1], qa[ks][0], 0u, qa[ks][1], 0u, b10, b11);
  }
  tma_softmax_pv<D>(sc, stage + L::GROUP, lim, o, m_run, l_run, sl2, lane);
}

// Merge of the consumer warps' online-softmax states (after the last
// group): warp w's accumulator goes to sO[w][head][D]; per head, thread g < G
// forms the weights f[w][g] = exp2(m_w - M) and the CTA's max M (natural log)
// and sum.  Ends with a barrier over the CTA.
template <int D, int W>
__device__ __forceinline__ void merge_warps(const float (&o)[D / 16][4], int G, float* sO, float (*sM)[8],
                                            float (*sL)[8], float (*sF)[8], float* sHm, float* sHl) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < W) {
    const int r = lane >> 2, m = lane & 3;
#pragma unroll
    for (int t = 0; t < D / 16; ++t) {
      const int ch = 16 * t + r;
      sO[(warp * 8 + 2 * m) * D + ch] = o[t][0];
      sO[(warp * 8 + 2 * m + 1) * D + ch] = o[t][1];
      sO[(warp * 8 + 2 * m) * D + ch + 8] = o[t][2];
      sO[(warp * 8 + 2 * m + 1) * D + ch + 8] = o[t][3];
    }
  }
  if (threadIdx.x < G) {
    const int g = threadIdx.x;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < W; ++w) M = fmaxf(M, sM[w][g]);
    float Lh = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const float f = (M == kNegInf || sM[w][g] == kNegInf) ? 0.f : exp2f(sM[w][g] - M);
      sF[w][g] = f;
      Lh = fmaf(sL[w][g], f, Lh);
    }
    sHm[g] = M == kNegInf ? kNegInf : M * kLn2;
    sHl[g] = Lh;
  }
  __syncthreads();
}

// Receive buffers of the cluster combine (in the owner CTA's shared memory).
// 16-byte aligned: the combine moves its values as float4 (a static
// __shared__ instance would otherwise only be 4-byte aligned).
template <int D>
struct __align__(16) ClusterInbox {
  float o[8 * D + 4 * kMaxClusterSplits];  // S shares of round4(ceil(G D / S)) values
  float m[kMaxClusterSplits * 8];
  float l[kMaxClusterSplits * 8];
};

// Stage two inside the row's cluster: split `split` (= cluster rank) of S
// pushes its merged partial into the inboxes of the CTAs owning the outputs
// (rank r owns a contiguous share of the G x D outputs), one cluster barrier
// publishes the pushes, and each owner combines its share locally, the sink
// logit joining the normaliser once.  With wait_first the caller has an
// outstanding "barrier.cluster.arrive.relaxed" from the kernel's start, and
// its wait here guarantees that every peer runs before its shared memory is
// written; without it the caller has already synchronised the cluster.
// After this call nothing reads the CTA's shared memory any more.
template <int D, int W, int NT>
__device__ __forceinline__ void cluster_push_combine(const AttendArgs& a, int row, int split, const float* sO,
                                                     const float (*sF)[8], const float* sHm, const float* sHl,
                                                     ClusterInbox<D>* inbox, bool wait_first) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  const int S = a.S, G = a.G, GD = G * D;
  const int b = row / a.Hkv, h = row % a.Hkv;
  // owner r holds the values [r chunk, (r + 1) chunk): a multiple of 4, so
  // that every float4 below stays inside one head and one owner (D % 4 == 0)
  const int chunk = ((GD + S - 1) / S + 3) & ~3;
  if (wait_first) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  for (int it = 4 * threadIdx.x; it < GD; it += 4 * NT) {
    const int g = it / D, d = it % D;
    float4 av = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const float4 x = *reinterpret_cast<const float4*>(sO + (w * 8 + g) * D + d);
      const float f = sF[w][g];
      av.x = fmaf(x.x, f, av.x);
      av.y = fmaf(x.y, f, av.y);
      av.z = fmaf(x.z, f, av.z);
      av.w = fmaf(x.w, f, av.w);
    }
    const int owner = it / chunk;
    *reinterpret_cast<float4*>(cl.map_shared_rank(inbox->o, owner) + split * chunk + (it - owner * chunk)) = av;
  }
  if (threadIdx.x < S * G) {
    const int owner = threadIdx.x / G, g = threadIdx.x % G;
    cl.map_shared_rank(inbox->m, owner)[split * 8 + g] = sHm[g];
    cl.map_shared_rank(inbox->l, owner)[split * 8 + g] = sHl[g];
  }
  cl.sync();
  const size_t hq0 = (size_t)b * a.Hq + (size_t)h * G;
  const int i0 = split * chunk, i1 = min(GD, i0 + chunk);
  for (int it = i0 + 4 * threadIdx.x; it < i1; it += 4 * NT) {
    const int g = it / D, d = it % D;
    float M = kNegInf;
    for (int s = 0; s < S; ++s) M = fmaxf(M, inbox->m[s * 8 + g]);
    const float sk = a.sink ? a.sink[h * G + g] : kNegInf;
    M = fmaxf(M, sk);
    float Ls = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < S; ++s) {
      const float ms = inbox->m[s * 8 + g];
      if (ms == kNegInf || M == kNegInf) continue;
      const float w = expf(ms - M);
      Ls = fmaf(inbox->l[s * 8 + g], w, Ls);
      const float4 x = *reinterpret_cast<const float4*>(inbox->o + s * chunk + (it - i0));
      acc.x = fmaf(x.x, w, acc.x);
      acc.y = fmaf(x.y, w, acc.y);
      acc.z = fmaf(x.z, w, acc.z);
      acc.w = fmaf(x.w, w, acc.w);
    }
    if (a.sink && M != kNegInf) Ls += expf(sk - M);
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    __nv_bfloat162* op = reinterpret_cast<__nv_bfloat162*>(static_cast<bf16*>(a.out) + (hq0 + g) * D + d);
    op[0] = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    op[1] = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    if (d == 0 && a.lse) a.lse[hq0 + g] = Ls == 0.f ? kNegInf : M + logf(Ls);
  }
}

// Host: 3-D tensor map over `rows` rows of D bf16 channels (a K or V cache
// viewed as [tokens, D], or page metadata as [pages, D]), box 64 x 16 x D/64.
bool encode_rows_map(CUtensorMap* map, const void* base, uint64_t rows, int D);
// Host: 2-D tensor map over `rows` rows of row_bytes bytes (thumbnail codes
// or 8-bit residuals), box row_bytes x 16 rows; rows of 128 bytes use the
// 128-byte swizzle.  False if the driver refuses it.
bool encode_bytes_map(CUtensorMap* map, const void* base, uint64_t rows, int row_bytes);

}  // namespace sls
