// Tensor-core split-K sparse decode attention for bf16 page lists with pages
// of 16 tokens or more, fed by the tensor memory accelerator (stage one of
// two-stage flash-decoding over the selected pages; "Don't read the
// haystack", Part one, and its sparse counterpart in Part two).
//
// One CTA per (row, split): one producer warp and W consumer warps around a
// ring of NST shared-memory stages.  A stage holds one 16-token group (16
// contiguous tokens of one page) of K and of V, copied by 64-channel boxes
// of 2-D tensor maps over the caches ([rows * Cap tokens, D] bf16) with the
// 128-byte swizzle, so that the ldmatrix reads below are free of bank
// conflicts.  The producer's lane 0 walks the CTA's groups in order; stage
// s is consumed by warp s % W, which keeps its own online softmax:
//   S^T = Q K^T    m16n8k16, A = Q (the G <= 8 heads of the GQA group as
//                  rows, zero-padded to 16), B = K^T from ldmatrix;
//   online softmax per head on the accumulators (base 2);
//   O^T += V^T P^T A = V^T from transposed ldmatrix, B = P^T, which is the
//                  QK accumulator of the same lanes packed to bf16.
// Each K and V byte is read from memory once for all heads of the group.
// Tokens of a group that lie past the context are masked: their scores are
// set to -inf and their V values to zero before the product.
#include "attend_common.cuh"
#include "launch.h"
#include "mma.cuh"
#include "tma.cuh"

#include <algorithm>
#include <cooperative_groups.h>
#include <cudaTypedefs.h>

namespace sls {

constexpr int kTmaConsumers = 4;      // consumer warps per CTA
constexpr int kTmaStages = 8;         // ring stages (a multiple of the consumer warps)
constexpr int kTmaMinBlocks = 3;      // resident CTAs per SM the budgets are sized for
constexpr int kTmaStaged = 256;       // page-list entries staged in shared memory
constexpr int kMaxClusterSplits = 16;  // splits of a row that may combine inside one cluster
static_assert(kTmaStages % kTmaConsumers == 0, "a stage must always be consumed by the same warp");

__device__ unsigned int g_attend_wait_timeouts = 0;

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
struct TmaLayout {
  static constexpr int GROUP = 16 * D * 2;          // bytes of K (or V) of a 16-token group
  static constexpr int STAGE = 2 * GROUP;           // K then V
  static constexpr int BOX = 16 * 128;              // one 64-channel box: 16 rows of 128 bytes
  static constexpr int NBOX = D / 64;
  static constexpr size_t RING = (size_t)kTmaStages * STAGE;
  static constexpr size_t MERGE = (size_t)kTmaConsumers * 8 * D * sizeof(float);  // warps' accumulators
  static constexpr size_t SMEM = (RING > MERGE ? RING : MERGE) + 1024;  // + alignment slack
};

// First cache position of group gi of the slice and the number of its tokens
// inside the context (<= 0 when the group is empty: padded entry, page out
// of range or past the context).
__device__ __forceinline__ int group_base(const AttendArgs& a, const Slice& sl, const int* s_pg,
                                          const int32_t* plist, int gi, int& lim) {
  const int j0 = gi << 4;
  const int e = j0 >> a.pshift;
  const int pg = e < kTmaStaged ? s_pg[e] : (plist ? __ldg(plist + e) : sl.e0 + e);
  lim = 0;
  if ((unsigned)pg >= (unsigned)(a.Cap >> a.pshift)) return 0;
  const int base = (pg << a.pshift) + (j0 & (a.P - 1));
  lim = min(sl.N - base, 16);
  return base;
}

// One group from the stage at shared address `stage`.  Lane (r, m) supplies
// ldmatrix row addresses for matrix j = lane / 8, row i = lane % 8: token
// 8 * (j / 2) + i and 8-channel chunk 2 * step + (j % 2), which makes the
// four matrices the two n-tiles' (or the k-halves') fragments in the order
// the mma wants.
template <int D>
__device__ __forceinline__ void tma_group(uint32_t stage, int lim, const uint32_t (&qa)[D / 16][2],
                                          float (&o)[D / 16][4], float& m_run, float& l_run, float sl2,
                                          int lane) {
  using L = TmaLayout<D>;
  constexpr int KS = D / 16;
  const int m = lane & 3;
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
  // lane (r, m): head r, tokens 2m, 2m+1 (n-tile 0) and 8+2m, 9+2m (n-tile 1)
  const int t0 = 2 * m;
  float s4[4];
  s4[0] = t0 < lim ? (sc[0][0][0] + sc[0][1][0]) * sl2 : kNegInf;
  s4[1] = t0 + 1 < lim ? (sc[0][0][1] + sc[0][1][1]) * sl2 : kNegInf;
  s4[2] = t0 + 8 < lim ? (sc[1][0][0] + sc[1][1][0]) * sl2 : kNegInf;
  s4[3] = t0 + 9 < lim ? (sc[1][0][1] + sc[1][1][1]) * sl2 : kNegInf;
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
  const uint32_t vstage = stage + L::GROUP;
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

template <int D>
__global__ void __launch_bounds__((kTmaConsumers + 1) * 32, kTmaMinBlocks)
attend_tma_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                  const AttendArgs a) {
  using L = TmaLayout<D>;
  constexpr int W = kTmaConsumers, NST = kTmaStages, KS = D / 16;
  constexpr int NT = (W + 1) * 32;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* ring = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t full[NST], empty[NST];
  __shared__ int s_pg[kTmaStaged];
  __shared__ float sM[W][8], sL[W][8], sF[W][8];  // warps' max, sum and merge weight per head
  __shared__ float sHm[8], sHl[8];                 // the CTA's merged max (natural log) and sum
  // cluster mode: the partials pushed here by the row's splits (this CTA owns
  // a contiguous share of the row's G x D outputs)
  __shared__ float s_in_o[8 * D + kMaxClusterSplits];
  __shared__ float s_in_m[kMaxClusterSplits * 8], s_in_l[kMaxClusterSplits * 8];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // every CTA of the cluster announces that it runs; the matching wait comes
  // before the first write into a peer's shared memory
  if (a.cluster) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_fence_init();
    tma_prefetch_map(&tk);
    tma_prefetch_map(&tv);
  }
  pdl_wait();

  const int row = blockIdx.x / a.S, split = blockIdx.x % a.S;
  const Slice sl = attend_slice(a, row, split);
  const int32_t* plist = a.page_idx ? a.page_idx + (size_t)row * a.idx_stride + sl.e0 : nullptr;
  for (int e = threadIdx.x; e < min(sl.nent, kTmaStaged); e += NT) s_pg[e] = plist ? __ldg(plist + e) : sl.e0 + e;
  __syncthreads();
  const int ngroups = (sl.nent << a.pshift) >> 4;
  const int b = row / a.Hkv, h = row % a.Hkv;
  const int G = a.G;

  float o[KS][4];
  float m_run = kNegInf, l_run = 0.f;
#pragma unroll
  for (int t = 0; t < KS; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;

  if (warp == W) {
    // producer: lane 0 issues the copies of every group in order
    if (lane == 0) {
      bool ok = true;
      int issued = 0;
      for (int gi = 0; gi < ngroups; ++gi) {
        const int st = gi % NST;
        const uint32_t use = gi / NST;
        if (use > 0 && !mbar_wait(&empty[st], (use - 1) & 1)) {
          ok = false;
          break;
        }
        int lim;
        const int base = group_base(a, sl, s_pg, plist, gi, lim);
        if (lim > 0) {
          mbar_arrive_expect_tx(&full[st], L::STAGE);
          const int y = row * a.Cap + base;
          unsigned char* dst = ring + st * L::STAGE;
#pragma unroll
          for (int bx = 0; bx < L::NBOX; ++bx) tma_load_2d(dst + bx * L::BOX, &tk, 64 * bx, y, &full[st]);
#pragma unroll
          for (int bx = 0; bx < L::NBOX; ++bx)
            tma_load_2d(dst + L::GROUP + bx * L::BOX, &tv, 64 * bx, y, &full[st]);
        } else {
          mbar_arrive(&full[st]);  // nothing to copy: the phase completes at once
        }
        issued = gi + 1;
      }
      // every copy issued has landed before the CTA reuses or leaves the ring
      for (int gi = max(0, issued - NST); gi < issued; ++gi)
        if (!mbar_wait(&full[gi % NST], (gi / NST) & 1)) ok = false;
      if (!ok) atomicAdd(&g_attend_wait_timeouts, 1u);
    }
  } else {
    const int r = lane >> 2, m = lane & 3;
    // Q as the A operand: a0 = Q[head r][16ks + 2m, +1], a2 = Q[r][16ks + 8 + 2m, +1]
    uint32_t qa[KS][2];
    const bf16* qp = static_cast<const bf16*>(a.q) + ((size_t)b * a.Hq + (size_t)h * G + r) * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qa[ks][0] = r < G ? __ldg(reinterpret_cast<const uint32_t*>(qp + 16 * ks + 2 * m)) : 0u;
      qa[ks][1] = r < G ? __ldg(reinterpret_cast<const uint32_t*>(qp + 16 * ks + 8 + 2 * m)) : 0u;
    }
    const float sl2 = a.qscale;
    const uint32_t ring_u32 = smem_u32(ring);
    bool ok = true;
    for (int gi = warp; gi < ngroups; gi += W) {
      const int st = gi % NST;
      if (!mbar_wait(&full[st], (gi / NST) & 1)) {
        ok = false;
        break;
      }
      int lim;
      group_base(a, sl, s_pg, plist, gi, lim);
      if (lim > 0) tma_group<D>(ring_u32 + st * L::STAGE, lim, qa, o, m_run, l_run, sl2, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (!ok) {
      if (lane == 0) atomicAdd(&g_attend_wait_timeouts, 1u);
      m_run = __int_as_float(0x7fffffff);  // the row's output becomes NaN
    }
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    if (m == 0) {
      sM[warp][r] = m_run;
      sL[warp][r] = l_run;
    }
  }
  __syncthreads();  // every stage has been consumed (or drained): the ring becomes the merge area

  float* sO = reinterpret_cast<float*>(ring);  // [W][8 heads][D]
  if (warp < W) {
    const int r = lane >> 2, m = lane & 3;
#pragma unroll
    for (int t = 0; t < KS; ++t) {
      const int ch = 16 * t + r;
      sO[(warp * 8 + 2 * m) * D + ch] = o[t][0];
      sO[(warp * 8 + 2 * m + 1) * D + ch] = o[t][1];
      sO[(warp * 8 + 2 * m) * D + ch + 8] = o[t][2];
      sO[(warp * 8 + 2 * m + 1) * D + ch + 8] = o[t][3];
    }
  }
  // per head: the warps' weights exp2(m_w - M) and the CTA's max and sum
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
  const int GD = G * D;
  if (a.cluster) {
    // stage two inside the row's cluster: each split pushes its merged
    // partial into the shared memory of the CTAs owning the outputs, one
    // cluster barrier publishes the pushes, each owner combines locally
    namespace cg = cooperative_groups;
    cg::cluster_group cl = cg::this_cluster();
    const int S = a.S;
    const int chunk = (GD + S - 1) / S;
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    for (int it = threadIdx.x; it < GD; it += NT) {
      const int g = it / D, d = it % D;
      float av = 0.f;
#pragma unroll
      for (int w = 0; w < W; ++w) av = fmaf(sO[(w * 8 + g) * D + d], sF[w][g], av);
      const int owner = it / chunk;
      cl.map_shared_rank(s_in_o, owner)[split * chunk + (it - owner * chunk)] = av;
    }
    if (threadIdx.x < S * G) {
      const int owner = threadIdx.x / G, g = threadIdx.x % G;
      cl.map_shared_rank(s_in_m, owner)[split * 8 + g] = sHm[g];
      cl.map_shared_rank(s_in_l, owner)[split * 8 + g] = sHl[g];
    }
    cl.sync();
    const size_t hq0 = (size_t)b * a.Hq + (size_t)h * G;
    const int i0 = split * chunk, i1 = min(GD, i0 + chunk);
    for (int it = i0 + threadIdx.x; it < i1; it += NT) {
      const int g = it / D, d = it % D;
      float M = kNegInf;
      for (int s = 0; s < S; ++s) M = fmaxf(M, s_in_m[s * 8 + g]);
      const float sk = a.sink ? a.sink[h * G + g] : kNegInf;
      M = fmaxf(M, sk);
      float Ls = 0.f, acc = 0.f;
      for (int s = 0; s < S; ++s) {
        const float ms = s_in_m[s * 8 + g];
        if (ms == kNegInf || M == kNegInf) continue;
        const float w = expf(ms - M);
        Ls = fmaf(s_in_l[s * 8 + g], w, Ls);
        acc = fmaf(s_in_o[s * chunk + (it - i0)], w, acc);
      }
      if (a.sink && M != kNegInf) Ls += expf(sk - M);
      static_cast<bf16*>(a.out)[(hq0 + g) * D + d] = __float2bfloat16_rn(Ls > 0.f ? acc / Ls : 0.f);
      if (d == 0 && a.lse) a.lse[hq0 + g] = Ls > 0.f ? M + logf(Ls) : kNegInf;
    }
    return;  // nothing reads this CTA's shared memory after the barrier
  }
  for (int it = threadIdx.x; it < GD; it += NT) {
    const int g = it / D, d = it % D;
    float av = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) av = fmaf(sO[(w * 8 + g) * D + d], sF[w][g], av);
    const size_t hq = (size_t)b * a.Hq + (size_t)h * G + g;
    a.o_part[(hq * a.S + split) * D + d] = av;
    if (d == 0) {
      a.m_part[hq * a.S + split] = sHm[g];
      a.l_part[hq * a.S + split] = sHl[g];
    }
  }
  if (a.tickets) combine_row_if_last<bf16, D, NT>(a, row, a.S);
}

// ---------------------------------------------------------------- host side

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// [tokens, D] bf16 rows of D * 2 bytes; 64-channel x 16-token boxes, 128-byte swizzle.
static bool encode_cache_map(CUtensorMap* map, const void* base, uint64_t tokens, int D) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)tokens};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, 16};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool attend_tma_eligible(const Shape& s) {
  return s.dtype == 1 && !(s.flags & 3) && s.G <= 8 && s.P >= 16 && (s.D == 64 || s.D == 128) &&
         (long long)s.B * s.Hkv * s.Cap < (1ll << 31) && encode_fn() != nullptr;
}

template <int D>
static int tma_per_sm() {
  static int per_sm = 0;
  if (per_sm == 0) {
    cudaFuncSetAttribute(attend_tma_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)TmaLayout<D>::SMEM);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attend_tma_kernel<D>, (kTmaConsumers + 1) * 32,
                                                      TmaLayout<D>::SMEM) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
  }
  return per_sm;
}

int attend_tma_per_sm(const Shape& s) { return s.D == 64 ? tma_per_sm<64>() : tma_per_sm<128>(); }

// Whether clusters of S attend CTAs can be resident (cached per S).
template <int D>
static int tma_max_clusters(int S);
template <int D>
static bool tma_cluster_ok(int S) {
  return tma_max_clusters<D>(S) > 0;
}
template <int D>
static int tma_max_clusters(int S) {
  static int ok[kMaxClusterSplits + 1] = {0};
  if (ok[S] == 0) {
    cudaFuncSetAttribute(attend_tma_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TmaLayout<D>::SMEM);
    if (S > 8)  // more than the portable cluster size
      cudaFuncSetAttribute(attend_tma_kernel<D>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S);
    cfg.blockDim = dim3((kTmaConsumers + 1) * 32);
    cfg.dynamicSmemBytes = TmaLayout<D>::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    const bool good = cudaOccupancyMaxActiveClusters(&n, attend_tma_kernel<D>, &cfg) == cudaSuccess && n > 0;
    ok[S] = good ? n : -1;
  }
  return ok[S];
}

// Splits per row for the fused call: about two CTAs per SM over all rows
// (the per-SM read rate, not the CTA count, bounds this kernel, and a third
// CTA on some SMs lengthens the slowest), at least four 16-token groups per
// split, at most one cluster, and no more clusters than fit at once.
int attend_tma_splits(const Shape& s, int groups_per_row) {
  const int rows = s.B * s.Hkv;
  int S = (2 * sm_count()) / rows + 1;
  S = std::min(S, std::max(1, groups_per_row / 4));
  S = std::min(S, kMaxClusterSplits);
  while (S > 1) {
    const int fit = s.D == 64 ? tma_max_clusters<64>(S) : tma_max_clusters<128>(S);
    if (fit <= 0 || fit >= rows || rows > fit * 4) break;  // unknown, one wave, or many waves anyway
    --S;
  }
  return std::max(S, 1);
}

template <int D>
static cudaError_t tma_launch(const Shape& s, const AttendArgs& a, cudaStream_t st, bool* handled) {
  CUtensorMap tk, tv;
  const uint64_t tokens = (uint64_t)s.B * s.Hkv * s.Cap;
  if (!encode_cache_map(&tk, a.k, tokens, D) || !encode_cache_map(&tv, a.v, tokens, D)) return cudaSuccess;
  *handled = true;
  cudaError_t e = cudaFuncSetAttribute(attend_tma_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)TmaLayout<D>::SMEM);
  if (e != cudaSuccess) return e;
  AttendArgs ac = a;
  // fused calls combine inside the row's cluster (a single CTA is a cluster of one)
  ac.cluster = (a.tickets && a.S <= kMaxClusterSplits && (a.S == 1 || tma_cluster_ok<D>(a.S))) ? 1 : 0;
  e = launch_pdl_cluster(attend_tma_kernel<D>, dim3(s.B * s.Hkv * a.S), dim3((kTmaConsumers + 1) * 32),
                         TmaLayout<D>::SMEM, ac.cluster ? a.S : 1, st, tk, tv, ac);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_attend_tma(const Shape& s, const AttendArgs& a, cudaStream_t st, bool* handled) {
  *handled = false;
  if (!attend_tma_eligible(s) || a.S < 1) return cudaSuccess;
  // tensor maps want 16-byte aligned bases
  if ((reinterpret_cast<uintptr_t>(a.k) | reinterpret_cast<uintptr_t>(a.v)) & 15) return cudaSuccess;
  return s.D == 64 ? tma_launch<64>(s, a, st, handled) : tma_launch<128>(s, a, st, handled);
}

unsigned int take_attend_wait_timeouts() {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_attend_wait_timeouts, sizeof(v)) != cudaSuccess) return 0;
  if (v) {
    const unsigned int zero = 0;
    cudaMemcpyToSymbol(g_attend_wait_timeouts, &zero, sizeof(zero));
  }
  return v;
}

}  // namespace sls
