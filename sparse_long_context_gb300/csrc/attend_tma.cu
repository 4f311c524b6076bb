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
#include "attend_tma.cuh"
#include "launch.h"

#include <algorithm>
#include <cudaTypedefs.h>

namespace sls {

constexpr int kTmaMinBlocks = 3;      // resident CTAs per SM the budgets are sized for
constexpr int kTmaStaged = 256;       // page-list entries staged in shared memory


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
  __shared__ ClusterInbox<D> inbox;                // cluster mode: partials pushed by the row's splits

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
  stage_page_list(s_pg, kTmaStaged, plist, sl.e0, sl.nent, a.Cap >> a.pshift, threadIdx.x, NT);
  __syncthreads();
  const int ngroups = (sl.nent << a.pshift) >> 4;
  const int b = row / a.Hkv, h = row % a.Hkv;
  const int G = a.G;

  float o[KS][4];
  float m_run = kNegInf, l_run = 0.f;
#pragma unroll
  for (int t = 0; t < KS; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;

  // the wait-timeout test hook: CTA 0 announces bytes for its first stage
  // that it never requests, and its waits poll briefly
  const bool plant = a.test_wait && blockIdx.x == 0;
  const uint32_t tries = plant ? kTestWaitTries : kWaitTries;

  if (warp == W) {
    // producer: lane 0 issues the copies of every group in order
    if (lane == 0) {
      bool ok = true;
      int issued = 0;
      for (int gi = 0; gi < ngroups; ++gi) {
        const int st = gi % NST;
        const uint32_t use = gi / NST;
        if (use > 0 && !mbar_wait(&empty[st], (use - 1) & 1, tries)) {
          ok = false;
          break;
        }
        int lim;
        const int base = group_base(a, sl, s_pg, plist, gi, lim);
        if (plant && gi == 0) {
          mbar_arrive_expect_tx(&full[st], 16);  // no copy is issued: this phase never completes
        } else if (lim > 0) {
          mbar_arrive_expect_tx(&full[st], L::STAGE);
          const int y = row * a.Cap + base;
          unsigned char* dst = ring + st * L::STAGE;
          tma_load_3d(dst, &tk, 0, y, 0, &full[st]);
          tma_load_3d(dst + L::GROUP, &tv, 0, y, 0, &full[st]);
        } else {
          mbar_arrive(&full[st]);  // nothing to copy: the phase completes at once
        }
        issued = gi + 1;
      }
      // every copy issued has landed before the CTA reuses or leaves the ring
      for (int gi = max(0, issued - NST); gi < issued; ++gi)
        if (!mbar_wait(&full[gi % NST], (gi / NST) & 1, tries)) ok = false;
      if (!ok) note_wait_timeout();
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
      if (!mbar_wait(&full[st], (gi / NST) & 1, tries)) {
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
      if (lane == 0) note_wait_timeout();
      // an infinite running max makes this warp's merge weight inf - inf = NaN
      // at every later merge, so the row's output and lse become NaN (a NaN
      // max would be dropped by fmaxf and the partial silently ignored)
      m_run = __int_as_float(0x7f800000);
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
  merge_warps<D, W>(o, G, sO, sM, sL, sF, sHm, sHl);
  const int GD = G * D;
  if (a.cluster) {
    cluster_push_combine<D, W, NT>(a, row, split, sO, sF, sHm, sHl, &inbox, true);
    return;
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

// The driver's tensor-map encoder, looked up once.  A function-local static
// with an initialiser is initialised exactly once even when several host
// threads call this together (C++11), so no thread sees a half-set state.
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return nullptr;
  }();
  return fn;
}

bool encode_rows_map(CUtensorMap* map, const void* base, uint64_t rows, int D) {
  auto fn = encode_fn();
  if (!fn) return false;
  // dims: 64 channels, rows, D/64 halves (the halves' stride, 128 bytes, is
  // smaller than the rows' one: the box lands as [half][16 rows][64])
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(D / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, 128};
  cuuint32_t box[3] = {64, 16, (cuuint32_t)(D / 64)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_bytes_map(CUtensorMap* map, const void* base, uint64_t rows, int row_bytes) {
  auto fn = encode_fn();
  if (!fn || (row_bytes != 128 && row_bytes % 16 != 0) || row_bytes > 256) return false;
  // rows of row_bytes bytes, box 16 rows; rows of exactly 128 bytes land
  // with the 128-byte swizzle (chunk c of row t at chunk c ^ (t % 8))
  cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {(cuuint32_t)row_bytes, 16};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
  if (!encode_rows_map(&tk, a.k, tokens, D) || !encode_rows_map(&tv, a.v, tokens, D)) return cudaSuccess;
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

DeviceStatus take_status_attend_tma() { return take_status_here(); }

}  // namespace sls
