// Tensor-core split-K sparse decode attention for bf16 (stage one of
// two-stage flash-decoding over a page list; "Don't read the haystack",
// Part one and the sparse twin of Part two).
//
// One CTA per (row, split) with 4 warps; each warp walks 16-token groups
// of the split's slice and keeps its own online softmax.  Per group:
//   S^T = Q K^T   m16n8k16 with A = Q (the G <= 8 heads of the GQA group
//                 as rows, zero-padded to 16) and B = K^T (two n-tiles of
//                 8 tokens), fed straight from 16-byte loads of K;
//   online softmax per head on the accumulator registers (base 2);
//   O^T += V^T P^T   with A = V^T (channels as rows) built from 16-byte
//                 loads of V by byte permutes, and B = P^T, which is the
//                 QK accumulator of the same lanes packed to bf16.
// Every K and V byte of a group is read once by one warp, for all heads of
// the group (GQA sharing).  The warps merge in shared memory at the end.
#include "attend_common.cuh"
#include "launch.h"
#include "mma.cuh"

namespace sls {

// A warp walks 16-token groups of its slice with two groups in flight in
// registers: the loads of group g + NW are issued before group g is computed
// (register loads keep more bytes in flight per SM for this gather than
// shared-memory staging does).  Per group, lane (r, m) holds:
//   K rows of tokens r and r + 8, NS 16-byte chunks each (B operand of S^T),
//   V of tokens 2m, 2m+1, 2m+8, 2m+9, VL chunks each (A operand of O^T),
// and the positions that decide which tokens are valid.
constexpr int kAttnWarps = 8;
// Resident CTAs per SM the register budget is sized for: one at D = 128;
// two at D = 64, whose groups need half the registers, so that twice the
// warps keep gathers in flight (one-token pages gather single 128-byte rows).
template <int D>
constexpr int attn_min_blocks() { return D == 64 ? 2 : 1; }
constexpr int kStagedEntries = 1024;  // page-list entries staged in shared memory

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// A contiguous run of one row's token list handled by one CTA: tokens
// j = 0 .. ntok-1 of the run sit at list position joff + j after entry e0
// (entry = e0 + ((joff + j) >> log2 P), offset in the page = (joff + j) & (P-1)).
struct Seg {
  int N, e0, joff, ntok, nent;
};

template <int D>
struct Group {
  static constexpr int NS = D / 32, VL = D / 64;
  uint4 kc[2][NS];
  uint4 vc[4][VL];
  int pv[4];
};

// Positions (or -1) of the tokens lane (r, m) touches in group gi.  With
// pages of at least 16 tokens a group lies inside one page, so the lane
// derives them from the group's page without shuffles.
template <bool PAGED>
__device__ __forceinline__ void group_positions(const AttendArgs& a, const Seg& sl, const int* s_pg,
                                                const int32_t* plist, int gi, int lane, int& pk0, int& pk1,
                                                int (&pv)[4]) {
  const int r = lane >> 2, m = lane & 3;
  const int ntok = sl.ntok;
  if constexpr (PAGED) {
    const int j0 = gi << 4;  // a 16-token group starts at a multiple of 16 and stays inside one page
    int base = -1, lim = 0;
    if (j0 < ntok) {
      const int J = sl.joff + j0;
      const int e = J >> a.pshift;
      const int pg = e < kStagedEntries ? s_pg[e] : (plist ? __ldg(plist + e) : sl.e0 + e);
      if ((unsigned)pg < (unsigned)(a.Cap >> a.pshift)) {
        base = (pg << a.pshift) + (J & (a.P - 1));
        lim = min(sl.N - base, ntok - j0);  // inside the context and inside the run
      }
    }
    auto at = [&](int t) { return (base >= 0 && t < lim) ? base + t : -1; };
    pk0 = at(r);
    pk1 = at(r + 8);
    pv[0] = at(2 * m);
    pv[1] = at(2 * m + 1);
    pv[2] = at(2 * m + 8);
    pv[3] = at(2 * m + 9);
  } else {
    int mypos = -1;
    const int j = (gi << 4) + (lane & 15);
    if (j < ntok) {
      const int J = sl.joff + j;
      const int e = J >> a.pshift;
      const int pg = e < kStagedEntries ? s_pg[e] : (plist ? __ldg(plist + e) : sl.e0 + e);
      mypos = token_position(a, pg, J, sl.N);
    }
    pk0 = __shfl_sync(0xffffffffu, mypos, r);
    pk1 = __shfl_sync(0xffffffffu, mypos, r + 8);
    pv[0] = __shfl_sync(0xffffffffu, mypos, 2 * m);
    pv[1] = __shfl_sync(0xffffffffu, mypos, 2 * m + 1);
    pv[2] = __shfl_sync(0xffffffffu, mypos, 2 * m + 8);
    pv[3] = __shfl_sync(0xffffffffu, mypos, 2 * m + 9);
  }
}

template <int D, bool PAGED>
__device__ __forceinline__ void load_group(Group<D>& g, const AttendArgs& a, const Seg& sl, const int* s_pg,
                                           const int32_t* plist, int gi, const bf16* kl, const bf16* vl) {
  constexpr int NS = Group<D>::NS, VL = Group<D>::VL;
  int pk0, pk1;
  group_positions<PAGED>(a, sl, s_pg, plist, gi, threadIdx.x & 31, pk0, pk1, g.pv);
  const bf16* k0 = kl + (size_t)max(pk0, 0) * D;
  const bf16* k1 = kl + (size_t)max(pk1, 0) * D;
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    g.kc[0][s] = pk0 >= 0 ? ldg_stream(k0 + 32 * s) : make_uint4(0, 0, 0, 0);
    g.kc[1][s] = pk1 >= 0 ? ldg_stream(k1 + 32 * s) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const bf16* v = vl + (size_t)max(g.pv[t], 0) * D;
#pragma unroll
    for (int u = 0; u < VL; ++u) g.vc[t][u] = g.pv[t] >= 0 ? ldg_stream(v + 8 * u) : make_uint4(0, 0, 0, 0);
  }
}

template <int D>
__device__ __forceinline__ void compute_group(const Group<D>& g, const uint32_t (&qa)[D / 32][4],
                                              float (&o)[D / 16][4], float& m_run, float& l_run, float sl2,
                                              int lane) {
  constexpr int NS = Group<D>::NS, MT = D / 16;
  const int m = lane & 3;
  // S^T tile: rows = heads, columns = tokens (n-tile nt: tokens 8nt..8nt+7);
  // the channel sum runs in two independent chains per n-tile
  float sc[2][2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
    for (int c = 0; c < 2; ++c) sc[nt][c][0] = sc[nt][c][1] = sc[nt][c][2] = sc[nt][c][3] = 0.f;
  }
#pragma unroll
  for (int s = 0; s < NS; ++s) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      mma_bf16(sc[nt][0], qa[s][0], 0u, qa[s][1], 0u, g.kc[nt][s].x, g.kc[nt][s].y);
      mma_bf16(sc[nt][1], qa[s][2], 0u, qa[s][3], 0u, g.kc[nt][s].z, g.kc[nt][s].w);
    }
  }
  // head r, tokens 2m, 2m+1, 2m+8, 2m+9
  float s4[4];
  s4[0] = g.pv[0] >= 0 ? (sc[0][0][0] + sc[0][1][0]) * sl2 : kNegInf;
  s4[1] = g.pv[1] >= 0 ? (sc[0][0][1] + sc[0][1][1]) * sl2 : kNegInf;
  s4[2] = g.pv[2] >= 0 ? (sc[1][0][0] + sc[1][1][0]) * sl2 : kNegInf;
  s4[3] = g.pv[3] >= 0 ? (sc[1][0][1] + sc[1][1][1]) * sl2 : kNegInf;
  float gm = fmaxf(fmaxf(s4[0], s4[1]), fmaxf(s4[2], s4[3]));
  gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 1));
  gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 2));
  const float mn = fmaxf(m_run, gm);
  const bool live = mn != kNegInf;
  const float alpha = live ? ex2(m_run - mn) : 1.f;
  m_run = mn;
  float p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = live ? ex2(s4[i] - mn) : 0.f;
  l_run = fmaf(l_run, alpha, (p[0] + p[1]) + (p[2] + p[3]));
  const uint32_t pb0 = pack_bf16(p[0], p[1]), pb1 = pack_bf16(p[2], p[3]);
  // rescale the accumulators: columns are heads 2m and 2m+1
  const float a_lo = __shfl_sync(0xffffffffu, alpha, 8 * m);
  const float a_hi = __shfl_sync(0xffffffffu, alpha, 8 * m + 4);
  if (!__all_sync(0xffffffffu, a_lo == 1.f && a_hi == 1.f)) {
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      o[t][0] *= a_lo; o[t][1] *= a_hi; o[t][2] *= a_lo; o[t][3] *= a_hi;
    }
  }
  // O^T += V^T P^T: m-tile t covers channels CPR*r + 2t (row r) and +1 (row r+8)
#pragma unroll
  for (int t = 0; t < MT; ++t) {
    const int u = t >> 2, wsel = t & 3;
    const uint32_t w0 = (&g.vc[0][u].x)[wsel], w1 = (&g.vc[1][u].x)[wsel];
    const uint32_t w2 = (&g.vc[2][u].x)[wsel], w3 = (&g.vc[3][u].x)[wsel];
    mma_bf16(o[t], __byte_perm(w0, w1, 0x5410), __byte_perm(w0, w1, 0x7632),
             __byte_perm(w2, w3, 0x5410), __byte_perm(w2, w3, 0x7632), pb0, pb1);
  }
}

template <int D>
constexpr size_t attend_mma_smem() {
  return (size_t)kAttnWarps * 8 * D * sizeof(float);  // the warps' partial outputs
}

struct AttendSmem {
  float sM[kAttnWarps][8];
  float sL[kAttnWarps][8];
  int s_pg[kStagedEntries];
};

// One CTA's work on one row: the run `sl` of the row's list, written to
// partial slot `slot`; `nseg` CTAs write partials of this row.
template <int D, bool PAGED>
__device__ __forceinline__ void attend_run(const AttendArgs& a, int row, const Seg& sl, int slot, int nseg,
                                           float* sO, AttendSmem& sh) {
  constexpr int NW = kAttnWarps;
  constexpr int NS = D / 32;   // 16-byte chunks of a row per lane (chunk 4s + m)
  constexpr int MT = D / 16;   // m-tiles of the P.V product (channels)
  constexpr int CPR = D / 8;   // channels of V owned by one lane row r
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, m = lane & 3;
  const int b = row / a.Hkv, h = row % a.Hkv;
  const int G = a.G;
  const int32_t* plist = a.page_idx ? a.page_idx + (size_t)row * a.idx_stride + sl.e0 : nullptr;
  const bf16* kl = static_cast<const bf16*>(a.k) + (size_t)row * a.Cap * D + m * 8;    // chunk 4s+m: +32s
  const bf16* vl = static_cast<const bf16*>(a.v) + (size_t)row * a.Cap * D + r * CPR;  // lane's V channels

  stage_page_list(sh.s_pg, kStagedEntries, plist, sl.e0, sl.nent, a.Cap >> a.pshift, threadIdx.x, NW * 32);

  // Q as the A operand: row r = head r (rows 8..15 are zero)
  uint32_t qa[NS][4];
  {
    const bf16* qp = static_cast<const bf16*>(a.q) + ((size_t)b * a.Hq + (size_t)h * G + r) * D;
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      uint4 c = r < G ? ldg_stream(qp + (4 * s + m) * 8) : make_uint4(0, 0, 0, 0);
      qa[s][0] = c.x; qa[s][1] = c.y; qa[s][2] = c.z; qa[s][3] = c.w;
    }
  }
  float o[MT][4];
#pragma unroll
  for (int t = 0; t < MT; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
  float m_run = kNegInf, l_run = 0.f;
  const float sl2 = a.qscale;
  __syncthreads();

  const int ngroups = (sl.ntok + 15) >> 4;
  Group<D> ga, gb;
  int gi = warp;
  if (gi < ngroups) load_group<D, PAGED>(ga, a, sl, sh.s_pg, plist, gi, kl, vl);
  while (gi < ngroups) {
    if (gi + NW < ngroups) load_group<D, PAGED>(gb, a, sl, sh.s_pg, plist, gi + NW, kl, vl);
    compute_group<D>(ga, qa, o, m_run, l_run, sl2, lane);
    gi += NW;
    if (gi >= ngroups) break;
    if (gi + NW < ngroups) load_group<D, PAGED>(ga, a, sl, sh.s_pg, plist, gi + NW, kl, vl);
    compute_group<D>(gb, qa, o, m_run, l_run, sl2, lane);
    gi += NW;
  }

  // per-warp state to shared memory
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
  if (m == 0) {
    sh.sM[warp][r] = m_run;
    sh.sL[warp][r] = l_run;
  }
#pragma unroll
  for (int t = 0; t < MT; ++t) {
    const int ch = CPR * r + 2 * t;
    sO[(warp * 8 + 2 * m) * D + ch] = o[t][0];
    sO[(warp * 8 + 2 * m + 1) * D + ch] = o[t][1];
    sO[(warp * 8 + 2 * m) * D + ch + 1] = o[t][2];
    sO[(warp * 8 + 2 * m + 1) * D + ch + 1] = o[t][3];
  }
  __syncthreads();

  for (int i = threadIdx.x; i < G * D; i += NW * 32) {
    const int g = i / D, d = i % D;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, sh.sM[w][g]);
    float av = 0.f, lv = 0.f;
    if (M != kNegInf) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        if (sh.sM[w][g] == kNegInf) continue;
        const float f = exp2f(sh.sM[w][g] - M);
        av += sO[(w * 8 + g) * D + d] * f;
        lv += sh.sL[w][g] * f;
      }
    }
    const size_t hq = (size_t)b * a.Hq + (size_t)h * G + g;
    a.o_part[(hq * a.S + slot) * D + d] = av;
    if (d == 0) {
      a.m_part[hq * a.S + slot] = M == kNegInf ? kNegInf : M * kLn2;
      a.l_part[hq * a.S + slot] = lv;
    }
  }
  if (a.tickets) combine_row_if_last<bf16, D, NW * 32>(a, row, nseg);
  __syncthreads();  // shared memory is reused by the next run of this CTA
}

template <int D, bool PAGED>
__global__ void __launch_bounds__(kAttnWarps * 32, attn_min_blocks<D>())
attend_mma_kernel(const AttendArgs a) {
  pdl_wait_then_release();
  extern __shared__ float sO[];  // [NW][8][D]
  __shared__ AttendSmem sh;
  const int row = blockIdx.x / a.S, split = blockIdx.x % a.S;
  const Slice sl = attend_slice(a, row, split);
  Seg sg;
  sg.N = sl.N;
  sg.e0 = sl.e0;
  sg.joff = 0;
  sg.ntok = sl.nent << a.pshift;
  sg.nent = sl.nent;
  attend_run<D, PAGED>(a, row, sg, split, a.S, sO, sh);
}

template <int D, bool PAGED>
static cudaError_t attend_mma_launch(const AttendArgs& a, int grid, cudaStream_t st) {
  constexpr size_t smem = attend_mma_smem<D>();
  cudaError_t e = cudaFuncSetAttribute(attend_mma_kernel<D, PAGED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(attend_mma_kernel<D, PAGED>, dim3(grid), dim3(kAttnWarps * 32), smem, st, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

const void* attend_mma_kernel_ptr(int D) {
  return D == 64 ? reinterpret_cast<const void*>(attend_mma_kernel<64, false>)
                 : reinterpret_cast<const void*>(attend_mma_kernel<128, true>);
}
size_t attend_mma_kernel_smem(int D) { return D == 64 ? attend_mma_smem<64>() : attend_mma_smem<128>(); }
int attend_mma_kernel_threads() { return kAttnWarps * 32; }

cudaError_t launch_attend_mma(const Shape& s, const AttendArgs& a, cudaStream_t st, bool* handled) {
  *handled = false;
  if (s.dtype != 1 || s.G > 8) return cudaSuccess;
  *handled = true;
  const int grid = s.B * s.Hkv * a.S;
  const bool paged = s.P >= 16;
  if (s.D == 128) return paged ? attend_mma_launch<128, true>(a, grid, st) : attend_mma_launch<128, false>(a, grid, st);
  return paged ? attend_mma_launch<64, true>(a, grid, st) : attend_mma_launch<64, false>(a, grid, st);
}

DeviceStatus take_status_attend_mma() { return take_status_here(); }

}  // namespace sls
