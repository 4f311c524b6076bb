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

template <int D>
__global__ void __launch_bounds__(128)
attend_mma_kernel(const AttendArgs a) {
  constexpr int NW = 4;
  constexpr int NS = D / 32;   // 16-byte chunks of a row per lane (chunk 4s + m)
  constexpr int MT = D / 16;   // m-tiles of the P.V product (channels)
  constexpr int VL = D / 64;   // 16-byte V loads per token per lane
  constexpr int CPR = D / 8;   // channels of V owned by one lane row r
  __shared__ float sO[NW][8][D];
  __shared__ float sM[NW][8];
  __shared__ float sL[NW][8];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, m = lane & 3;
  const int row = blockIdx.x / a.S, split = blockIdx.x % a.S;
  const int b = row / a.Hkv, h = row % a.Hkv;
  const int G = a.G;
  const Slice sl = attend_slice(a, row, split);
  const int ntok = sl.nent << a.pshift;
  const int32_t* plist = a.page_idx ? a.page_idx + (size_t)row * a.idx_stride + sl.e0 : nullptr;
  const bf16* kb = static_cast<const bf16*>(a.k) + (size_t)row * a.Cap * D;
  const bf16* vb = static_cast<const bf16*>(a.v) + (size_t)row * a.Cap * D;

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

  const int ngroups = (ntok + 15) >> 4;
  for (int gi = warp; gi < ngroups; gi += NW) {
    // position of token (lane & 15) of the group
    int mypos = -1;
    {
      const int j = (gi << 4) + (lane & 15);
      if (j < ntok) {
        const int e = j >> a.pshift;
        const int pg = plist ? __ldg(plist + e) : sl.e0 + e;
        mypos = token_position(a, pg, j, sl.N);
      }
    }
    const int pk0 = __shfl_sync(0xffffffffu, mypos, r);
    const int pk1 = __shfl_sync(0xffffffffu, mypos, r + 8);
    int pv[4];
    pv[0] = __shfl_sync(0xffffffffu, mypos, 2 * m);
    pv[1] = __shfl_sync(0xffffffffu, mypos, 2 * m + 1);
    pv[2] = __shfl_sync(0xffffffffu, mypos, 2 * m + 8);
    pv[3] = __shfl_sync(0xffffffffu, mypos, 2 * m + 9);

    uint4 kc[2][NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      kc[0][s] = pk0 >= 0 ? ldg_stream(kb + (size_t)pk0 * D + (4 * s + m) * 8) : make_uint4(0, 0, 0, 0);
      kc[1][s] = pk1 >= 0 ? ldg_stream(kb + (size_t)pk1 * D + (4 * s + m) * 8) : make_uint4(0, 0, 0, 0);
    }
    uint4 vc[4][VL];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
#pragma unroll
      for (int u = 0; u < VL; ++u)
        vc[t][u] = pv[t] >= 0 ? ldg_stream(vb + (size_t)pv[t] * D + r * CPR + u * 8) : make_uint4(0, 0, 0, 0);
    }

    // S^T tile: rows = heads, columns = tokens (n-tile nt: tokens 8nt..8nt+7)
    float sc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        mma_bf16(sc[nt], qa[s][0], 0u, qa[s][1], 0u, kc[nt][s].x, kc[nt][s].y);
        mma_bf16(sc[nt], qa[s][2], 0u, qa[s][3], 0u, kc[nt][s].z, kc[nt][s].w);
      }
    }
    // head r, tokens 2m, 2m+1, 2m+8, 2m+9
    float s4[4];
    s4[0] = pv[0] >= 0 ? sc[0][0] * sl2 : kNegInf;
    s4[1] = pv[1] >= 0 ? sc[0][1] * sl2 : kNegInf;
    s4[2] = pv[2] >= 0 ? sc[1][0] * sl2 : kNegInf;
    s4[3] = pv[3] >= 0 ? sc[1][1] * sl2 : kNegInf;
    float gm = fmaxf(fmaxf(s4[0], s4[1]), fmaxf(s4[2], s4[3]));
    gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 1));
    gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 2));
    const float mn = fmaxf(m_run, gm);
    float alpha = 1.f, p[4] = {0.f, 0.f, 0.f, 0.f};
    if (mn != kNegInf) {
      alpha = exp2f(m_run - mn);
#pragma unroll
      for (int i = 0; i < 4; ++i) p[i] = exp2f(s4[i] - mn);
    }
    m_run = mn;
    const uint32_t pb0 = pack_bf16(p[0], p[1]), pb1 = pack_bf16(p[2], p[3]);
    // the denominator sums exactly the rounded weights the numerator uses
    l_run = l_run * alpha + (bf16_lo_f(pb0) + bf16_hi_f(pb0) + bf16_lo_f(pb1) + bf16_hi_f(pb1));

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
      const uint32_t w0 = (&vc[0][u].x)[wsel], w1 = (&vc[1][u].x)[wsel];
      const uint32_t w2 = (&vc[2][u].x)[wsel], w3 = (&vc[3][u].x)[wsel];
      mma_bf16(o[t], __byte_perm(w0, w1, 0x5410), __byte_perm(w0, w1, 0x7632),
               __byte_perm(w2, w3, 0x5410), __byte_perm(w2, w3, 0x7632), pb0, pb1);
    }
  }

  // per-warp state to shared memory
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
  if (m == 0) {
    sM[warp][r] = m_run;
    sL[warp][r] = l_run;
  }
#pragma unroll
  for (int t = 0; t < MT; ++t) {
    const int ch = CPR * r + 2 * t;
    sO[warp][2 * m][ch] = o[t][0];
    sO[warp][2 * m + 1][ch] = o[t][1];
    sO[warp][2 * m][ch + 1] = o[t][2];
    sO[warp][2 * m + 1][ch + 1] = o[t][3];
  }
  __syncthreads();

  for (int i = threadIdx.x; i < G * D; i += NW * 32) {
    const int g = i / D, d = i % D;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, sM[w][g]);
    float av = 0.f, lv = 0.f;
    if (M != kNegInf) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        if (sM[w][g] == kNegInf) continue;
        const float f = exp2f(sM[w][g] - M);
        av += sO[w][g][d] * f;
        lv += sL[w][g] * f;
      }
    }
    const size_t hq = (size_t)b * a.Hq + (size_t)h * G + g;
    a.o_part[(hq * a.S + split) * D + d] = av;
    if (d == 0) {
      a.m_part[hq * a.S + split] = M == kNegInf ? kNegInf : M * kLn2;
      a.l_part[hq * a.S + split] = lv;
    }
  }
}

cudaError_t launch_attend_mma(const Shape& s, const AttendArgs& a, cudaStream_t st, bool* handled) {
  *handled = false;
  if (s.dtype != 1 || s.G > 8) return cudaSuccess;
  *handled = true;
  const int grid = s.B * s.Hkv * a.S;
  if (s.D == 128)
    attend_mma_kernel<128><<<grid, 128, 0, st>>>(a);
  else
    attend_mma_kernel<64><<<grid, 128, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sls
