// Refined top-delta attention for bf16 caches ("Faster Than Flash",
// Methodology 3 step 3, eq. 4): split-K online-softmax attention over a
// row's kept blocks in which every token of a complete block is scored with
// its refined key k~ = k^ + r s / 508 (the 2-bit thumbnail level plus the
// 8-bit residual on the thumbnail's block/channel scale s) instead of the
// bf16 key.  Tokens of the newest, partial block have no thumbnail yet and
// use the bf16 key.  Values are bf16.
//
// Top-delta keeps a different number of blocks in every row (a few percent
// in one head, most of the context in another), so a fixed split count per
// row leaves the kernel as slow as its longest row.  Here the rows' lists,
// concatenated, are cut into one range of entries per CTA (one CTA per SM,
// stream-K style: 8 warps, 12 in the refined tensor-map kernel), equal but
// for a CTA whose range crosses a row start, which takes a little less.
// Three kernels share that partition: where the shape allows tensor maps,
// attend_stream_tma_kernel (bf16 keys) and attend_refined_tma_kernel
// (refined keys, D = 128), in which every warp streams its groups through
// its own ring of tensor-map copies; otherwise the register-fed
// attend_balanced_kernel (either kind of key).
//
// In attend_balanced_kernel a warp walks 16-token groups with two groups in
// flight in registers (the shape of the register-fed attend).  Lane (r, m) owns the
// channels [m D/4, (m+1) D/4) of the score product and loads, for tokens r
// and r + 8 of a group, either D/16 bytes of codes and D/4 bytes of
// residuals (a refined group) or D/2 bytes of bf16 key (a group of the
// partial block, or every group without codes).
//
// Refined scores run on the tensor cores in fp16:
//   n = 254 code - 381 + r   is an integer in [-508, 508], exact in fp16,
//   q s                      is exact in fp32 (bf16 x bf16) and splits into
//                            fp16 hi + lo (q s - hi is exact in fp32),
//   S^T = (Q s)_hi N + (Q s)_lo N   accumulated in fp32,
// which is 508 q . k~ to about 2^-22 relative (|q s| < 65504 assumed).  The
// heads' hi parts fill A rows 0-7 and their lo parts rows 8-15 of the same
// MMA (at most 8 heads), so both products cost one MMA per k-step; the
// accumulator rows r and r + 8 are then added.
// Softmax and O^T += V^T P^T follow the register-fed attend.
#include <cuda_fp16.h>

#include <algorithm>

#include "attend_common.cuh"
#include "attend_tma.cuh"
#include "launch.h"
#include "mma.cuh"

namespace sls {

constexpr int kRefWarps = 8;
constexpr int kRefStaged = 1024;  // block-list entries staged in shared memory

struct RefinedArgs {
  AttendArgs a;         // q, k, v, block list (page_idx with P = block), count, ctx_len, combine
  const uint8_t* codes; // [rows, Cap, D/4], or null: every token scored with its bf16 key
  const bf16* scales;   // [rows, Cap/P, D]
  const int8_t* res;    // [rows, Cap, D]
  int rows;
  float* po;            // [slot][G][D] partial accumulators (two slots per CTA)
  float* pm;            // [slot][G] running max (natural-log units)
  float* pl;            // [slot][G] normaliser
};

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The refined scores' MMAs carry the heads' q s hi parts in A rows 0-7 and
// the lo parts in rows 8-15 (at most 8 heads), so one MMA forms both: the
// score of head r is the sum of accumulator rows r and r + 8 (entries 0, 1
// and 2, 3 of a lane), folded here into entries 0, 1 (rows 8-15 are unused
// after this).
__device__ __forceinline__ void refined_fold(float (&sc)[2][2][4]) {
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      sc[nt][c][0] += sc[nt][c][2];
      sc[nt][c][1] += sc[nt][c][3];
    }
}

__device__ __forceinline__ uint2 ldg_stream2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}
__device__ __forceinline__ uint32_t ldg_stream1(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// n = 254 code - 381 + r of the 8 channels of one step as four fp16x2
// (channel pairs 0-1, 2-3, 4-5, 6-7): c16 holds the step's 16 code bits,
// w0 and w1 its 8 residual bytes.  Codes: x = b * 0x4001 places a code byte
// at bit 0 and again at bit 14, so the fields at bits 0-1 and 16-17 of x
// (of x >> 4) are the byte's codes 0 and 1 (2 and 3), and under the
// exponent field 0x6400 each reads as 1024 + code.  Residuals: the signed
// byte plus 128 (xor 0x80) under the same exponent reads as 1152 + r.
// Then 254 (c' - 1024) + (1152 + r) <= 2041 and the final - 1533 are exact.
__device__ __forceinline__ void refined_step(uint32_t c16, uint32_t w0, uint32_t w1, uint32_t (&n)[4]) {
  const __half2 k1024 = __float2half2_rn(1024.f), k254 = __float2half2_rn(254.f), k1533 = __float2half2_rn(1533.f);
  const uint32_t x0 = (c16 & 0xffu) * 0x4001u, x1 = ((c16 >> 8) & 0xffu) * 0x4001u;
  const uint32_t ch[4] = {(x0 & 0x00030003u) | 0x64006400u, ((x0 >> 4) & 0x00030003u) | 0x64006400u,
                          (x1 & 0x00030003u) | 0x64006400u, ((x1 >> 4) & 0x00030003u) | 0x64006400u};
  const uint32_t v0 = w0 ^ 0x80808080u, v1 = w1 ^ 0x80808080u;
  const uint32_t rh[4] = {__byte_perm(v0, 0x64646464u, 0x4140u), __byte_perm(v0, 0x64646464u, 0x4342u),
                          __byte_perm(v1, 0x64646464u, 0x4140u), __byte_perm(v1, 0x64646464u, 0x4342u)};
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const __half2 t = __hfma2(__hsub2(bits_h2(ch[p]), k1024), k254, bits_h2(rh[p]));
    n[p] = h2_bits(__hsub2(t, k1533));
  }
}

template <int D>
struct RGroup {
  static constexpr int NS = D / 32, VL = D / 64;
  uint4 kc[2][NS];  // exact: bf16 key chunks; refined: [0] codes, [1..] residual bytes
  uint4 vc[4][VL];
  int pv[4];
  int pg;           // the group's block, -1 when the group is empty
  bool refined;
};

struct RSeg {
  int N, nent, ntok;
};

template <int D>
__device__ __forceinline__ void load_rgroup(RGroup<D>& g, const RefinedArgs& ra, const RSeg& sl, const int* s_pg,
                                            const int32_t* plist, int gi, int row) {
  constexpr int NS = RGroup<D>::NS, VL = RGroup<D>::VL;
  constexpr int CPR = D / 8;
  const AttendArgs& a = ra.a;
  const int lane = threadIdx.x & 31, r = lane >> 2, m = lane & 3;
  const int j0 = gi << 4;  // 16 tokens inside one block (P >= 16)
  int base = -1, lim = 0, pg = -1;
  if (j0 < sl.ntok) {
    const int e = j0 >> a.pshift;
    pg = e < kRefStaged ? s_pg[e] : __ldg(plist + e);
    if ((unsigned)pg < (unsigned)(a.Cap >> a.pshift)) {
      base = (pg << a.pshift) + (j0 & (a.P - 1));
      lim = min(sl.N - base, 16);
    } else {
      pg = -1;
    }
  }
  g.pg = pg;
  g.refined = ra.codes && pg >= 0 && ((pg + 1) << a.pshift) <= sl.N;  // a complete block has its thumbnail
  auto at = [&](int t) { return (base >= 0 && t < lim) ? base + t : -1; };
  const int pk[2] = {at(r), at(r + 8)};
  g.pv[0] = at(2 * m);
  g.pv[1] = at(2 * m + 1);
  g.pv[2] = at(2 * m + 8);
  g.pv[3] = at(2 * m + 9);
  const size_t rbase = (size_t)row * a.Cap;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const size_t tok = rbase + (size_t)max(pk[t], 0);
    const bool ok = pk[t] >= 0;
    if (g.refined) {
      if constexpr (D == 128) {
        const uint2 c = ok ? ldg_stream2(ra.codes + tok * (D / 4) + m * (D / 16)) : make_uint2(0u, 0u);
        g.kc[t][0] = make_uint4(c.x, c.y, 0u, 0u);
      } else {
        g.kc[t][0] = make_uint4(ok ? ldg_stream1(ra.codes + tok * (D / 4) + m * (D / 16)) : 0u, 0u, 0u, 0u);
      }
      const int8_t* rp = ra.res + tok * D + m * (D / 4);
#pragma unroll
      for (int u = 0; u < D / 64; ++u) g.kc[t][1 + u] = ok ? ldg_stream(rp + 16 * u) : make_uint4(0u, 0u, 0u, 0u);
    } else {
      const bf16* kp = static_cast<const bf16*>(a.k) + tok * D + m * (D / 4);
#pragma unroll
      for (int s = 0; s < NS; ++s) g.kc[t][s] = ok ? ldg_stream(kp + 8 * s) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  const bf16* vl = static_cast<const bf16*>(a.v) + rbase * D + r * CPR;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const bf16* v = vl + (size_t)max(g.pv[t], 0) * D;
#pragma unroll
    for (int u = 0; u < VL; ++u) g.vc[t][u] = g.pv[t] >= 0 ? ldg_stream(v + 8 * u) : make_uint4(0, 0, 0, 0);
  }
}

// wq: the warp's cache of the fp16 hi/lo parts of q s for the block being
// scored ([step][hi, lo][lane], 32 D bytes), or null.  fresh: compute them
// from the block's scales (and fill the cache), else read the cache; a warp
// that scores a block's groups one after the other computes them once.
template <int D>
__device__ __forceinline__ void compute_rgroup(const RGroup<D>& g, const RefinedArgs& ra, int row,
                                               const uint32_t (&qa)[D / 32][4], float (&o)[D / 16][4],
                                               float& m_run, float& l_run, uint4* wq, bool fresh) {
  constexpr int NS = RGroup<D>::NS, MT = D / 16;
  const AttendArgs& a = ra.a;
  const int lane = threadIdx.x & 31, m = lane & 3;
  float sc[2][2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int c = 0; c < 2; ++c) sc[nt][c][0] = sc[nt][c][1] = sc[nt][c][2] = sc[nt][c][3] = 0.f;
  float mul = a.qscale;
  if (g.refined) {
    mul = a.qscale * (1.f / 508.f);
    const bf16* sp = ra.scales + ((size_t)row * (a.Cap >> a.pshift) + g.pg) * D + m * (D / 4);
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      uint32_t hi[4], lo[4];
      if (fresh) {
        const uint4 s8 = __ldg(reinterpret_cast<const uint4*>(sp + 8 * s));
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const uint32_t sw = (&s8.x)[p];
          const float xa = bf16_lo_f(qa[s][p]) * bf16_lo_f(sw);  // exact
          const float xb = bf16_hi_f(qa[s][p]) * bf16_hi_f(sw);
          const __half2 h = __floats2half2_rn(xa, xb);
          hi[p] = h2_bits(h);
          lo[p] = h2_bits(__floats2half2_rn(xa - __low2float(h), xb - __high2float(h)));
        }
        if (wq) {
          wq[(2 * s) * 32 + lane] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          wq[(2 * s + 1) * 32 + lane] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      } else {
        const uint4 h4 = wq[(2 * s) * 32 + lane], l4 = wq[(2 * s + 1) * 32 + lane];
        hi[0] = h4.x; hi[1] = h4.y; hi[2] = h4.z; hi[3] = h4.w;
        lo[0] = l4.x; lo[1] = l4.y; lo[2] = l4.z; lo[3] = l4.w;
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const uint32_t c16 = (&g.kc[nt][0].x)[s >> 1] >> (16 * (s & 1));
        const uint32_t* rw = &g.kc[nt][1].x;
        const uint32_t w0 = rw[2 * s], w1 = rw[2 * s + 1];
        uint32_t n[4];
        refined_step(c16, w0, w1, n);
        // A rows 0-7: the heads' hi parts, rows 8-15: their lo parts
        mma_f16(sc[nt][0], hi[0], lo[0], hi[1], lo[1], n[0], n[1]);
        mma_f16(sc[nt][1], hi[2], lo[2], hi[3], lo[3], n[2], n[3]);
      }
    }
    refined_fold(sc);
  } else {
#pragma unroll
    for (int s = 0; s < NS; ++s) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        mma_bf16(sc[nt][0], qa[s][0], 0u, qa[s][1], 0u, g.kc[nt][s].x, g.kc[nt][s].y);
        mma_bf16(sc[nt][1], qa[s][2], 0u, qa[s][3], 0u, g.kc[nt][s].z, g.kc[nt][s].w);
      }
    }
  }
  // head r, tokens 2m, 2m+1, 2m+8, 2m+9 (base-2 units)
  float s4[4];
  s4[0] = g.pv[0] >= 0 ? (sc[0][0][0] + sc[0][1][0]) * mul : kNegInf;
  s4[1] = g.pv[1] >= 0 ? (sc[0][0][1] + sc[0][1][1]) * mul : kNegInf;
  s4[2] = g.pv[2] >= 0 ? (sc[1][0][0] + sc[1][1][0]) * mul : kNegInf;
  s4[3] = g.pv[3] >= 0 ? (sc[1][0][1] + sc[1][1][1]) * mul : kNegInf;
  float gm = fmaxf(fmaxf(s4[0], s4[1]), fmaxf(s4[2], s4[3]));
  gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 1));
  gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 2));
  const float mn = fmaxf(m_run, gm);
  const bool live = mn != kNegInf;
  const float alpha = live ? exp2f(m_run - mn) : 1.f;
  m_run = mn;
  float p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = live ? exp2f(s4[i] - mn) : 0.f;
  l_run = fmaf(l_run, alpha, (p[0] + p[1]) + (p[2] + p[3]));
  const uint32_t pb0 = pack_bf16(p[0], p[1]), pb1 = pack_bf16(p[2], p[3]);
  const float a_lo = __shfl_sync(0xffffffffu, alpha, 8 * m);
  const float a_hi = __shfl_sync(0xffffffffu, alpha, 8 * m + 4);
#pragma unroll
  for (int t = 0; t < MT; ++t) {
    o[t][0] *= a_lo; o[t][1] *= a_hi; o[t][2] *= a_lo; o[t][3] *= a_hi;
  }
#pragma unroll
  for (int t = 0; t < MT; ++t) {
    const int u = t >> 2, wsel = t & 3;
    const uint32_t w0 = (&g.vc[0][u].x)[wsel], w1 = (&g.vc[1][u].x)[wsel];
    const uint32_t w2 = (&g.vc[2][u].x)[wsel], w3 = (&g.vc[3][u].x)[wsel];
    mma_bf16(o[t], __byte_perm(w0, w1, 0x5410), __byte_perm(w0, w1, 0x7632),
             __byte_perm(w2, w3, 0x5410), __byte_perm(w2, w3, 0x7632), pb0, pb1);
  }
}

constexpr int kRefMaxRows = 4096;  // rows whose list prefix one CTA keeps in shared memory

constexpr int kRefMaxContrib = 1024;  // CTAs sharing one row (one CTA per SM)

constexpr int kRefMaxWarps = 16;  // warps of any kernel that uses RefSmem

struct RefSmem {
  float sM[kRefWarps][8], sL[kRefWarps][8];
  int s_pg[kRefStaged];
  int s_tmp[kRefMaxWarps];
  int s_fail;
  int s_slot[kRefMaxContrib];
  int s_lo[kRefMaxContrib + 1];  // first entry of every CTA's range, and the total
  int s_ncontrib;
  int s_last;
  float s_w[8][64], s_m[8], s_inv[8];
};

// Exclusive scan of one int per thread (NW warps); `total` gets the sum.
template <int NW>
__device__ __forceinline__ int ref_scan(int v, int* tmp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  int before = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const int t = tmp[w];
    before += w < warp ? t : 0;
    total += t;
  }
  __syncthreads();
  return before + x - v;
}

// Work of a CTA's row change in the stream-K kernels (drain, merge, partial
// and refill), in tokens of the list, as measured best on the 256k top-delta
// workload (0 to 1536 swept): 768 for bf16 keys (and the register-fed
// kernel), 1024 for the refined kernel, whose 12 warps merge more state.
constexpr int kSegCostTokens = 768;
constexpr int kSegCostTokensRefined = 1024;

// The CTA whose entry range [s_lo[c], s_lo[c + 1]) holds entry x < T: the
// last c with s_lo[c] <= x (CTAs with empty ranges share their s_lo with the
// next CTA, so the last of them is the one whose range is not empty).
__device__ __forceinline__ int cta_of(const int* s_lo, int x, int grid) {
  int l = 0, u = grid - 1;
  while (l < u) {
    const int mid = (l + u + 1) >> 1;
    if (s_lo[mid] <= x) l = mid;
    else u = mid - 1;
  }
  return l;
}

// Writes the finished output of one head: accumulator sum `av` and
// normaliser `lv` relative to exp(M) (natural log units), the sink joining
// the normaliser.
__device__ __forceinline__ void finish_head(const AttendArgs& a, size_t hq, int h, int g, float M, float lv,
                                            float av, int d, int D) {
  const float sk = a.sink ? a.sink[h * a.G + g] : kNegInf;
  const float Mx = fmaxf(M, sk);
  float f = 0.f, L = 0.f;
  if (Mx != kNegInf) {
    f = M == kNegInf ? 0.f : expf(M - Mx);
    L = lv * f + (a.sink ? expf(sk - Mx) : 0.f);
  }
  // a NaN normaliser (a wait that gave up) stays NaN in the output and lse
  static_cast<bf16*>(a.out)[hq * D + d] = __float2bfloat16(L == 0.f ? 0.f : av * f / L);
  if (d == 0 && a.lse) a.lse[hq] = L == 0.f ? kNegInf : Mx + logf(L);
}

// Stream-K setup: s_pref[row] = the first entry of each row's list in the
// concatenation (s_pref[rows] = T, the total), rows with an empty list
// written (output 0, lse -inf or the sink alone), and this CTA's entry range
// [lo, hi) with the row holding lo.  False when the CTA has no entries.
template <int D, int NT>
__device__ __forceinline__ bool stream_k_begin(const AttendArgs& a, int rows, RefSmem& sh, int* s_pref, int& T,
                                               long long& lo, long long& hi, int& row,
                                               int seg_cost_tokens = kSegCostTokens) {
  const int G = a.G, grid = gridDim.x, c = blockIdx.x;
  const int RPT = (rows + NT - 1) / NT;
  const int r0 = threadIdx.x * RPT;
  int csum = 0;
  for (int i = 0; i < RPT; ++i) {
    const int row = r0 + i;
    if (row < rows) csum += min(max(a.count[row], 0), a.idx_stride);
  }
  int acc = ref_scan<NT / 32>(csum, sh.s_tmp, T);
  for (int i = 0; i < RPT; ++i) {
    const int row = r0 + i;
    if (row < rows) {
      s_pref[row] = acc;
      acc += min(max(a.count[row], 0), a.idx_stride);
    }
  }
  if (threadIdx.x == 0) s_pref[rows] = T;
  __syncthreads();
  // Every CTA's range, once, a CTA per thread (the contributors of a shared
  // row are read from here).  The ranges are equal in a list where every row
  // start after the first counts seg_cost_tokens of extra work: a CTA whose
  // range crosses a row start drains, merges and refills its rings there, so
  // it takes that much less of the real list.  Row r's entries x sit at
  // x + beta r; the entries of CTA k start at the first real entry at or
  // after phantom position Tp k / grid.
  {
    const long long beta = seg_cost_tokens >> a.pshift;
    const long long Tp = (long long)T + beta * (rows - 1);
    for (int k = threadIdx.x; k <= grid; k += NT) {
      const long long Lp = Tp * k / grid;
      int l = 0, u = rows - 1;  // the last row whose phantom start is <= Lp
      while (l < u) {
        const int mid = (l + u + 1) >> 1;
        if (s_pref[mid] + beta * mid <= Lp) l = mid;
        else u = mid - 1;
      }
      sh.s_lo[k] = (int)min(Lp - beta * l, (long long)s_pref[l + 1]);
    }
  }
  __syncthreads();

  // rows with an empty list: output 0, lse -inf (or the sink alone)
  for (int row = c; row < rows; row += grid) {
    if (s_pref[row + 1] != s_pref[row]) continue;
    const int b = row / a.Hkv, h = row % a.Hkv;
    for (int i = threadIdx.x; i < G * D; i += NT)
      finish_head(a, (size_t)b * a.Hq + (size_t)h * G + i / D, h, i / D, kNegInf, 0.f, 0.f, i % D, D);
  }
  if (T == 0) return false;
  lo = sh.s_lo[c];
  hi = sh.s_lo[c + 1];
  if (lo >= hi) return false;
  // the row holding entry lo: the last row whose first entry is <= lo
  {
    int l = 0, u = rows - 1;
    while (l < u) {
      const int mid = (l + u + 1) >> 1;
      if (s_pref[mid] <= lo) l = mid;
      else u = mid - 1;
    }
    row = l;
  }
  return true;
}

// End of one row segment of a stream-K CTA: `partial(g, d, M, av, lv)`
// gives the CTA's merged state of head g, channel d (running max M in
// natural-log units, accumulator av and normaliser lv relative to exp(M)).
// A row the CTA holds entirely is finished in place; otherwise the CTA
// writes its partial to its slot (2c for the segment its range starts in,
// 2c + 1 for the one it ends in) and the row's last contributor to arrive
// merges the slots in CTA order.
template <int D, int NT, typename Partial>
__device__ __forceinline__ void finish_segment(const RefinedArgs& ra, RefSmem& sh, const int* s_pref, int row,
                                               long long e, long long seg_end, long long lo, int c, int T, int grid,
                                               Partial partial) {
  const AttendArgs& a = ra.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int NW = NT / 32;
  const int G = a.G;
  const int b = row / a.Hkv, h = row % a.Hkv;
  const bool whole = e == s_pref[row] && seg_end == s_pref[row + 1];
  const int slot = e == lo ? 2 * c : 2 * c + 1;
  const size_t hq0 = (size_t)b * a.Hq + (size_t)h * G;
  for (int i = threadIdx.x; i < G * D; i += NT) {
    const int g = i / D, d = i % D;
    float Mn, av, lv;
    partial(g, d, Mn, av, lv);
    if (whole) {
      finish_head(a, hq0 + g, h, g, Mn, lv, av, d, D);
    } else {
      const size_t sg = (size_t)slot * G + g;
      ra.po[sg * D + d] = av;
      if (d == 0) {
        ra.pm[sg] = Mn;
        ra.pl[sg] = lv;
      }
    }
  }
  if (!whole) {
    // the row's contributors are the CTAs from the one holding its first
    // entry to the one holding its last; the last to arrive merges
    // (skipping CTAs with empty ranges, which exist when T < grid); CTA k
    // wrote slot 2k when its range starts inside the row, else 2k + 1
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const int cf = cta_of(sh.s_lo, s_pref[row], grid), cl = cta_of(sh.s_lo, s_pref[row + 1] - 1, grid);
      int n = 0;
      for (int k = cf; k <= cl && n < kRefMaxContrib; ++k) {
        const int klo = sh.s_lo[k];
        if (klo < sh.s_lo[k + 1]) sh.s_slot[n++] = klo >= s_pref[row] ? 2 * k : 2 * k + 1;
      }
      sh.s_ncontrib = n;
      sh.s_last = atomicAdd(a.tickets + row, 1) == n - 1;
    }
    __syncthreads();
    const int ncontrib = sh.s_ncontrib;
    if (sh.s_last) {
      __threadfence();
      auto slot_of = [&](int j) -> size_t { return (size_t)sh.s_slot[j]; };
      for (int g = warp; g < G; g += NW) {
        // the first 64 contributors' max and sum in registers, loaded at once
        float pm2[2], pl2[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int j = lane + 32 * u;
          pm2[u] = j < ncontrib ? __ldcg(ra.pm + slot_of(j) * G + g) : kNegInf;
          pl2[u] = j < ncontrib ? __ldcg(ra.pl + slot_of(j) * G + g) : 0.f;
        }
        float M = fmaxf(pm2[0], pm2[1]);
        for (int j = lane + 64; j < ncontrib; j += 32) M = fmaxf(M, __ldcg(ra.pm + slot_of(j) * G + g));
        M = warp_max(M);
        const float sk = a.sink ? a.sink[h * G + g] : kNegInf;
        M = fmaxf(M, sk);
        float Ls = 0.f;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int j = lane + 32 * u;
          const float w = (pm2[u] == kNegInf || M == kNegInf) ? 0.f : expf(pm2[u] - M);
          Ls += pl2[u] * w;
          if (j < ncontrib) sh.s_w[g][j] = w;
        }
        for (int j = lane + 64; j < ncontrib; j += 32) {
          const float ms = __ldcg(ra.pm + slot_of(j) * G + g);
          const float w = (ms == kNegInf || M == kNegInf) ? 0.f : expf(ms - M);
          Ls += __ldcg(ra.pl + slot_of(j) * G + g) * w;
        }
        Ls = warp_sum(Ls);
        if (a.sink && M != kNegInf) Ls += expf(sk - M);
        if (lane == 0) {
          sh.s_m[g] = M;
          sh.s_inv[g] = Ls == 0.f ? 0.f : 1.f / Ls;  // NaN stays NaN
          if (a.lse) a.lse[hq0 + g] = Ls == 0.f ? kNegInf : M + logf(Ls);
        }
      }
      __syncthreads();
      constexpr int C4 = D / 4;
      for (int i = threadIdx.x; i < G * C4; i += NT) {
        const int g = i / C4, cc = i % C4;
        const float M = sh.s_m[g];
        float4 accv = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j0 = 0; j0 < ncontrib; j0 += 8) {
          float4 v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            v[u] = j0 + u < ncontrib
                       ? __ldcg(reinterpret_cast<const float4*>(ra.po + (slot_of(j0 + u) * G + g) * D) + cc)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int j = j0 + u;
            if (j >= ncontrib) break;
            float w;
            if (j < 64) {
              w = sh.s_w[g][j];
            } else {
              const float ms = __ldcg(ra.pm + slot_of(j) * G + g);
              w = (ms == kNegInf || M == kNegInf) ? 0.f : expf(ms - M);
            }
            accv.x = fmaf(v[u].x, w, accv.x);
            accv.y = fmaf(v[u].y, w, accv.y);
            accv.z = fmaf(v[u].z, w, accv.z);
            accv.w = fmaf(v[u].w, w, accv.w);
          }
        }
        const float inv = sh.s_inv[g];
        bf16* op = static_cast<bf16*>(a.out) + (hq0 + g) * D + 4 * cc;
        op[0] = __float2bfloat16(accv.x * inv);
        op[1] = __float2bfloat16(accv.y * inv);
        op[2] = __float2bfloat16(accv.z * inv);
        op[3] = __float2bfloat16(accv.w * inv);
      }
      if (threadIdx.x == 0) a.tickets[row] = 0;  // ready for the next call
    }
  }
}

// Stream-K over the rows' lists (top-delta keeps a different number of
// blocks in every row): the lists, concatenated row after row (T entries),
// are cut into one range of entries per CTA (equal, but for the row-change
// cost that stream_k_begin charges a CTA crossing a row start).  A CTA attends the row
// segments of its range; a row entirely inside the range is finished in
// place, a row shared with neighbouring CTAs gets a partial from each of
// them (slot 2c for the segment a CTA's range starts in, 2c + 1 for the one
// it ends in) and the row's last contributor to arrive merges them in CTA
// order, so the result does not depend on timing.  Rows with an empty list
// are written by CTA row % grid.
template <int D>
__global__ void __launch_bounds__(kRefWarps * 32, 1) attend_balanced_kernel(const RefinedArgs ra) {
  pdl_wait_then_release();
  constexpr int NW = kRefWarps, NT = NW * 32, NS = D / 32, MT = D / 16, CPR = D / 8;
  extern __shared__ float smem_f[];
  float* sO = smem_f;                                         // [NW][8][D]
  int* s_pref = reinterpret_cast<int*>(smem_f + NW * 8 * D);  // [rows + 1] first entry of each row
  __shared__ RefSmem sh;
  const AttendArgs& a = ra.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, m = lane & 3;
  const int G = a.G, rows = ra.rows, grid = gridDim.x, c = blockIdx.x;

  int T, row;
  long long lo, hi;
  if (!stream_k_begin<D, NT>(a, rows, sh, s_pref, T, lo, hi, row)) return;
  long long e = lo;
  while (e < hi) {
    const long long seg_end = min(hi, (long long)s_pref[row + 1]);
    const int b = row / a.Hkv, h = row % a.Hkv;
    const int e0 = (int)(e - s_pref[row]);
    RSeg sl;
    sl.N = clamp_len(a.ctx_len[b], a.Cap);
    sl.nent = (int)(seg_end - e);
    sl.ntok = sl.nent << a.pshift;
    const int32_t* plist = a.page_idx + (size_t)row * a.idx_stride + e0;
    stage_page_list(sh.s_pg, kRefStaged, plist, 0, sl.nent, a.Cap >> a.pshift, threadIdx.x, NT);

    uint32_t qa[NS][4];
    {
      const bf16* qp = static_cast<const bf16*>(a.q) + ((size_t)b * a.Hq + (size_t)h * G + r) * D + m * (D / 4);
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        const uint4 cq = r < G ? ldg_stream(qp + 8 * s) : make_uint4(0, 0, 0, 0);
        qa[s][0] = cq.x; qa[s][1] = cq.y; qa[s][2] = cq.z; qa[s][3] = cq.w;
      }
    }
    float o[MT][4];
#pragma unroll
    for (int t = 0; t < MT; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
    float m_run = kNegInf, l_run = 0.f;
    __syncthreads();

    const int ngroups = (sl.ntok + 15) >> 4;  // whole blocks: P / 16 groups each
    // With codes, a warp takes whole blocks (entries warp, warp + NW, ...)
    // and scores a block's groups one after the other, so the hi/lo parts of
    // q s are computed once per block and cached in the warp's slice of sO
    // (free until the warp's own partial is written there).  Without codes
    // the warps interleave 16-token groups.
    const int gpb = a.P >> 4;
    const bool bmajor = ra.codes != nullptr && gpb > 1;
    uint4* wq = bmajor ? reinterpret_cast<uint4*>(sO + warp * 8 * D) : nullptr;
    auto next_group = [&](int g) {
      return bmajor ? (((g + 1) & (gpb - 1)) ? g + 1 : g + 1 + (NW - 1) * gpb) : g + NW;
    };
    auto fresh = [&](int g) { return !bmajor || (g & (gpb - 1)) == 0; };
    RGroup<D> ga, gb;
    int gi = bmajor ? warp * gpb : warp;
    if (gi < ngroups) load_rgroup<D>(ga, ra, sl, sh.s_pg, plist, gi, row);
    while (gi < ngroups) {
      int gn = next_group(gi);
      if (gn < ngroups) load_rgroup<D>(gb, ra, sl, sh.s_pg, plist, gn, row);
      compute_rgroup<D>(ga, ra, row, qa, o, m_run, l_run, wq, fresh(gi));
      gi = gn;
      if (gi >= ngroups) break;
      gn = next_group(gi);
      if (gn < ngroups) load_rgroup<D>(ga, ra, sl, sh.s_pg, plist, gn, row);
      compute_rgroup<D>(gb, ra, row, qa, o, m_run, l_run, wq, fresh(gi));
      gi = gn;
    }

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
    finish_segment<D, NT>(ra, sh, s_pref, row, e, seg_end, lo, c, T, grid, [&](int g, int d, float& M, float& av,
                                                                                float& lv) {
      float Mb = kNegInf;
#pragma unroll
      for (int w = 0; w < NW; ++w) Mb = fmaxf(Mb, sh.sM[w][g]);
      av = 0.f;
      lv = 0.f;
      if (Mb != kNegInf) {
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          if (sh.sM[w][g] == kNegInf) continue;
          const float f = exp2f(sh.sM[w][g] - Mb);
          av += sO[(w * 8 + g) * D + d] * f;
          lv += sh.sL[w][g] * f;
        }
      }
      M = Mb == kNegInf ? kNegInf : Mb * kLn2;
    });
    __syncthreads();  // shared memory is reused by the next segment
    e = seg_end;
    ++row;
    while (row < rows && s_pref[row + 1] == s_pref[row]) ++row;  // empty rows hold no entries
  }
}

// The same stream-K partition with bf16 keys, fed by the tensor memory
// accelerator (the top-delta step's default attend).  The segment's 16-token
// groups go to the W warps in turn (group gi to warp gi % W), and every warp
// streams its own groups through its own ring of S shared-memory stages: its
// lane 0 copies a group's K and V with the split-K tensor-map attend's boxes
// (stage layout, tensor maps and group arithmetic shared with it) and refills
// a stage with the warp's group S further on once the warp has scored it.
// A late copy then holds up one warp, not the CTA.  The ring positions run
// on across the CTA's row segments; a segment ends with the warps' merge and
// the stream-K epilogue.  A wait that gives up poisons the segment's output
// (NaN) and every later segment of the CTA, and is counted.
template <int D, int W, int S>
struct StreamLayout {
  static constexpr size_t RING = (size_t)W * S * TmaLayout<D>::STAGE;
  static constexpr size_t MERGE = (size_t)W * 8 * D * sizeof(float);  // the warps' accumulators
  static constexpr size_t REGION = RING > MERGE ? RING : MERGE;
};

// First cache position of group gi of the segment and its token count
// inside the context (<= 0: padded entry, bad page or past the context).
// Page ids come from the staged copy s_pg, or from the list in global memory
// when s_pg is null (before the staging barrier) or past the staged entries.
__device__ __forceinline__ int stream_group_base(const AttendArgs& a, int N, const int* s_pg, const int32_t* plist,
                                                 int gi, int& lim) {
  const int j0 = gi << 4;
  const int e = j0 >> a.pshift;
  const int pg = s_pg && e < kRefStaged ? s_pg[e] : __ldg(plist + e);
  lim = 0;
  if ((unsigned)pg >= (unsigned)(a.Cap >> a.pshift)) return 0;
  const int base = (pg << a.pshift) + (j0 & (a.P - 1));
  lim = min(N - base, 16);
  return base;
}

template <int D, int W, int S>
__global__ void __launch_bounds__(W * 32, 1)
attend_stream_tma_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                         const RefinedArgs ra) {
  using L = TmaLayout<D>;
  constexpr int KS = D / 16;
  constexpr int NT = W * 32;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* ring = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  int* s_pref = reinterpret_cast<int*>(ring + StreamLayout<D, W, S>::REGION);  // [rows + 1]
  __shared__ RefSmem sh;
  __shared__ uint64_t full[W][S];
  __shared__ float sM[W][8], sL[W][8], sF[W][8];  // warps' max, sum and merge weight per head
  __shared__ float sHm[8], sHl[8];                 // the CTA's merged max (natural log) and sum
  const AttendArgs& a = ra.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, m = lane & 3;
  const int G = a.G, rows = ra.rows, grid = gridDim.x, c = blockIdx.x;
  if (threadIdx.x == 0) {
    for (int w = 0; w < W; ++w)
      for (int s = 0; s < S; ++s) mbar_init(&full[w][s], 1);
    mbar_fence_init();
    tma_prefetch_map(&tk);
    tma_prefetch_map(&tv);
    sh.s_fail = 0;
  }
  pdl_wait_then_release();
  int T, row;
  long long lo, hi;
  if (!stream_k_begin<D, NT>(a, rows, sh, s_pref, T, lo, hi, row)) return;  // after its barrier: inits visible

  // the wait-timeout test hook: warp 0 of CTA 0 announces bytes for its first
  // stage that it never requests, and its waits poll briefly
  const bool plant = a.test_wait && c == 0 && warp == 0;
  const uint32_t tries = plant ? kTestWaitTries : kWaitTries;
  unsigned char* wring = ring + (size_t)warp * S * L::STAGE;
  const uint32_t wring_u32 = smem_u32(wring);
  uint32_t wseq = 0;  // this warp's ring position (groups it has taken so far)
  long long e = lo;
  while (e < hi) {
    const long long seg_end = min(hi, (long long)s_pref[row + 1]);
    const int b = row / a.Hkv, h = row % a.Hkv;
    const int N = clamp_len(a.ctx_len[b], a.Cap);
    const int nent = (int)(seg_end - e);
    const int32_t* plist = a.page_idx + (size_t)row * a.idx_stride + (int)(e - s_pref[row]);
    // an earlier segment gave up: no more copies (set before that segment's closing barrier)
    const bool failed = sh.s_fail != 0;
    const int ngroups = (nent << a.pshift) >> 4;
    const int nk = ngroups > warp ? (ngroups - warp + W - 1) / W : 0;  // this warp's groups: warp + W k
    const int* pg_src = nullptr;  // page ids from global memory until the list is staged

    // lane 0: the copy of the warp's k-th group of the segment into its stage
    auto issue = [&](int k) {
      const uint32_t q = wseq + k;
      const int st = q % S;
      int lim;
      const int base = stream_group_base(a, N, pg_src, plist, warp + W * k, lim);
      if (plant && q == 0) {
        mbar_arrive_expect_tx(&full[warp][st], 16);  // no copy is issued: this phase never completes
      } else if (lim > 0) {
        mbar_arrive_expect_tx(&full[warp][st], L::STAGE);
        const int y = row * a.Cap + base;
        unsigned char* dst = wring + st * L::STAGE;
        tma_load_3d(dst, &tk, 0, y, 0, &full[warp][st]);
        tma_load_3d(dst + L::GROUP, &tv, 0, y, 0, &full[warp][st]);
      } else {
        mbar_arrive(&full[warp][st]);  // nothing to copy: the phase completes at once
      }
    };
    // S - 1 groups in flight ahead of the one being scored: the stage of
    // group k + S - 1 is the one group k - 1 left, refilled before group k is
    // scored.  The first copies leave before the list is staged (the ring is
    // free since the previous segment's closing barrier).
    if (lane == 0 && !failed) {
      fence_proxy_async_smem();  // the merge's reads of the ring before the copies write it
      for (int k = 0; k < min(S - 1, nk); ++k) issue(k);
    }
    __syncwarp();
    stage_page_list(sh.s_pg, kRefStaged, plist, 0, nent, a.Cap >> a.pshift, threadIdx.x, NT);
    __syncthreads();
    pg_src = sh.s_pg;

    float o[KS][4];
    float m_run = kNegInf, l_run = 0.f;
#pragma unroll
    for (int t = 0; t < KS; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
    // Q as the A operand: a0 = Q[head r][16ks + 2m, +1], a2 = Q[r][16ks + 8 + 2m, +1]
    uint32_t qa[KS][2];
    const bf16* qp = static_cast<const bf16*>(a.q) + ((size_t)b * a.Hq + (size_t)h * G + r) * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qa[ks][0] = r < G ? __ldg(reinterpret_cast<const uint32_t*>(qp + 16 * ks + 2 * m)) : 0u;
      qa[ks][1] = r < G ? __ldg(reinterpret_cast<const uint32_t*>(qp + 16 * ks + 8 + 2 * m)) : 0u;
    }
    bool ok = !failed;
    int k = 0;
    if (ok) {
      for (; k < nk; ++k) {
        if (lane == 0 && k + S - 1 < nk) issue(k + S - 1);  // into the stage group k - 1 has left
        const uint32_t q = wseq + k;
        const int st = q % S;
        if (!mbar_wait(&full[warp][st], (q / S) & 1, tries)) {
          ok = false;
          break;
        }
        int lim;
        stream_group_base(a, N, sh.s_pg, plist, warp + W * k, lim);
        if (lim > 0) tma_group<D>(wring_u32 + st * L::STAGE, lim, qa, o, m_run, l_run, a.qscale, lane);
        // the stage is read before the copy engine may write it again
        __syncwarp();
        if (lane == 0) fence_proxy_async_smem();
      }
    }
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) {
        note_wait_timeout();
        sh.s_fail = 1;
        // the copies still in flight land before the ring is reused or left
        if (!failed)
          for (int k2 = k; k2 < min(nk, k + S - 1); ++k2)
            mbar_wait(&full[warp][(wseq + k2) % S], ((wseq + k2) / S) & 1, tries);
      }
      // an infinite running max makes this warp's merge weight inf - inf =
      // NaN at every later merge: the row's output and lse become NaN
      m_run = __int_as_float(0x7f800000);
    }
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    if (m == 0) {
      sM[warp][r] = m_run;
      sL[warp][r] = l_run;
    }
    wseq += failed ? 0u : (uint32_t)nk;
    __syncthreads();  // every warp's stages have been consumed (or drained): the rings become the merge area

    float* sO = reinterpret_cast<float*>(ring);  // [W][8 heads][D]
    merge_warps<D, W>(o, G, sO, sM, sL, sF, sHm, sHl);
    finish_segment<D, NT>(ra, sh, s_pref, row, e, seg_end, lo, c, T, grid,
                          [&](int g, int d, float& M, float& av, float& lv) {
                            av = 0.f;
#pragma unroll
                            for (int w = 0; w < W; ++w) av = fmaf(sO[(w * 8 + g) * D + d], sF[w][g], av);
                            M = sHm[g];
                            lv = sHl[g];
                          });
    __syncthreads();  // shared memory is reused by the next segment
    e = seg_end;
    ++row;
    while (row < rows && s_pref[row + 1] == s_pref[row]) ++row;  // empty rows hold no entries
  }
}

// The refined attend of attend_balanced_kernel fed by the tensor memory
// accelerator (D = 128): the same stream-K partition, and every warp streams
// its own groups through its own ring of S stages, as in
// attend_stream_tma_kernel.  A warp takes whole blocks (list entries warp,
// warp + W, ...) and their groups one after the other, so the fp16 hi/lo
// parts of q s are formed once per block, from scales loaded while the
// warp's previous block was attended.  A stage holds, for a group of a
// complete block, its 8-bit residuals (16 rows of D bytes, 128-byte swizzle:
// chunk c of token t at chunk c ^ (t % 8)) at offset 0, its codes (16 rows
// of D/4 bytes) at kRefCodesOff and its V at TmaLayout::GROUP; for a group
// of the newest, partial block its bf16 K and V as in the bf16 kernel.
constexpr int kRefCodesOff = 2048;  // after the 16 residual rows of 128 bytes

// Scores of a refined group from its stage: lane (r, m) reads the codes
// (8 bytes) and residuals (32 bytes) of its channel quarter for tokens r and
// r + 8 and forms sc with the B operands decoded by refined_step, as the
// register-fed kernel does from its loads.
__device__ __forceinline__ void refined_scores_smem(uint32_t stage, const uint32_t (&hi)[4][4],
                                                    const uint32_t (&lo)[4][4], float (&sc)[2][2][4], int lane) {
  const int r = lane >> 2, m = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int c = 0; c < 2; ++c) sc[nt][c][0] = sc[nt][c][1] = sc[nt][c][2] = sc[nt][c][3] = 0.f;
  uint32_t cw[2][2], rw[2][8];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const int tok = r + 8 * nt;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                 : "=r"(cw[nt][0]), "=r"(cw[nt][1])
                 : "r"(stage + kRefCodesOff + tok * 32 + m * 8));
#pragma unroll
    for (int u = 0; u < 2; ++u)
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(rw[nt][4 * u]), "=r"(rw[nt][4 * u + 1]), "=r"(rw[nt][4 * u + 2]), "=r"(rw[nt][4 * u + 3])
                   : "r"(stage + tok * 128 + (((2 * m + u) ^ r) << 4)));
  }
#pragma unroll
  for (int s = 0; s < 4; ++s) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      uint32_t n[4];
      refined_step(cw[nt][s >> 1] >> (16 * (s & 1)), rw[nt][2 * s], rw[nt][2 * s + 1], n);
      // A rows 0-7: the heads' hi parts, rows 8-15: their lo parts
      mma_f16(sc[nt][0], hi[s][0], lo[s][0], hi[s][1], lo[s][1], n[0], n[1]);
      mma_f16(sc[nt][1], hi[s][2], lo[s][2], hi[s][3], lo[s][3], n[2], n[3]);
    }
  }
  refined_fold(sc);
}

template <int W, int S>
__global__ void __launch_bounds__(W * 32, 1)
attend_refined_tma_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                          const __grid_constant__ CUtensorMap tcodes, const __grid_constant__ CUtensorMap tres,
                          const RefinedArgs ra) {
  constexpr int D = 128;
  using L = TmaLayout<D>;
  constexpr int KS = D / 16, NS = D / 32;
  constexpr int NT = W * 32;
  constexpr uint32_t kRefinedBytes = 16 * D + 16 * (D / 4) + L::GROUP;  // residuals, codes, V
  extern __shared__ unsigned char smem_raw[];
  unsigned char* ring = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  int* s_pref = reinterpret_cast<int*>(ring + StreamLayout<D, W, S>::REGION);  // [rows + 1]
  __shared__ RefSmem sh;
  __shared__ uint64_t full[W][S];
  __shared__ float sM[W][8], sL[W][8], sF[W][8];
  __shared__ float sHm[8], sHl[8];
  __shared__ __align__(16) bf16 s_q[8 * 128];  // the segment's query heads
  const AttendArgs& a = ra.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, m = lane & 3;
  const int G = a.G, rows = ra.rows, grid = gridDim.x, c = blockIdx.x;
  const int gpb = a.P >> 4;  // groups per block
  if (threadIdx.x == 0) {
    for (int w = 0; w < W; ++w)
      for (int s = 0; s < S; ++s) mbar_init(&full[w][s], 1);
    mbar_fence_init();
    tma_prefetch_map(&tk);
    tma_prefetch_map(&tv);
    tma_prefetch_map(&tcodes);
    tma_prefetch_map(&tres);
    sh.s_fail = 0;
  }
  pdl_wait_then_release();
  int T, row;
  long long lo, hi;
  // after its barrier: inits visible
  if (!stream_k_begin<D, NT>(a, rows, sh, s_pref, T, lo, hi, row, kSegCostTokensRefined)) return;

  const bool plant = a.test_wait && c == 0 && warp == 0;
  const uint32_t tries = plant ? kTestWaitTries : kWaitTries;
  unsigned char* wring = ring + (size_t)warp * S * L::STAGE;
  const uint32_t wring_u32 = smem_u32(wring);
  uint32_t wseq = 0;
  long long e = lo;
  while (e < hi) {
    const long long seg_end = min(hi, (long long)s_pref[row + 1]);
    const int b = row / a.Hkv, h = row % a.Hkv;
    const int N = clamp_len(a.ctx_len[b], a.Cap);
    const int nent = (int)(seg_end - e);
    const int32_t* plist = a.page_idx + (size_t)row * a.idx_stride + (int)(e - s_pref[row]);
    // an earlier segment gave up: no more copies (set before that segment's closing barrier)
    const bool failed = sh.s_fail != 0;
    const int nblk = nent > warp ? (nent - warp + W - 1) / W : 0;  // this warp's blocks: warp + W j
    const int nk = nblk * gpb;
    const int* pg_src = nullptr;  // page ids from global memory until the list is staged
    auto page_of = [&](int eb) { return eb < kRefStaged ? sh.s_pg[eb] : __ldg(plist + eb); };
    // group k of this warp: group k % gpb of its block k / gpb
    auto group_of = [&](int k) { return (warp + W * (k / gpb)) * gpb + (k % gpb); };
    auto refined_at = [&](int base, int lim) { return lim > 0 && (((base >> a.pshift) + 1) << a.pshift) <= N; };

    auto issue = [&](int k) {
      const uint32_t q = wseq + k;
      const int st = q % S;
      int lim;
      const int base = stream_group_base(a, N, pg_src, plist, group_of(k), lim);
      unsigned char* dst = wring + st * L::STAGE;
      const int y = row * a.Cap + base;
      if (plant && q == 0) {
        mbar_arrive_expect_tx(&full[warp][st], 16);  // no copy is issued: this phase never completes
      } else if (refined_at(base, lim)) {
        mbar_arrive_expect_tx(&full[warp][st], kRefinedBytes);
        tma_load_2d(dst, &tres, 0, y, &full[warp][st]);
        tma_load_2d(dst + kRefCodesOff, &tcodes, 0, y, &full[warp][st]);
        tma_load_3d(dst + L::GROUP, &tv, 0, y, 0, &full[warp][st]);
      } else if (lim > 0) {
        mbar_arrive_expect_tx(&full[warp][st], L::STAGE);
        tma_load_3d(dst, &tk, 0, y, 0, &full[warp][st]);
        tma_load_3d(dst + L::GROUP, &tv, 0, y, 0, &full[warp][st]);
      } else {
        mbar_arrive(&full[warp][st]);
      }
    };
    // the first copies leave before the list and q are staged (the ring is
    // free since the previous segment's closing barrier)
    if (lane == 0 && !failed) {
      fence_proxy_async_smem();  // the merge's reads of the ring before the copies write it
      for (int k = 0; k < min(S - 1, nk); ++k) issue(k);
    }
    __syncwarp();
    stage_page_list(sh.s_pg, kRefStaged, plist, 0, nent, a.Cap >> a.pshift, threadIdx.x, NT);
    {
      const uint4* qg = reinterpret_cast<const uint4*>(static_cast<const bf16*>(a.q) +
                                                       ((size_t)b * a.Hq + (size_t)h * G) * D);
      for (int i = threadIdx.x; i < G * D / 8; i += NT) reinterpret_cast<uint4*>(s_q)[i] = __ldg(qg + i);
    }
    __syncthreads();
    pg_src = sh.s_pg;

    float o[KS][4];
    float m_run = kNegInf, l_run = 0.f;
#pragma unroll
    for (int t = 0; t < KS; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
    // Q from shared memory where it is used: per block for the refined
    // weights, per group for the bf16 groups of the newest block
    const bf16* qp = s_q + r * D;
    // the scales of the warp's next block (lane's channel quarter), in flight
    const bf16* srow = ra.scales + (size_t)row * (a.Cap >> a.pshift) * D + m * (D / 4);
    uint4 sv[NS];
    auto load_scales = [&](int eb) {
      const int pg = eb < nent ? page_of(eb) : -1;
      const bool okp = (unsigned)pg < (unsigned)(a.Cap >> a.pshift);
#pragma unroll
      for (int s = 0; s < NS; ++s)
        sv[s] = okp ? __ldg(reinterpret_cast<const uint4*>(srow + (size_t)pg * D + 8 * s)) : make_uint4(0, 0, 0, 0);
    };
    if (nk > 0) load_scales(warp);
    uint32_t whi[NS][4], wlo[NS][4];
    bool ok = !failed;
    int k = 0;
    if (ok) {
      for (; k < nk; ++k) {
        if (lane == 0 && k + S - 1 < nk) issue(k + S - 1);
        if (k % gpb == 0) {
          // a new block: the fp16 hi/lo parts of q s (lane (r, m): head r,
          // channels [m D/4, (m+1) D/4) as pairs), then the next block's scales
#pragma unroll
          for (int s = 0; s < NS; ++s) {
            const uint4 cq =
                r < G ? *reinterpret_cast<const uint4*>(qp + m * (D / 4) + 8 * s) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              const uint32_t sw = (&sv[s].x)[p], qw = (&cq.x)[p];
              const float xa = bf16_lo_f(qw) * bf16_lo_f(sw);  // exact
              const float xb = bf16_hi_f(qw) * bf16_hi_f(sw);
              const __half2 hh = __floats2half2_rn(xa, xb);
              whi[s][p] = h2_bits(hh);
              wlo[s][p] = h2_bits(__floats2half2_rn(xa - __low2float(hh), xb - __high2float(hh)));
            }
          }
          load_scales(warp + W * (k / gpb + 1));
        }
        const uint32_t q = wseq + k;
        const int st = q % S;
        if (!mbar_wait(&full[warp][st], (q / S) & 1, tries)) {
          ok = false;
          break;
        }
        int lim;
        const int base = stream_group_base(a, N, sh.s_pg, plist, group_of(k), lim);
        const uint32_t stage = wring_u32 + st * L::STAGE;
        if (refined_at(base, lim)) {
          float sc[2][2][4];
          refined_scores_smem(stage, whi, wlo, sc, lane);
          tma_softmax_pv<D>(sc, stage + L::GROUP, lim, o, m_run, l_run, a.qscale * (1.f / 508.f), lane);
        } else if (lim > 0) {
          uint32_t qa[KS][2];  // tma_group's fragments: a0 = Q[head r][16ks + 2m, +1], a2 = Q[r][16ks + 8 + 2m, +1]
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            qa[ks][0] = r < G ? *reinterpret_cast<const uint32_t*>(qp + 16 * ks + 2 * m) : 0u;
            qa[ks][1] = r < G ? *reinterpret_cast<const uint32_t*>(qp + 16 * ks + 8 + 2 * m) : 0u;
          }
          tma_group<D>(stage, lim, qa, o, m_run, l_run, a.qscale, lane);
        }
        __syncwarp();
        if (lane == 0) fence_proxy_async_smem();
      }
    }
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) {
        note_wait_timeout();
        sh.s_fail = 1;
        if (!failed)
          for (int k2 = k; k2 < min(nk, k + S - 1); ++k2)
            mbar_wait(&full[warp][(wseq + k2) % S], ((wseq + k2) / S) & 1, tries);
      }
      // an infinite running max makes this warp's merge weight inf - inf =
      // NaN at every later merge: the row's output and lse become NaN
      m_run = __int_as_float(0x7f800000);
    }
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    if (m == 0) {
      sM[warp][r] = m_run;
      sL[warp][r] = l_run;
    }
    wseq += failed ? 0u : (uint32_t)nk;
    __syncthreads();  // every warp's stages have been consumed (or drained): the rings become the merge area

    float* sO = reinterpret_cast<float*>(ring);  // [W][8 heads][D]
    merge_warps<D, W>(o, G, sO, sM, sL, sF, sHm, sHl);
    finish_segment<D, NT>(ra, sh, s_pref, row, e, seg_end, lo, c, T, grid,
                          [&](int g, int d, float& M, float& av, float& lv) {
                            av = 0.f;
#pragma unroll
                            for (int w = 0; w < W; ++w) av = fmaf(sO[(w * 8 + g) * D + d], sF[w][g], av);
                            M = sHm[g];
                            lv = sHl[g];
                          });
    __syncthreads();
    e = seg_end;
    ++row;
    while (row < rows && s_pref[row + 1] == s_pref[row]) ++row;
  }
}

bool refined_supported(const Shape& s) {
  return s.dtype == 1 && s.G <= 8 && s.P >= 16 && (s.D == 64 || s.D == 128) && s.B * s.Hkv <= kRefMaxRows;
}

// one CTA per SM (8 warps, 12 in the refined tensor-map kernel: the register budget)
static int balanced_grid() { return std::min(sm_count(), kRefMaxContrib); }

size_t refined_workspace(const Shape& s) {
  const size_t rows = (size_t)s.B * s.Hkv;
  const size_t slots = 2 * (size_t)balanced_grid();
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  return al(rows * 4) + al(slots * s.G * s.D * 4) + 2 * al(slots * s.G * 4);
}

// One CTA of kStreamWarps warps per SM, each warp with a ring of two
// 16-token groups at D = 128 (four at D = 64): the ring depth beyond that
// bought nothing measurable, and more warps or CTAs per SM were slower.
constexpr int kStreamWarps = 8;
// The refined kernel: its groups take longer to score than to copy, so it
// wants warps rather than stages.  Twelve warps (at most 170 registers a
// thread) with two stages each fill the shared memory; three stages measured
// the same as two, and 10 and 12 warps were 6% and 11% faster than 8.
constexpr int kRefinedWarps = 12;
constexpr int kRefinedStages = 2;

template <int D>
static cudaError_t stream_tma_launch(const Shape& s, const RefinedArgs& ra, cudaStream_t st, bool* handled) {
  constexpr int W = kStreamWarps, S = 256 / D;
  CUtensorMap tk, tv;
  const uint64_t tokens = (uint64_t)s.B * s.Hkv * s.Cap;
  if (!encode_rows_map(&tk, ra.a.k, tokens, D) || !encode_rows_map(&tv, ra.a.v, tokens, D)) return cudaSuccess;
  const size_t smem = StreamLayout<D, W, S>::REGION + (size_t)(ra.rows + 1) * sizeof(int) + 1024;
  if (smem > 227 * 1024) return cudaSuccess;
  *handled = true;
  cudaError_t e = cudaFuncSetAttribute(attend_stream_tma_kernel<D, W, S>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  stat_add(kStatAttendStreamKTma);
  e = launch_pdl(attend_stream_tma_kernel<D, W, S>, dim3(balanced_grid()), dim3(W * 32), smem, st, tk, tv, ra);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// The refined attend on tensor-map fed rings (D = 128; the bf16 kernel's
// grid).
static cudaError_t refined_tma_launch(const Shape& s, const RefinedArgs& ra, cudaStream_t st, bool* handled) {
  constexpr int D = 128, W = kRefinedWarps, S = kRefinedStages;
  CUtensorMap tk, tv, tc, tr;
  const uint64_t tokens = (uint64_t)s.B * s.Hkv * s.Cap;
  if (!encode_rows_map(&tk, ra.a.k, tokens, D) || !encode_rows_map(&tv, ra.a.v, tokens, D) ||
      !encode_bytes_map(&tc, ra.codes, tokens, D / 4) || !encode_bytes_map(&tr, ra.res, tokens, D))
    return cudaSuccess;
  const size_t smem = StreamLayout<D, W, S>::REGION + (size_t)(ra.rows + 1) * sizeof(int) + 1024;
  if (smem > 227 * 1024) return cudaSuccess;
  *handled = true;
  cudaError_t e = cudaFuncSetAttribute(attend_refined_tma_kernel<W, S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  stat_add(kStatAttendRefinedTma);
  e = launch_pdl(attend_refined_tma_kernel<W, S>, dim3(balanced_grid()), dim3(W * 32), smem, st, tk, tv, tc, tr, ra);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D>
static cudaError_t balanced_launch(const RefinedArgs& ra, cudaStream_t st) {
  const size_t smem = (size_t)kRefWarps * 8 * D * sizeof(float) + (size_t)(ra.rows + 1) * sizeof(int);
  cudaError_t e = cudaFuncSetAttribute(attend_balanced_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(attend_balanced_kernel<D>, dim3(balanced_grid()), dim3(kRefWarps * 32), smem, st, ra);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_attend_refined(const Shape& s, const void* q, const void* k, const void* v, const uint8_t* codes,
                                  const void* scales, const int8_t* res, const int32_t* block_idx, int idx_stride,
                                  const int32_t* count, const int32_t* ctx_len, const float* sink, void* out,
                                  float* lse, void* ws, cudaStream_t st) {
  RefinedArgs ra;
  AttendArgs& a = ra.a;
  a = AttendArgs{};
  ra.rows = s.B * s.Hkv;
  const size_t items = 2 * (size_t)balanced_grid();  // partial slots
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  char* w = static_cast<char*>(ws);
  a.tickets = reinterpret_cast<int32_t*>(w);
  w += al((size_t)ra.rows * 4);
  ra.po = reinterpret_cast<float*>(w);
  w += al(items * s.G * s.D * 4);
  ra.pm = reinterpret_cast<float*>(w);
  w += al(items * s.G * 4);
  ra.pl = reinterpret_cast<float*>(w);
  a.sink = sink;
  a.out = out;
  a.lse = lse;
  a.q = q; a.k = k; a.v = v;
  a.page_idx = block_idx; a.count = count; a.ctx_len = ctx_len;
  a.idx_stride = idx_stride; a.k_fixed = idx_stride; a.S = 1;
  a.Hq = s.Hq; a.Hkv = s.Hkv; a.G = s.G; a.Cap = s.Cap; a.P = s.P; a.pshift = s.pshift;
  a.qscale = s.scale * kLog2e;
  ra.codes = codes;
  ra.scales = static_cast<const bf16*>(scales);
  ra.res = res;
  a.test_wait = (s.flags & kFlagTestWaitTimeout) ? 1 : 0;
  // the tensor-map fed kernels where the shape allows them
  const bool aligned = !((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
                          reinterpret_cast<uintptr_t>(codes) | reinterpret_cast<uintptr_t>(res)) & 15);
  if (!codes && attend_tma_eligible(s) && aligned) {
    bool handled = false;
    const cudaError_t e = s.D == 128 ? stream_tma_launch<128>(s, ra, st, &handled)
                                     : stream_tma_launch<64>(s, ra, st, &handled);
    if (handled || e != cudaSuccess) return e;
  }
  if (codes && s.D == 128 && attend_tma_eligible(s) && aligned) {
    bool handled = false;
    const cudaError_t e = refined_tma_launch(s, ra, st, &handled);
    if (handled || e != cudaSuccess) return e;
  }
  return s.D == 128 ? balanced_launch<128>(ra, st) : balanced_launch<64>(ra, st);
}

DeviceStatus take_status_attend_refined() { return take_status_here(); }

}  // namespace sls
