// Top-delta block selection over 2-bit key thumbnails ("Faster Than
// Flash", Methodology 2 and 3): a pseudo-max m~ from the exact scores of
// the first and the newest block (eq. 3), a streaming scan of the
// thumbnails that scores every token of every complete block and keeps the
// block when its best margin reaches -delta (eqs. 1-2), then an ordered
// compaction of the kept blocks into a per-row list with a device-side
// count (the list length is data dependent, so the attend kernel derives
// its split boundaries on the device).
#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace sls {

constexpr int kDeltaThreads = 256;
constexpr int kDeltaWarps = kDeltaThreads / 32;
constexpr int kMaxScanTiles = 4;  // 16-token tiles of a block in the tensor-core scan (block <= 64)

struct DeltaArgs {
  const void* q;
  const void* k;
  const uint8_t* codes;
  const void* scales;
  const int32_t* ctx_len;
  uint8_t* flags;
  int32_t* count;
  int32_t* block_idx;
  int idx_stride, block, bshift, nblk_cap, SPL;
  int Hq, Hkv, G, Cap;
  float scale, delta;
};

// Blocks [1, jend) are scanned; 0 and the newest block are forced.
__device__ __forceinline__ void delta_layout(int N, int bshift, int block, int& nfull, int& last,
                                             int& jend) {
  nfull = N >> bshift;
  last = N > 0 ? (N - 1) >> bshift : -1;
  jend = (N & (block - 1)) == 0 ? nfull - 1 : nfull;
}

// The row's pseudo-max m~ ("Faster Than Flash", eq. 3): the best exact
// score of each head over block 0 and the newest block, into s_m (every CTA
// of a row recomputes it: at most two blocks of keys, L2-resident).
template <typename T, int D, int GM>
__device__ __forceinline__ void pseudo_max_cta(const DeltaArgs& a, const T* qrow, const T* krow, int N, int last,
                                               float (*s_mt)[GM], float* s_m) {
  constexpr int EPL = Vec16<T>::N;
  constexpr int L = D / EPL;  // lanes per exact key
  constexpr int TPW = 32 / L;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.G;
  const int grp = lane / L, sub = lane % L;
  float qv[GM][EPL];
#pragma unroll
  for (int g = 0; g < GM; ++g) {
    float t[EPL];
    if (g < G) load_vec(qrow + (size_t)g * D + sub * EPL, t);
#pragma unroll
    for (int e = 0; e < EPL; ++e) qv[g][e] = g < G ? t[e] * a.scale : 0.f;
  }
  const int nb0 = min(a.block, N);
  const int lb0 = max(last << a.bshift, nb0);
  const int ntk = nb0 + (N - lb0);
  float mx[GM];
#pragma unroll
  for (int g = 0; g < GM; ++g) mx[g] = kNegInf;
  // the keys of up to kPmRounds rounds are requested together (the scan waits on this)
  constexpr int kPmRounds = 8;
  const int step = kDeltaWarps * TPW;
  for (int i00 = warp * TPW; i00 < ntk; i00 += kPmRounds * step) {
    uint4 kraw[kPmRounds];
#pragma unroll
    for (int u = 0; u < kPmRounds; ++u) {
      const int i = i00 + u * step + grp;
      const int t = i < nb0 ? i : lb0 + (i - nb0);
      kraw[u] = i < ntk ? ldg_stream(krow + (size_t)t * D + sub * EPL) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kPmRounds; ++u) {
      const int i = i00 + u * step + grp;
      const bool ok = i < ntk;
      float kf[EPL];
      unpack_vec(kraw[u], kf);
      float s[GM];
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        s[g] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) s[g] = fmaf(qv[g][e], kf[e], s[g]);
      }
#pragma unroll
      for (int o = L / 2; o > 0; o >>= 1) {
#pragma unroll
        for (int g = 0; g < GM; ++g) s[g] += __shfl_xor_sync(0xffffffffu, s[g], o);
      }
      if (ok) {
#pragma unroll
        for (int g = 0; g < GM; ++g) mx[g] = fmaxf(mx[g], s[g]);
      }
    }
  }
#pragma unroll
  for (int g = 0; g < GM; ++g) {
    const float w = warp_max(mx[g]);
    if (lane == 0) s_mt[warp][g] = w;
  }
  __syncthreads();
  if (threadIdx.x < GM) {
    float w = kNegInf;
#pragma unroll
    for (int i = 0; i < kDeltaWarps; ++i) w = fmaxf(w, s_mt[i][threadIdx.x]);
    s_m[threadIdx.x] = w;
  }
  __syncthreads();
}

// One CTA per (row, part of the row's blocks).  Every CTA recomputes the
// row's pseudo-max (at most two blocks of exact keys, L2-resident).
template <typename T, int D, int GM>
__global__ void __launch_bounds__(kDeltaThreads)
delta_scan_kernel(const DeltaArgs a) {
  pdl_wait_then_release();
  constexpr int EPL = Vec16<T>::N;
  constexpr int CPL = 16;          // channels per lane in the scan (one 32-bit code word)
  constexpr int LC = D / CPL;      // lanes per thumbnail token
  constexpr int TPS = 32 / LC;     // tokens per warp step in the scan
  __shared__ float s_mt[kDeltaWarps][GM];
  __shared__ float s_m[GM];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x / a.SPL, part = blockIdx.x % a.SPL;
  const int b = row / a.Hkv, h = row % a.Hkv;
  const int G = a.G;
  const int N = clamp_len(a.ctx_len[b], a.Cap);
  int nfull, last, jend;
  delta_layout(N, a.bshift, a.block, nfull, last, jend);
  const int nscan = jend > 1 ? jend - 1 : 0;
  const int per = (nscan + a.SPL - 1) / a.SPL;
  const int j0 = 1 + part * per, j1 = 1 + min(nscan, (part + 1) * per);
  if (j0 >= j1) return;

  const T* qrow = static_cast<const T*>(a.q) + ((size_t)b * a.Hq + (size_t)h * G) * D;
  const T* krow = static_cast<const T*>(a.k) + (size_t)row * a.Cap * D;

  pseudo_max_cta<T, D, GM>(a, qrow, krow, N, last, s_mt, s_m);

  // ---- scan: one warp per block, LC lanes per token, 16 channels per lane
  const int grp = lane / LC, sub = lane % LC;
  float qs[GM][CPL];  // q * scale * 1/2 on this lane's channels
#pragma unroll
  for (int g = 0; g < GM; ++g) {
#pragma unroll
    for (int v = 0; v < CPL / EPL; ++v) {
      float t[EPL];
      if (g < G) load_vec(qrow + (size_t)g * D + sub * CPL + v * EPL, t);
#pragma unroll
      for (int e = 0; e < EPL; ++e) qs[g][v * EPL + e] = g < G ? t[e] * a.scale * 0.5f : 0.f;
    }
  }
  float mt[GM];
#pragma unroll
  for (int g = 0; g < GM; ++g) mt[g] = g < G ? s_m[g] : 0.f;
  const T* srow = static_cast<const T*>(a.scales) + (size_t)row * a.nblk_cap * D + sub * CPL;
  const uint32_t* crow = reinterpret_cast<const uint32_t*>(a.codes + (size_t)row * a.Cap * (D / 4)) + sub;
  constexpr int WPT = D / 16;  // 32-bit code words per token
  for (int j = j0 + warp; j < j1; j += kDeltaWarps) {
    // weights w = q * scale * s / 2 and their sum (level = (code - 1.5) * s / 2)
    float w[GM][CPL], wsum[GM];
    {
      float sv[CPL];
#pragma unroll
      for (int v = 0; v < CPL / EPL; ++v) {
        float t[EPL];
        load_vec(srow + (size_t)j * D + v * EPL, t);
#pragma unroll
        for (int e = 0; e < EPL; ++e) sv[v * EPL + e] = t[e];
      }
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        wsum[g] = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          w[g][c] = qs[g][c] * sv[c];
          wsum[g] += w[g][c];
        }
      }
    }
    float best = kNegInf;
    const uint32_t* cb = crow + (size_t)j * a.block * WPT;
    for (int t0 = 0; t0 < a.block; t0 += TPS * 8) {
      uint32_t cw[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int t = t0 + u * TPS + grp;
        cw[u] = t < a.block ? __ldg(cb + (size_t)t * WPT) : 0u;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        float s[GM];
#pragma unroll
        for (int g = 0; g < GM; ++g) s[g] = -1.5f * wsum[g];
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          const float code = (float)((cw[u] >> (2 * c)) & 3u);
#pragma unroll
          for (int g = 0; g < GM; ++g) s[g] = fmaf(w[g][c], code, s[g]);
        }
#pragma unroll
        for (int o = LC / 2; o > 0; o >>= 1) {
#pragma unroll
          for (int g = 0; g < GM; ++g) s[g] += __shfl_xor_sync(0xffffffffu, s[g], o);
        }
        const bool ok = t0 + u * TPS + grp < a.block;
#pragma unroll
        for (int g = 0; g < GM; ++g)
          if (g < G && ok) best = fmaxf(best, s[g] - mt[g]);
      }
    }
    best = warp_max(best);
    if (lane == 0) a.flags[(size_t)row * a.nblk_cap + j] = best >= -a.delta ? 1 : 0;
  }
}

// The same scan on the tensor cores (bf16 keys, any G <= 8).  Per complete
// block the tentative scores of all its tokens and heads are one product
//   S[t][g] = sum_c code[t][c] * w[g][c]  -  1.5 * sum_c w[g][c],
//   w[g][c] = scale * q[g][c] * s[c] / 2   (the level is (code - 1.5) s / 2),
// with A = the codes (16 tokens x 16 channels per m16n8k16, exact in fp16)
// and B = w split into fp16 hi + lo parts (w - hi is exact in fp32),
// accumulated in fp32: the same scores as the CUDA-core scan to about 2^-22
// relative.  Lane (r, m) owns channels [m D/4, (m+1) D/4), tokens r and
// r + 8 of each 16-token tile and column r of B.
//
// Codes go to the tensor cores as fp16 subnormals, decoded by one AND each:
// a 32-bit code word holds the 16 codes of 16 consecutive channels (channel
// i at bits 2i), and the mask 3 << 2j applied to both 16-bit halves keeps
// the codes of channels j and 8 + j (j < 4) in place, where the half reads
// as 4^j code 2^-24 (all below 2^-14: subnormal, exact); the word shifted
// right by 8 gives channels 4 + j and 12 + j the same way.  Register i
// (0..7) of a word thus pairs channels (i, i + 8) with the factor 4^(i & 3);
// k-step ks of the lane uses registers 2u and 2u + 1 (u = ks & 3) of word
// ks >> 2 for the k-slots {2m, 2m + 1} and {8 + 2m, 9 + 2m}.  Any channel
// order works as long as A and B agree on it: every lane pairs its k-slots
// with channels by the same rule.  The weights carry 64 / 4^(c & 3), so
// every product is 64 2^-24 times the level's.
template <int I>
__device__ __forceinline__ uint32_t code_pair_sub(uint32_t w, uint32_t w8) {
  return (I < 4 ? w : w8) & (0x00030003u << (2 * (I & 3)));
}
// The same with the pair index I given at run time (unrolled loops fold it).
__device__ __forceinline__ uint32_t code_pair_sub_rt(uint32_t w, uint32_t w8, int I) {
  return (I < 4 ? w : w8) & (0x00030003u << (2 * (I & 3)));
}

__device__ __forceinline__ void mma_f16_d(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The codes of NTILE 16-token tiles of one block: lane (r, m) holds words
// [m W, (m + 1) W) of tokens r and r + 8 of each tile.
template <int D, int NTILE>
struct ScanTiles {
  static constexpr int W = D / 64;  // 32-bit code words per token and lane (D/4 channels)
  uint32_t c[NTILE][2][W];          // [m-tile][token r, r + 8][word]
};

template <int D, int NTILE>
__device__ __forceinline__ void load_scan_tiles(ScanTiles<D, NTILE>& sc, const uint8_t* cblk, int lane) {
  constexpr int W = ScanTiles<D, NTILE>::W;
  const int r = lane >> 2, m = lane & 3;
#pragma unroll
  for (int mt = 0; mt < NTILE; ++mt) {
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const uint8_t* p = cblk + (size_t)(16 * mt + 8 * t + r) * (D / 4) + m * (D / 16);
      if constexpr (W == 2) {
        const uint2 v = *reinterpret_cast<const uint2*>(p);
        sc.c[mt][t][0] = v.x;
        sc.c[mt][t][1] = v.y;
      } else {
        sc.c[mt][t][0] = *reinterpret_cast<const uint32_t*>(p);
      }
    }
  }
}

// The block's scales (bf16) of the lane's D/4 channels; zero for a block
// past the part's end.
template <int D>
__device__ __forceinline__ void load_scan_scales(uint4 (&sv)[D / 32], const bf16* sblk, bool valid, int lane) {
  const int m = lane & 3;
#pragma unroll
  for (int v = 0; v < D / 32; ++v)
    sv[v] = valid ? __ldg(reinterpret_cast<const uint4*>(sblk + m * (D / 4) + 8 * v)) : make_uint4(0u, 0u, 0u, 0u);
}

// Best margin over the block's tokens for this lane's output columns 2m,
// 2m + 1 (scale * q.k^ - m~ = level sums + off), with the codes entering the
// MMA as fp16 subnormals and the weights as fp16 hi parts (and lo parts with
// LO).  The k-steps run outermost, so the NTILE accumulator chains are
// independent and their MMAs overlap.
template <int D, int NTILE, bool LO>
__device__ __forceinline__ float scan_tiles(const ScanTiles<D, NTILE>& cur, const uint32_t (&whi)[D / 16][2],
                                            const uint32_t (&wlo)[D / 16][2], bool hv0, bool hv1, float off0,
                                            float off1) {
  constexpr int CPL = D / 4;
  float acc[NTILE][4];
#pragma unroll
  for (int mt = 0; mt < NTILE; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
#pragma unroll
  for (int wd = 0; wd < CPL / 16; ++wd) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // channel pairs (2k, 2k + 1) of the word's two 8-channel halves
#pragma unroll
      for (int mt = 0; mt < NTILE; ++mt) {
        const uint32_t x = cur.c[mt][0][wd], y = cur.c[mt][1][wd];  // tokens r and r + 8
        const uint32_t x8 = x >> 8, y8 = y >> 8;
        const uint32_t a0 = code_pair_sub_rt(x, x8, 2 * k), a1 = code_pair_sub_rt(y, y8, 2 * k);
        const uint32_t a2 = code_pair_sub_rt(x, x8, 2 * k + 1), a3 = code_pair_sub_rt(y, y8, 2 * k + 1);
        mma_f16_d(acc[mt], a0, a1, a2, a3, whi[4 * wd + k][0], whi[4 * wd + k][1]);
        if constexpr (LO) mma_f16_d(acc[mt], a0, a1, a2, a3, wlo[4 * wd + k][0], wlo[4 * wd + k][1]);
      }
    }
  }
  // acc (64 2^-24 times the level sums): tokens r (0, 1) and r + 8 (2, 3), columns 2m (0, 2) and 2m + 1 (1, 3)
  constexpr float kUnscale = 262144.f;  // 2^24 / 64
  float best = kNegInf;
#pragma unroll
  for (int mt = 0; mt < NTILE; ++mt) {
    if (hv0) best = fmaxf(best, fmaxf(acc[mt][0], acc[mt][2]) * kUnscale + off0);
    if (hv1) best = fmaxf(best, fmaxf(acc[mt][1], acc[mt][3]) * kUnscale + off1);
  }
  return best;
}

// The lane's weights for B column r: hi parts per k-step (word wd holds
// channels 16 wd + i and 16 wd + i + 8 in register i), the column's fp32
// level-sum weight total and the total of their magnitudes (over the lane's
// channels), or the lo parts w - hi.
template <int D, bool LO>
__device__ __forceinline__ void scan_weights(const float* qh, const uint4 (&sv)[D / 32], uint32_t (&wout)[D / 16][2],
                                             float& wsum, float& wabs) {
  constexpr int CPL = D / 4;
  wsum = 0.f;
  wabs = 0.f;
#pragma unroll
  for (int wd = 0; wd < CPL / 16; ++wd) {
    float sa[8], sb[8];
    unpack_vec(sv[2 * wd], sa);
    unpack_vec(sv[2 * wd + 1], sb);
    const float4 qa0 = *reinterpret_cast<const float4*>(qh + 16 * wd);
    const float4 qa1 = *reinterpret_cast<const float4*>(qh + 16 * wd + 4);
    const float4 qb0 = *reinterpret_cast<const float4*>(qh + 16 * wd + 8);
    const float4 qb1 = *reinterpret_cast<const float4*>(qh + 16 * wd + 12);
    const float qa[8] = {qa0.x, qa0.y, qa0.z, qa0.w, qa1.x, qa1.y, qa1.z, qa1.w};
    const float qb[8] = {qb0.x, qb0.y, qb0.z, qb0.w, qb1.x, qb1.y, qb1.z, qb1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float w0 = qa[i] * sa[i], w1 = qb[i] * sb[i];
      const __half2 hi = __floats2half2_rn(w0, w1);
      if constexpr (LO) {
        const __half2 lo = __floats2half2_rn(w0 - __low2float(hi), w1 - __high2float(hi));
        wout[4 * wd + (i >> 1)][i & 1] = *reinterpret_cast<const uint32_t*>(&lo);
      } else {
        wout[4 * wd + (i >> 1)][i & 1] = *reinterpret_cast<const uint32_t*>(&hi);
        // the level sum takes the unscaled weights (exact: powers of two)
        const float u = 1.f / (64 >> (2 * (i & 3)));
        wsum = fmaf(w0 + w1, u, wsum);
        wabs = fmaf(fabsf(w0) + fabsf(w1), u, wabs);
      }
    }
  }
}

// A block scored again with hi + lo weights (exact to fp32 rounding): its
// codes and the pair's scales read again, outside the main loop's registers
// (rare: only blocks whose hi-only margin lies near -delta come here).
template <int D, int NTILE>
__device__ __noinline__ float rescan_block(const uint8_t* cblk, const bf16* sblk, bool svalid, const float* qh,
                                          bool hv0, bool hv1, float off0, float off1) {
  const int lane = threadIdx.x & 31;
  ScanTiles<D, NTILE> c;
  load_scan_tiles<D, NTILE>(c, cblk, lane);
  uint4 sv[D / 32];
  load_scan_scales<D>(sv, sblk, svalid, lane);
  uint32_t whi[D / 16][2], wlo[D / 16][2];
  float ds, da;
  scan_weights<D, false>(qh, sv, whi, ds, da);
  scan_weights<D, true>(qh, sv, wlo, ds, da);
  return warp_max(scan_tiles<D, NTILE, true>(c, whi, wlo, hv0, hv1, off0, off1));
}

// One CTA per (row, part of the row's blocks); a warp scores NB blocks at a
// time (NB = 2 when G <= 4: B columns 0..3 carry the heads' weights for the
// first block and columns 4..7 those for the second, so every lane computes
// weights that are used, once per two blocks).  The codes of the warp's next
// block, and the scales of its next pair, are in flight while it scores.
template <int D, int NTILE, int NB>
__global__ void __launch_bounds__(kDeltaThreads, 2)
delta_scan_mma_kernel(const DeltaArgs a) {
  pdl_wait_then_release();
  constexpr int KS = D / 16;  // k-steps
  constexpr int CPL = D / 4;  // channels per lane
  __shared__ float s_mt[kDeltaWarps][8];
  __shared__ float s_m[8];
  __shared__ __align__(16) float s_qh[32][CPL + 4];  // per lane: its column's q, padded against bank conflicts
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, m = lane & 3;
  const int row = blockIdx.x / a.SPL, part = blockIdx.x % a.SPL;
  const int b = row / a.Hkv, h = row % a.Hkv;
  const int G = a.G;
  const int N = clamp_len(a.ctx_len[b], a.Cap);
  int nfull, last, jend;
  delta_layout(N, a.bshift, a.block, nfull, last, jend);
  const int nscan = jend > 1 ? jend - 1 : 0;
  const int per = (nscan + a.SPL - 1) / a.SPL;
  const int j0 = 1 + part * per, j1 = 1 + min(nscan, (part + 1) * per);
  if (j0 >= j1) return;
  const bf16* qrow = static_cast<const bf16*>(a.q) + ((size_t)b * a.Hq + (size_t)h * G) * D;
  const bf16* krow = static_cast<const bf16*>(a.k) + (size_t)row * a.Cap * D;

  // column r of B is head r (NB = 1) or head r & 3 of block r >> 2 (NB = 2);
  // lane l = 4 r + m holds q * scale / 2 of that head on channels
  // [m D/4, (m+1) D/4), times 64 / f for the code scaling f = 1, 4, 16, 64
  // of the channel's place in its code byte
  for (int i = threadIdx.x; i < 32 * CPL; i += kDeltaThreads) {
    const int l = i / CPL, e = i % CPL;
    const int g = NB == 2 ? ((l >> 2) & 3) : (l >> 2);
    s_qh[l][e] = g < G ? __bfloat162float(qrow[(size_t)g * D + (l & 3) * CPL + e]) * a.scale *
                             (0.5f * (64 >> (2 * (e & 3))))
                       : 0.f;
  }
  pseudo_max_cta<bf16, D, 8>(a, qrow, krow, N, last, s_mt, s_m);  // ends with a CTA barrier
  const float* qh = s_qh[lane];
  // output columns 2m, 2m + 1: their heads, and the block of the pair they score
  const int h0 = NB == 2 ? (2 * m) & 3 : 2 * m, h1 = h0 + 1;
  const int out_half = NB == 2 ? m >> 1 : 0;
  const int w_half = NB == 2 ? r >> 2 : 0;  // the block of the pair whose weights this lane computes
  const bool hv0 = h0 < G, hv1 = h1 < G;
  const float mt0 = hv0 ? s_m[h0] : 0.f, mt1 = hv1 ? s_m[h1] : 0.f;
  const bf16* srow = static_cast<const bf16*>(a.scales) + (size_t)row * a.nblk_cap * D;
  const uint8_t* crow = a.codes + (size_t)row * a.Cap * (D / 4);
  constexpr int kStride = kDeltaWarps * NB;

  ScanTiles<D, NTILE> cur, nxt;
  uint4 sv[D / 32];
  int jg = j0 + warp * NB;
  if (jg < j1) {
    load_scan_tiles<D, NTILE>(cur, crow + (size_t)jg * a.block * (D / 4), lane);
    load_scan_scales<D>(sv, srow + (size_t)(jg + w_half) * D, jg + w_half < j1, lane);
  }
  while (jg < j1) {
    const int jn = jg + kStride;
    // the pair's weights: fp16 hi parts, and the fp32 sums that give each
    // column's offset and bound what the lo parts w - hi add
    uint32_t whi[KS][2];
    float wsum, wabs;
    scan_weights<D, false>(qh, sv, whi, wsum, wabs);
    wsum += __shfl_xor_sync(0xffffffffu, wsum, 1);
    wsum += __shfl_xor_sync(0xffffffffu, wsum, 2);  // column r's sum over all channels
    const float ws0 = __shfl_sync(0xffffffffu, wsum, 8 * m), ws1 = __shfl_sync(0xffffffffu, wsum, 8 * m + 4);
    const float off0 = -1.5f * ws0 - mt0, off1 = -1.5f * ws1 - mt1;
    // A token's score differs from the hi-only one by sum_c code_c (w_c - hi_c)
    // <= 3 sum_c |w_c - hi_c|, with |w - hi| <= 2^-11 |w| for a normal fp16 hi
    // and at most the subnormal step 2^-25 below that (in the scaled units of
    // the weights, so 2^-25 u in the level sums); fp32 accumulation adds far
    // less than the 2x slack taken here.  Only a block whose hi-only margin
    // lies that close to -delta can decide the other way: it is scored again
    // with hi + lo (exact to fp32 rounding).  The bound is the largest over
    // every column of the pair.
    wabs += __shfl_xor_sync(0xffffffffu, wabs, 1);
    wabs += __shfl_xor_sync(0xffffffffu, wabs, 2);
    const float err = warp_max(6.f * (wabs * 0x1p-11f + (float)D * 0x1p-25f));
#pragma unroll
    for (int hb = 0; hb < NB; ++hb) {
      const int j = jg + hb;
      if (j >= j1) break;  // warp-uniform
      const int jnext = hb + 1 < NB ? j + 1 : jn;
      if (jnext < j1) load_scan_tiles<D, NTILE>(nxt, crow + (size_t)jnext * a.block * (D / 4), lane);
      if (hb == 0 && jn < j1)  // this pair's scales are spent: the next pair's
        load_scan_scales<D>(sv, srow + (size_t)(jn + w_half) * D, jn + w_half < j1, lane);
      const bool mine = out_half == hb;
      float best = warp_max(scan_tiles<D, NTILE, false>(cur, whi, whi, hv0 && mine, hv1 && mine, off0, off1));
      if (fabsf(best + a.delta) <= err)  // warp-uniform
        best = rescan_block<D, NTILE>(crow + (size_t)j * a.block * (D / 4), srow + (size_t)(jg + w_half) * D,
                                      jg + w_half < j1, qh, hv0 && mine, hv1 && mine, off0, off1);
      if (lane == 0) a.flags[(size_t)row * a.nblk_cap + j] = best >= -a.delta ? 1 : 0;
      cur = nxt;
    }
    jg = jn;
  }
}

// One CTA per row: ordered list of the kept blocks and its length.
__global__ void __launch_bounds__(1024)
delta_compact_kernel(const DeltaArgs a) {
  pdl_wait_then_release();
  __shared__ int tmp[32];
  const int row = blockIdx.x;
  const int b = row / a.Hkv;
  const int N = clamp_len(a.ctx_len[b], a.Cap);
  int nfull, last, jend;
  delta_layout(N, a.bshift, a.block, nfull, last, jend);
  const int nb = last + 1;  // blocks holding valid positions
  const int per = (nb + 1023) / 1024;
  const int i0 = min((int)threadIdx.x * per, nb), i1 = min(i0 + per, nb);
  const uint8_t* f = a.flags + (size_t)row * a.nblk_cap;
  auto keep = [&](int j) { return j == 0 || j == last || (j < jend && f[j] != 0); };
  int n = 0;
  for (int j = i0; j < i1; ++j) n += keep(j);
  // exclusive scan over 1024 threads
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = tmp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    tmp[lane] = t;
  }
  __syncthreads();
  int pos = (warp > 0 ? tmp[warp - 1] : 0) + x - n;
  int32_t* out = a.block_idx + (size_t)row * a.idx_stride;
  for (int j = i0; j < i1; ++j)
    if (keep(j)) out[pos++] = j;
  if (threadIdx.x == 0) a.count[row] = tmp[31];
}

size_t select_delta_workspace(const Shape& s, int block) {
  const size_t bytes = (size_t)s.B * s.Hkv * (size_t)(s.Cap / block);
  return (bytes + 255) & ~(size_t)255;
}

template <typename T, int D, int GM>
static cudaError_t delta_launch(const DeltaArgs& a, int rows, cudaStream_t st) {
  cudaError_t e = launch_pdl(delta_scan_kernel<T, D, GM>, dim3(rows * a.SPL), dim3(kDeltaThreads), 0, st, a);
  if (e != cudaSuccess) return e;
  e = launch_pdl(delta_compact_kernel, dim3(rows), dim3(1024), 0, st, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D, int NTILE, int NB>
static cudaError_t delta_scan_launch(const DeltaArgs& a, int rows, cudaStream_t st) {
  return launch_pdl(delta_scan_mma_kernel<D, NTILE, NB>, dim3(rows * a.SPL), dim3(kDeltaThreads), 0, st, a);
}

template <int D, int NTILE>
static cudaError_t delta_mma_launch_t(const DeltaArgs& a, int rows, cudaStream_t st) {
  cudaError_t e = a.G <= 4 ? delta_scan_launch<D, NTILE, 2>(a, rows, st) : delta_scan_launch<D, NTILE, 1>(a, rows, st);
  if (e != cudaSuccess) return e;
  e = launch_pdl(delta_compact_kernel, dim3(rows), dim3(1024), 0, st, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t delta_g(const DeltaArgs& a, int rows, cudaStream_t st) {
  if (a.G <= 1) return delta_launch<T, D, 1>(a, rows, st);
  if (a.G <= 2) return delta_launch<T, D, 2>(a, rows, st);
  if (a.G <= 4) return delta_launch<T, D, 4>(a, rows, st);
  return delta_launch<T, D, 8>(a, rows, st);
}

cudaError_t launch_select_delta(const Shape& s, const void* q, const void* k,
                                const uint8_t* codes, const void* scales,
                                const int32_t* ctx_len, int block, float delta,
                                int32_t* count, int32_t* block_idx, int idx_stride,
                                void* ws, cudaStream_t st) {
  DeltaArgs a;
  a.q = q; a.k = k; a.codes = codes; a.scales = scales; a.ctx_len = ctx_len;
  a.flags = static_cast<uint8_t*>(ws); a.count = count; a.block_idx = block_idx;
  a.idx_stride = idx_stride; a.block = block;
  a.bshift = __builtin_ctz((unsigned)block);
  a.nblk_cap = s.Cap / block;
  a.Hq = s.Hq; a.Hkv = s.Hkv; a.G = s.G; a.Cap = s.Cap;
  a.scale = s.scale; a.delta = delta;
  const int rows = s.B * s.Hkv;
  // parts per row: enough CTAs to cover the SMs a few times over
  int spl = (4 * sm_count() + rows - 1) / rows;
  const int maxblk = a.nblk_cap;
  spl = spl < 1 ? 1 : spl;
  spl = spl > maxblk ? maxblk : spl;
  a.SPL = spl;
  if (s.dtype == 0) {
    stat_add(kStatDeltaCudaCores);
    return s.D == 64 ? delta_g<float, 64>(a, rows, st) : delta_g<float, 128>(a, rows, st);
  }
  if (!(s.flags & 1) && s.G <= 8 && block >= 16 && block <= 16 * kMaxScanTiles) {  // tensor cores unless asked for CUDA cores
    // one wave of two CTAs per SM (each recomputes the row's pseudo-max once)
    a.SPL = std::max(1, std::min(maxblk, (2 * sm_count()) / rows));
    stat_add(kStatDeltaTensorCores);
    const int nt = block >> 4;
    if (s.D == 64) return nt == 1 ? delta_mma_launch_t<64, 1>(a, rows, st) : nt == 2 ? delta_mma_launch_t<64, 2>(a, rows, st) : delta_mma_launch_t<64, 4>(a, rows, st);
    return nt == 1 ? delta_mma_launch_t<128, 1>(a, rows, st) : nt == 2 ? delta_mma_launch_t<128, 2>(a, rows, st) : delta_mma_launch_t<128, 4>(a, rows, st);
  }
  stat_add(kStatDeltaCudaCores);
  return s.D == 64 ? delta_g<bf16, 64>(a, rows, st) : delta_g<bf16, 128>(a, rows, st);
}

}  // namespace sls
