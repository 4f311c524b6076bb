// Top-delta block selection over 2-bit key thumbnails ("Faster Than
// Flash", Methodology 2 and 3): a pseudo-max m~ from the exact scores of
// the first and the newest block (eq. 3), a streaming scan of the
// thumbnails that scores every token of every complete block and keeps the
// block when its best margin reaches -delta (eqs. 1-2), then an ordered
// compaction of the kept blocks into a per-row list with a device-side
// count (the list length is data dependent, so the attend kernel derives
// its split boundaries on the device).
#include "common.cuh"
#include "launch.h"

namespace sls {

constexpr int kDeltaThreads = 256;
constexpr int kDeltaWarps = kDeltaThreads / 32;

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

// One CTA per (row, part of the row's blocks).  Every CTA recomputes the
// row's pseudo-max (at most two blocks of exact keys, L2-resident).
template <typename T, int D, int GM>
__global__ void __launch_bounds__(kDeltaThreads)
delta_scan_kernel(const DeltaArgs a) {
  pdl_wait_then_release();
  constexpr int EPL = Vec16<T>::N;
  constexpr int L = D / EPL;       // lanes per exact key
  constexpr int TPW = 32 / L;
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

  // ---- pseudo-max over block 0 and the newest block (exact keys)
  {
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
    for (int i0 = warp * TPW; i0 < ntk; i0 += kDeltaWarps * TPW) {
      const int i = i0 + grp;
      const bool ok = i < ntk;
      const int t = i < nb0 ? i : lb0 + (i - nb0);
      float kf[EPL];
      if (ok) load_vec(krow + (size_t)t * D + sub * EPL, kf);
      else {
#pragma unroll
        for (int e = 0; e < EPL; ++e) kf[e] = 0.f;
      }
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
  int spl = (4 * 152 + rows - 1) / rows;
  const int maxblk = a.nblk_cap;
  spl = spl < 1 ? 1 : spl;
  spl = spl > maxblk ? maxblk : spl;
  a.SPL = spl;
  if (s.dtype == 0)
    return s.D == 64 ? delta_g<float, 64>(a, rows, st) : delta_g<float, 128>(a, rows, st);
  return s.D == 64 ? delta_g<bf16, 64>(a, rows, st) : delta_g<bf16, 128>(a, rows, st);
}

}  // namespace sls
