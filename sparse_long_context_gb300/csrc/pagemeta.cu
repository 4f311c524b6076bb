// Selector metadata kept beside the KV cache:
//  * per-page, per-channel min/max keys ("Don't read the haystack", Part
//    two), built for a whole prefix or folded in one appended key at a time;
//  * 2-bit symmetric mid-rise thumbnails of complete 64-token blocks
//    ("Faster Than Flash", Methodology 1; the append path mirrors its
//    graph-friendly, tensor-indexed cache writes of Methodology 3).
#include "common.cuh"
#include "launch.h"

namespace sls {

// ---------------------------------------------------------------- min / max

// One thread per (page, 16-byte channel vector).
template <typename T, int D>
__global__ void __launch_bounds__(256)
pagemeta_build_kernel(const T* __restrict__ k, const int32_t* __restrict__ ctx_len, T* kmin,
                      T* kmax, int Hkv, int Cap, int P, int pshift, int pages_per_cta) {
  constexpr int EPL = Vec16<T>::N;
  constexpr int L = D / EPL;
  const int row = blockIdx.y;
  const int b = row / Hkv;
  const int N = clamp_len(ctx_len[b], Cap);
  const int NP = (N + P - 1) >> pshift;
  const int p = blockIdx.x * pages_per_cta + threadIdx.x / L;
  const int sub = threadIdx.x % L;
  if (threadIdx.x / L >= pages_per_cta || p >= NP) return;
  const T* src = k + ((size_t)row * Cap + ((size_t)p << pshift)) * D + sub * EPL;
  const int t1 = min(P, N - (p << pshift));
  float lo[EPL], hi[EPL];
  load_vec(src, lo);
#pragma unroll
  for (int e = 0; e < EPL; ++e) hi[e] = lo[e];
  for (int t = 1; t < t1; ++t) {
    float x[EPL];
    load_vec(src + (size_t)t * D, x);
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      lo[e] = fminf(lo[e], x[e]);
      hi[e] = fmaxf(hi[e], x[e]);
    }
  }
  const size_t o = ((size_t)row * (Cap >> pshift) + p) * D + sub * EPL;
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    kmin[o + e] = from_f32<T>(lo[e]);  // exact: the value is one of the keys
    kmax[o + e] = from_f32<T>(hi[e]);
  }
}

// One warp per (b, kv head) row.
template <typename T, int D>
__global__ void __launch_bounds__(128)
pagemeta_update_kernel(const T* __restrict__ k, const int32_t* __restrict__ pos, T* kmin,
                       T* kmax, int rows, int Hkv, int Cap, int P, int pshift) {
  constexpr int EPL = Vec16<T>::N;
  constexpr int L = D / EPL;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows || lane >= L) return;
  const int t = pos[row / Hkv];
  if (t < 0 || t >= Cap) return;
  const int p = t >> pshift;
  float x[EPL];
  load_vec(k + ((size_t)row * Cap + t) * D + lane * EPL, x);
  const size_t o = ((size_t)row * (Cap >> pshift) + p) * D + lane * EPL;
  if ((t & (P - 1)) == 0) {
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      kmin[o + e] = from_f32<T>(x[e]);
      kmax[o + e] = from_f32<T>(x[e]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      kmin[o + e] = from_f32<T>(fminf(to_f32<T>(kmin[o + e]), x[e]));
      kmax[o + e] = from_f32<T>(fmaxf(to_f32<T>(kmax[o + e]), x[e]));
    }
  }
}

// One CTA per sequence: the new token's key and value of every KV head go to
// position ctx_len[b] (when below Cap), the key is folded into its page's
// min/max (the page's first token resets them), the position is reported in
// pos_out, and ctx_len[b] advances by one.  Every thread reads ctx_len before
// the barrier; only then does thread 0 advance it.
template <typename T, int D>
__global__ void __launch_bounds__(256)
decode_append_kernel(const T* __restrict__ k_new, const T* __restrict__ v_new, T* k, T* v, T* kmin, T* kmax,
                     int32_t* ctx_len, int32_t* pos_out, int Hkv, int Cap, int P, int pshift) {
  // after the previous step (which reads ctx_len and the cache); the next
  // kernel of the loop may then start its launch, and waits for this one
  pdl_wait_then_release();
  const int b = blockIdx.x;
  const int t = ctx_len[b];
  __syncthreads();
  const bool ok = t >= 0 && t < Cap;
  if (ok) {
    for (int i = threadIdx.x; i < Hkv * D; i += blockDim.x) {
      const size_t row = (size_t)b * Hkv + i / D;
      const int c = i % D;
      const T kx = k_new[row * D + c];
      k[(row * Cap + t) * D + c] = kx;
      v[(row * Cap + t) * D + c] = v_new[row * D + c];
      if (kmin) {
        const size_t o = (row * (Cap >> pshift) + (t >> pshift)) * D + c;
        if ((t & (P - 1)) == 0) {
          kmin[o] = kx;
          kmax[o] = kx;
        } else {
          const float x = to_f32<T>(kx);
          kmin[o] = from_f32<T>(fminf(to_f32<T>(kmin[o]), x));
          kmax[o] = from_f32<T>(fmaxf(to_f32<T>(kmax[o]), x));
        }
      }
    }
  }
  if (threadIdx.x == 0) {
    if (pos_out) pos_out[b] = ok ? t : -1;
    if (ok) ctx_len[b] = t + 1;
  }
}

// ---------------------------------------------------------------- thumbnails

// Code of one element: 3 if k >= s/2, 2 if 0 <= k < s/2, 1 if -s/2 <= k < 0,
// 0 below; s/2 of a bf16 or fp32 magnitude is exact, so the comparisons are.
__device__ __forceinline__ uint32_t thumb_code(float x, float half) {
  return x >= half ? 3u : (x >= 0.f ? 2u : (x >= -half ? 1u : 0u));
}

// 8-bit residual of one element ("Faster Than Flash", Methodology 1: the
// key splits into the 2-bit thumbnail and an 8-bit residual): the error
// e = k - k^ of the mid-rise code lies in [-s/4, s/4] and is stored as
// r = rint(e * 508 / s) in [-127, 127] on the thumbnail's scale s (0 when
// s = 0).  Every step is one IEEE float32 operation, so the integer does not
// depend on contraction or on the division's implementation.
__device__ __forceinline__ int8_t residual_code(float x, float s, uint32_t code) {
  if (!(s > 0.f)) return 0;
  const float kh = __fmul_rn((float)code - 1.5f, s) * 0.5f;  // exact: a level of the thumbnail
  const float q = __fdiv_rn(__fmul_rn(__fsub_rn(x, kh), 508.f), s);
  return (int8_t)fminf(fmaxf(rintf(q), -127.f), 127.f);
}

// Quantise block j of `row` (block tokens, all valid), and its residuals
// when `res` is given.  blockDim.x == D.
template <typename T, int D>
__device__ __forceinline__ void quantise_block(const T* __restrict__ k, uint8_t* codes, T* scales,
                                               int8_t* res, int row, int j, int Cap, int block, int nblk_cap) {
  __shared__ float s_half[D];
  const int c = threadIdx.x;
  const T* src = k + ((size_t)row * Cap + (size_t)j * block) * D;
  float s = 0.f;
  for (int t = 0; t < block; ++t) s = fmaxf(s, fabsf(to_f32<T>(src[(size_t)t * D + c])));
  scales[((size_t)row * nblk_cap + j) * D + c] = from_f32<T>(s);
  s_half[c] = 0.5f * s;
  __syncthreads();
  constexpr int BPT = D / 4;  // code bytes per token
  uint8_t* dst = codes + ((size_t)row * Cap + (size_t)j * block) * BPT;
  for (int i = threadIdx.x; i < block * BPT; i += D) {
    const int t = i / BPT, by = i % BPT;
    const T* x = src + (size_t)t * D + by * 4;
    uint32_t v = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) v |= thumb_code(to_f32<T>(x[u]), s_half[by * 4 + u]) << (2 * u);
    dst[i] = (uint8_t)v;
  }
  if (res) {
    // thread c walks channel c: the scale is its own
    int8_t* rd = res + ((size_t)row * Cap + (size_t)j * block) * D + c;
    for (int t = 0; t < block; ++t) {
      const float x = to_f32<T>(src[(size_t)t * D + c]);
      rd[(size_t)t * D] = residual_code(x, s, thumb_code(x, s_half[c]));
    }
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(D)
thumb_build_kernel(const T* __restrict__ k, const int32_t* __restrict__ ctx_len, uint8_t* codes,
                   T* scales, int8_t* res, int Hkv, int Cap, int block, int nblk_cap) {
  const int row = blockIdx.y, j = blockIdx.x;
  const int N = clamp_len(ctx_len[row / Hkv], Cap);
  if ((j + 1) * block > N) return;
  quantise_block<T, D>(k, codes, scales, res, row, j, Cap, block, nblk_cap);
}

template <typename T, int D>
__global__ void __launch_bounds__(D)
thumb_update_kernel(const T* __restrict__ k, const int32_t* __restrict__ pos, uint8_t* codes,
                    T* scales, int8_t* res, int Hkv, int Cap, int block, int nblk_cap) {
  pdl_wait_then_release();
  const int row = blockIdx.x;
  const int t = pos[row / Hkv];
  if (t < 0 || t >= Cap || (t + 1) % block != 0) return;
  quantise_block<T, D>(k, codes, scales, res, row, t / block, Cap, block, nblk_cap);
}

// ---------------------------------------------------------------- launches

template <typename T, int D>
static cudaError_t pm_build(const Shape& s, const void* k, const int32_t* ctx, void* kmin,
                            void* kmax, cudaStream_t st) {
  constexpr int L = D / Vec16<T>::N;
  const int ppc = 256 / L;
  dim3 grid(((s.Cap >> s.pshift) + ppc - 1) / ppc, s.B * s.Hkv);
  pagemeta_build_kernel<T, D><<<grid, 256, 0, st>>>(static_cast<const T*>(k), ctx, static_cast<T*>(kmin),
                                                    static_cast<T*>(kmax), s.Hkv, s.Cap, s.P, s.pshift, ppc);
  return cudaGetLastError();
}

cudaError_t launch_pagemeta_build(const Shape& s, const void* k, const int32_t* ctx_len,
                                  void* kmin, void* kmax, cudaStream_t st) {
  if (s.dtype == 0)
    return s.D == 64 ? pm_build<float, 64>(s, k, ctx_len, kmin, kmax, st)
                     : pm_build<float, 128>(s, k, ctx_len, kmin, kmax, st);
  return s.D == 64 ? pm_build<bf16, 64>(s, k, ctx_len, kmin, kmax, st)
                   : pm_build<bf16, 128>(s, k, ctx_len, kmin, kmax, st);
}

template <typename T, int D>
static cudaError_t pm_update(const Shape& s, const void* k, const int32_t* pos, void* kmin,
                             void* kmax, cudaStream_t st) {
  const int rows = s.B * s.Hkv;
  pagemeta_update_kernel<T, D><<<(rows + 3) / 4, 128, 0, st>>>(
      static_cast<const T*>(k), pos, static_cast<T*>(kmin), static_cast<T*>(kmax), rows, s.Hkv, s.Cap,
      s.P, s.pshift);
  return cudaGetLastError();
}

cudaError_t launch_pagemeta_update(const Shape& s, const void* k, const int32_t* pos, void* kmin,
                                   void* kmax, cudaStream_t st) {
  if (s.dtype == 0)
    return s.D == 64 ? pm_update<float, 64>(s, k, pos, kmin, kmax, st)
                     : pm_update<float, 128>(s, k, pos, kmin, kmax, st);
  return s.D == 64 ? pm_update<bf16, 64>(s, k, pos, kmin, kmax, st)
                   : pm_update<bf16, 128>(s, k, pos, kmin, kmax, st);
}

template <typename T, int D>
static cudaError_t dec_append(const Shape& s, const void* k_new, const void* v_new, void* k, void* v, void* kmin,
                              void* kmax, int32_t* ctx_len, int32_t* pos_out, cudaStream_t st) {
  cudaError_t e = launch_pdl(decode_append_kernel<T, D>, dim3(s.B), dim3(256), 0, st,
                             static_cast<const T*>(k_new), static_cast<const T*>(v_new), static_cast<T*>(k),
                             static_cast<T*>(v), static_cast<T*>(kmin), static_cast<T*>(kmax), ctx_len, pos_out,
                             s.Hkv, s.Cap, s.P, s.pshift);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_decode_append(const Shape& s, const void* k_new, const void* v_new, void* k, void* v,
                                 void* kmin, void* kmax, int32_t* ctx_len, int32_t* pos_out, cudaStream_t st) {
  if (s.dtype == 0)
    return s.D == 64 ? dec_append<float, 64>(s, k_new, v_new, k, v, kmin, kmax, ctx_len, pos_out, st)
                     : dec_append<float, 128>(s, k_new, v_new, k, v, kmin, kmax, ctx_len, pos_out, st);
  return s.D == 64 ? dec_append<bf16, 64>(s, k_new, v_new, k, v, kmin, kmax, ctx_len, pos_out, st)
                   : dec_append<bf16, 128>(s, k_new, v_new, k, v, kmin, kmax, ctx_len, pos_out, st);
}

template <typename T, int D>
static cudaError_t th_build(const Shape& s, const void* k, const int32_t* ctx, int block,
                            uint8_t* codes, void* scales, int8_t* res, cudaStream_t st) {
  const int nblk = s.Cap / block;
  dim3 grid(nblk, s.B * s.Hkv);
  thumb_build_kernel<T, D><<<grid, D, 0, st>>>(static_cast<const T*>(k), ctx, codes, static_cast<T*>(scales),
                                               res, s.Hkv, s.Cap, block, nblk);
  return cudaGetLastError();
}

cudaError_t launch_thumb_build(const Shape& s, const void* k, const int32_t* ctx_len, int block,
                               uint8_t* codes, void* scales, int8_t* res, cudaStream_t st) {
  if (s.dtype == 0)
    return s.D == 64 ? th_build<float, 64>(s, k, ctx_len, block, codes, scales, res, st)
                     : th_build<float, 128>(s, k, ctx_len, block, codes, scales, res, st);
  return s.D == 64 ? th_build<bf16, 64>(s, k, ctx_len, block, codes, scales, res, st)
                   : th_build<bf16, 128>(s, k, ctx_len, block, codes, scales, res, st);
}

template <typename T, int D>
static cudaError_t th_update(const Shape& s, const void* k, const int32_t* pos, int block,
                             uint8_t* codes, void* scales, int8_t* res, cudaStream_t st) {
  cudaError_t e = launch_pdl(thumb_update_kernel<T, D>, dim3(s.B * s.Hkv), dim3(D), 0, st,
                             static_cast<const T*>(k), pos, codes, static_cast<T*>(scales), res, s.Hkv, s.Cap,
                             block, s.Cap / block);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_thumb_update(const Shape& s, const void* k, const int32_t* pos, int block,
                                uint8_t* codes, void* scales, int8_t* res, cudaStream_t st) {
  if (s.dtype == 0)
    return s.D == 64 ? th_update<float, 64>(s, k, pos, block, codes, scales, res, st)
                     : th_update<float, 128>(s, k, pos, block, codes, scales, res, st);
  return s.D == 64 ? th_update<bf16, 64>(s, k, pos, block, codes, scales, res, st)
                   : th_update<bf16, 128>(s, k, pos, block, codes, scales, res, st);
}

}  // namespace sls
