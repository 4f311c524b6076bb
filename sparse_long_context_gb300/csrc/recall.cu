// Selection quality: the share of each query head's full-context softmax
// mass that a page list holds ("Don't read the haystack", Part three:
// attention mass captured by the selected pages).  A diagnostic beside the
// decode step, not on it: it reads every key of the context.
//
// recall_partial_kernel  one CTA per (row, context split): a bitmap of the
//                        row's listed pages in shared memory; every thread
//                        walks tokens of the split and keeps, per head of the
//                        GQA group, the running max m, the total mass z and
//                        the selected mass s of exp(scale * q.k - m); the CTA
//                        merges its threads' triples and writes one per head.
// recall_combine_kernel  merges the splits of each (row, head): s / z.
#include "common.cuh"
#include "status.cuh"
#include "launch.h"

namespace sls {

constexpr int kRecallThreads = 256;
constexpr int kRecallMaxPages = 262144;  // bitmap of 32 KB

struct MassTriple {
  float m, z, s;
};

__device__ __forceinline__ MassTriple mass_merge(MassTriple a, MassTriple b) {
  const float M = fmaxf(a.m, b.m);
  if (M == kNegInf) return a;
  const float fa = a.m == kNegInf ? 0.f : expf(a.m - M);
  const float fb = b.m == kNegInf ? 0.f : expf(b.m - M);
  return MassTriple{M, a.z * fa + b.z * fb, a.s * fa + b.s * fb};
}

template <typename T, int D, int GM>
__global__ void __launch_bounds__(kRecallThreads)
recall_partial_kernel(const void* q_, const void* k_, const int32_t* page_idx, int idx_stride, const int32_t* count,
                      int k_fixed, const int32_t* ctx_len, int Hq, int Hkv, int G, int Cap, int P, int pshift,
                      float scale, int S, float* part) {
  constexpr int EPV = Vec16<T>::N;
  constexpr int NV = D / EPV;
  extern __shared__ uint32_t bitmap[];
  __shared__ float sq[GM][D];
  __shared__ MassTriple red[kRecallThreads / 32][GM];
  const int row = blockIdx.x / S, split = blockIdx.x % S;
  const int b = row / Hkv, h = row % Hkv;
  const int N = clamp_len(ctx_len[b], Cap);
  const int NP = (N + P - 1) >> pshift;
  const int nwords = (Cap >> pshift) / 32 + 1;
  for (int w = threadIdx.x; w < nwords; w += kRecallThreads) bitmap[w] = page_idx ? 0u : 0xffffffffu;
  for (int i = threadIdx.x; i < GM * D; i += kRecallThreads) {
    const int g = i / D, c = i % D;
    sq[g][c] = g < G ? to_f32<T>(static_cast<const T*>(q_)[((size_t)b * Hq + (size_t)h * G + g) * D + c]) * scale
                     : 0.f;
  }
  __syncthreads();
  if (page_idx) {
    int cnt = count ? count[row] : k_fixed;
    cnt = cnt < 0 ? 0 : (cnt > idx_stride ? idx_stride : cnt);
    const int32_t* pl = page_idx + (size_t)row * idx_stride;
    unsigned int bad = 0;
    for (int e = threadIdx.x; e < cnt; e += kRecallThreads) {
      const int pg = pl[e];
      if (pg >= 0 && pg < NP) atomicOr(&bitmap[pg >> 5], 1u << (pg & 31));
      bad += (split == 0 && bad_page_id(pg, Cap >> pshift)) ? 1u : 0u;  // counted by one CTA of the row
    }
    note_bad_pages(bad);
  }
  __syncthreads();
  const int per = (N + S - 1) / S;
  const int t0 = split * per, t1 = min(N, t0 + per);
  MassTriple acc[GM];
#pragma unroll
  for (int g = 0; g < GM; ++g) acc[g] = MassTriple{kNegInf, 0.f, 0.f};
  const T* kb = static_cast<const T*>(k_) + (size_t)row * Cap * D;
  for (int t = t0 + threadIdx.x; t < t1; t += kRecallThreads) {
    float x[GM];
#pragma unroll
    for (int g = 0; g < GM; ++g) x[g] = 0.f;
#pragma unroll 4
    for (int v = 0; v < NV; ++v) {
      float kv[EPV];
      load_vec(kb + (size_t)t * D + v * EPV, kv);
#pragma unroll
      for (int g = 0; g < GM; ++g)
#pragma unroll
        for (int e = 0; e < EPV; ++e) x[g] = fmaf(sq[g][v * EPV + e], kv[e], x[g]);
    }
    const int pg = t >> pshift;
    const float sel = (bitmap[pg >> 5] >> (pg & 31)) & 1u ? 1.f : 0.f;
#pragma unroll
    for (int g = 0; g < GM; ++g) acc[g] = mass_merge(acc[g], MassTriple{x[g], 1.f, sel});
  }
  // merge the CTA's threads per head
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int g = 0; g < GM; ++g) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      MassTriple other{__shfl_xor_sync(0xffffffffu, acc[g].m, o), __shfl_xor_sync(0xffffffffu, acc[g].z, o),
                       __shfl_xor_sync(0xffffffffu, acc[g].s, o)};
      acc[g] = mass_merge(acc[g], other);
    }
    if (lane == 0) red[warp][g] = acc[g];
  }
  __syncthreads();
  if (threadIdx.x < G) {
    const int g = threadIdx.x;
    MassTriple r = red[0][g];
    for (int w = 1; w < kRecallThreads / 32; ++w) r = mass_merge(r, red[w][g]);
    float* o = part + (((size_t)row * S + split) * G + g) * 3;
    o[0] = r.m;
    o[1] = r.z;
    o[2] = r.s;
  }
}

__global__ void recall_combine_kernel(const float* part, int rows, int G, int S, int Hq, int Hkv, float* recall) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= rows * G) return;
  const int row = i / G, g = i % G;
  MassTriple r{kNegInf, 0.f, 0.f};
  for (int s = 0; s < S; ++s) {
    const float* p = part + (((size_t)row * S + s) * G + g) * 3;
    r = mass_merge(r, MassTriple{p[0], p[1], p[2]});
  }
  const int b = row / Hkv, h = row % Hkv;
  recall[(size_t)b * Hq + (size_t)h * G + g] = r.z > 0.f ? r.s / r.z : 1.f;  // an empty context misses nothing
}

int recall_splits(const Shape& s) {
  const int rows = s.B * s.Hkv;
  int S = (2 * sm_count() + rows - 1) / rows;
  return S < 1 ? 1 : (S > 64 ? 64 : S);
}

size_t recall_workspace(const Shape& s) { return (size_t)s.B * s.Hkv * recall_splits(s) * s.G * 3 * sizeof(float); }

bool recall_supported(const Shape& s) { return (s.Cap >> s.pshift) <= kRecallMaxPages; }

template <typename T, int D>
static cudaError_t recall_launch_g(const Shape& s, const void* q, const void* k, const int32_t* page_idx,
                                   int idx_stride, const int32_t* count, int k_fixed, const int32_t* ctx_len,
                                   float* recall, float* part, cudaStream_t st) {
  const int rows = s.B * s.Hkv, S = recall_splits(s);
  const size_t smem = ((size_t)(s.Cap >> s.pshift) / 32 + 1) * 4;
  auto run = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<rows * S, kRecallThreads, smem, st>>>(q, k, page_idx, idx_stride, count, k_fixed, ctx_len, s.Hq, s.Hkv,
                                                  s.G, s.Cap, s.P, s.pshift, s.scale, S, part);
    return cudaGetLastError();
  };
  cudaError_t e;
  if (s.G <= 1) e = run(recall_partial_kernel<T, D, 1>);
  else if (s.G <= 2) e = run(recall_partial_kernel<T, D, 2>);
  else if (s.G <= 4) e = run(recall_partial_kernel<T, D, 4>);
  else e = run(recall_partial_kernel<T, D, 8>);
  if (e != cudaSuccess) return e;
  const int n = rows * s.G;
  recall_combine_kernel<<<(n + 255) / 256, 256, 0, st>>>(part, rows, s.G, S, s.Hq, s.Hkv, recall);
  return cudaGetLastError();
}

cudaError_t launch_recall(const Shape& s, const void* q, const void* k, const int32_t* page_idx, int idx_stride,
                          const int32_t* count, int k_fixed, const int32_t* ctx_len, float* recall, void* ws,
                          cudaStream_t st) {
  float* part = static_cast<float*>(ws);
  if (s.dtype == 0)
    return s.D == 64 ? recall_launch_g<float, 64>(s, q, k, page_idx, idx_stride, count, k_fixed, ctx_len, recall, part, st)
                     : recall_launch_g<float, 128>(s, q, k, page_idx, idx_stride, count, k_fixed, ctx_len, recall, part, st);
  return s.D == 64 ? recall_launch_g<bf16, 64>(s, q, k, page_idx, idx_stride, count, k_fixed, ctx_len, recall, part, st)
                   : recall_launch_g<bf16, 128>(s, q, k, page_idx, idx_stride, count, k_fixed, ctx_len, recall, part, st);
}

DeviceStatus take_status_recall() { return take_status_here(); }

}  // namespace sls
