// Arguments and page-list slicing shared by the attend kernels.
#pragma once

#include "common.cuh"
#include "status.cuh"

namespace sls {

struct AttendArgs {
  const void* q;
  const void* k;
  const void* v;
  const int32_t* page_idx;
  const int32_t* count;
  const int32_t* ctx_len;
  float* o_part;
  float* m_part;
  float* l_part;
  int idx_stride, k_fixed, S;
  int Hq, Hkv, G, Cap, P, pshift;
  float qscale;  // softmax scale * log2(e): scores are kept in base-2 units
  // fused combine (all null when the caller combines separately)
  int32_t* tickets;   // [rows] arrival counters, zero between calls
  const float* sink;  // [Hq] or null
  void* out;          // [B, Hq, D] dtype
  float* lse;         // [B, Hq] or null
  int cluster;        // 1: the S splits of a row form one thread-block cluster and
                      // combine through distributed shared memory (no partials in global memory)
  int test_wait = 0;  // wait-timeout test hook: CTA 0 plants a copy phase that never completes
};

// Slice [e0, e1) of row `row`'s page list handled by split `split`.
struct Slice {
  int N, e0, nent;
};
__device__ __forceinline__ Slice attend_slice(const AttendArgs& a, int row, int split) {
  const int b = row / a.Hkv;
  Slice sl;
  sl.N = clamp_len(a.ctx_len[b], a.Cap);
  int cnt;
  if (a.page_idx == nullptr) {
    cnt = (sl.N + a.P - 1) >> a.pshift;
  } else {
    cnt = a.count ? a.count[row] : a.k_fixed;
    cnt = cnt < 0 ? 0 : (cnt > a.idx_stride ? a.idx_stride : cnt);
  }
  const int per = (cnt + a.S - 1) / a.S;
  sl.e0 = split * per;
  const int e1 = min(sl.e0 + per, cnt);
  sl.nent = e1 > sl.e0 ? e1 - sl.e0 : 0;
  return sl;
}

// Copies list entries [0, min(nent, cap)) into s_pg (shared memory) and counts
// the entries of [0, nent) that are neither a page of the pool nor -1, once
// per CTA (bad entries are skipped by the kernels: they give no token).
// plist null: the dense list e0, e0 + 1, ...
__device__ __forceinline__ void stage_page_list(int* s_pg, int cap, const int32_t* plist, int e0, int nent,
                                                int npages, int tid, int nthreads) {
  unsigned int bad = 0;
  for (int e = tid; e < nent; e += nthreads) {
    const int pg = plist ? __ldg(plist + e) : e0 + e;
    if (e < cap) s_pg[e] = pg;
    bad += bad_page_id(pg, npages) ? 1u : 0u;
  }
  note_bad_pages(bad);
}

// Position of a token given its page (or -1 when the slot is empty, the
// page is out of range or the position is past the context).
__device__ __forceinline__ int token_position(const AttendArgs& a, int pg, int j, int N) {
  if ((unsigned)pg >= (unsigned)(a.Cap >> a.pshift)) return -1;
  const int p = (pg << a.pshift) + (j & (a.P - 1));
  return p < N ? p : -1;
}

// Stage two for one row, run by the CTA that finishes the row last: the
// CTAs of a row take a ticket after writing their partials (release), and
// the last one reads every split of the row's query heads (acquire) and
// writes the merged output.  Nothing waits on another CTA.  The weights
// exp(m_s - M) of all splits are formed in parallel (a lane per split), then
// the accumulators are gathered with independent 16-byte loads.
constexpr int kCombineMaxS = 64;  // splits whose weights are kept in shared memory (two per lane)

template <typename T, int D, int NT>
__device__ __forceinline__ void combine_row_if_last(const AttendArgs& a, int row, int nseg) {
  __shared__ int s_last;
  __shared__ float s_w[8][kCombineMaxS];
  __shared__ float s_m[8], s_inv[8];
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(a.tickets + row, 1) == nseg - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int b = row / a.Hkv, h = row % a.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int NW = NT / 32;
  const int S = nseg;  // partials written for this row (slot stride a.S)
  const size_t hq0 = (size_t)b * a.Hq + (size_t)h * a.G;
  for (int g = warp; g < a.G; g += NW) {
    const float* mp = a.m_part + (hq0 + g) * a.S;
    const float* lp = a.l_part + (hq0 + g) * a.S;
    // the first 64 splits' max and sum in registers, loaded at once
    float m2[2], l2[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int s = lane + 32 * u;
      m2[u] = s < S ? __ldcg(mp + s) : kNegInf;
      l2[u] = s < S ? __ldcg(lp + s) : 0.f;
    }
    float M = fmaxf(m2[0], m2[1]);
    for (int s = lane + 64; s < S; s += 32) M = fmaxf(M, __ldcg(mp + s));
    M = warp_max(M);
    const float sk = a.sink ? a.sink[h * a.G + g] : kNegInf;
    M = fmaxf(M, sk);
    float Ls = 0.f;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int s = lane + 32 * u;
      const float w = (m2[u] == kNegInf || M == kNegInf) ? 0.f : expf(m2[u] - M);
      Ls += l2[u] * w;
      if (s < S) s_w[g][s] = w;  // kCombineMaxS = 64
    }
    for (int s = lane + 64; s < S; s += 32) {
      const float ms = __ldcg(mp + s);
      const float w = (ms == kNegInf || M == kNegInf) ? 0.f : expf(ms - M);
      Ls += __ldcg(lp + s) * w;
    }
    Ls = warp_sum(Ls);
    if (a.sink && M != kNegInf) Ls += expf(sk - M);
    if (lane == 0) {
      s_m[g] = M;
      s_inv[g] = Ls > 0.f ? 1.f / Ls : 0.f;
      if (a.lse) a.lse[hq0 + g] = Ls == 0.f ? kNegInf : M + logf(Ls);
    }
  }
  __syncthreads();
  constexpr int C4 = D / 4;
  for (int it = threadIdx.x; it < a.G * C4; it += NT) {
    const int g = it / C4, c = it % C4;
    const float4* op = reinterpret_cast<const float4*>(a.o_part + (hq0 + g) * a.S * D) + c;
    const float* mp = a.m_part + (hq0 + g) * a.S;
    const float M = s_m[g];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < S; s0 += 8) {
      float4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        v[j] = s0 + j < S ? __ldcg(op + (size_t)(s0 + j) * C4) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int s = s0 + j;
        if (s >= S) break;
        float w;
        if (s < kCombineMaxS) {
          w = s_w[g][s];
        } else {
          const float ms = __ldcg(mp + s);
          w = (ms == kNegInf || M == kNegInf) ? 0.f : expf(ms - M);
        }
        acc.x = fmaf(v[j].x, w, acc.x);
        acc.y = fmaf(v[j].y, w, acc.y);
        acc.z = fmaf(v[j].z, w, acc.z);
        acc.w = fmaf(v[j].w, w, acc.w);
      }
    }
    const float inv = s_inv[g];
    T* o = static_cast<T*>(a.out) + (hq0 + g) * D + 4 * c;
    o[0] = from_f32<T>(acc.x * inv);
    o[1] = from_f32<T>(acc.y * inv);
    o[2] = from_f32<T>(acc.z * inv);
    o[3] = from_f32<T>(acc.w * inv);
  }
  if (threadIdx.x == 0) a.tickets[row] = 0;  // ready for the next call
}

}  // namespace sls
