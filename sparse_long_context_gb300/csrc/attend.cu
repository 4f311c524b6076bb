// Split-K sparse decode attention (stage one) and the split combine (stage
// two) of two-stage flash-decoding, over pages selected through a page list
// ("Don't read the haystack", Part one and the sparse twin of Part two;
// "perf(core): fused sparse-attention decode via page indirection", The
// reduction: token i of list entry e is position list[e]*P + i of the row).
//
// This file holds the CUDA-core kernels, which serve every dtype.  The
// tensor-core kernel for bf16 lives in attend_mma.cu.
#include "attend_common.cuh"
#include "launch.h"

namespace sls {

// One CTA per (row, split); NW warps each run an online softmax over
// 32-token chunks of the slice (scores of a chunk first, then one max
// update, then the P.V accumulation), and the warps merge at the end.
// A token's D elements are spread over L lanes as 16-byte vectors; dot
// products are reduced with butterfly shuffles.
template <typename T, int D, int GM, int NW>
__global__ void __launch_bounds__(NW * 32)
attend_cc_kernel(const AttendArgs a) {
  pdl_wait_then_release();
  constexpr int EPL = Vec16<T>::N;
  constexpr int L = D / EPL;
  constexpr int TPW = 32 / L;
  constexpr int CH = 32;
  constexpr int STEPS = CH / TPW;
  constexpr int UNR = STEPS < 8 ? STEPS : 8;
  __shared__ float sP[NW][GM][CH];
  __shared__ float sAcc[NW][GM][D];
  __shared__ float sM[NW][GM];
  __shared__ float sL[NW][GM];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / L, sub = lane % L;
  const int row = blockIdx.x / a.S, split = blockIdx.x % a.S;
  const int b = row / a.Hkv, h = row % a.Hkv;
  const int G = a.G;
  const Slice sl = attend_slice(a, row, split);
  const int ntok = sl.nent << a.pshift;
  const int32_t* plist = a.page_idx ? a.page_idx + (size_t)row * a.idx_stride + sl.e0 : nullptr;
  const T* kb = static_cast<const T*>(a.k) + (size_t)row * a.Cap * D + sub * EPL;
  const T* vb = static_cast<const T*>(a.v) + (size_t)row * a.Cap * D + sub * EPL;
  stage_page_list(nullptr, 0, plist, sl.e0, sl.nent, a.Cap >> a.pshift, threadIdx.x, NW * 32);  // count bad ids

  float qv[GM][EPL];
  {
    const T* qp = static_cast<const T*>(a.q) + ((size_t)b * a.Hq + (size_t)h * G) * D + sub * EPL;
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      float t[EPL];
      if (g < G) load_vec(qp + (size_t)g * D, t);
#pragma unroll
      for (int e = 0; e < EPL; ++e) qv[g][e] = g < G ? t[e] * a.qscale : 0.f;
    }
  }
  float m[GM], l[GM], acc[GM][EPL];
#pragma unroll
  for (int g = 0; g < GM; ++g) {
    m[g] = kNegInf;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[g][e] = 0.f;
  }

  const int nchunks = (ntok + CH - 1) / CH;
  for (int c = warp; c < nchunks; c += NW) {
    // page ids of the chunk: lane i holds list entry ebase + i
    const int ebase = (c * CH) >> a.pshift;
    int my_pg = -1;
    if (ebase + lane < sl.nent) my_pg = plist ? plist[ebase + lane] : sl.e0 + ebase + lane;
    int pos[STEPS];
#pragma unroll
    for (int st = 0; st < STEPS; ++st) {
      const int j = c * CH + st * TPW + grp;
      const int pg = __shfl_sync(0xffffffffu, my_pg, ((j >> a.pshift) - ebase) & 31);
      pos[st] = j < ntok ? token_position(a, pg, j, sl.N) : -1;
    }
    // pass A: scores of the chunk
#pragma unroll
    for (int s0 = 0; s0 < STEPS; s0 += UNR) {
      uint4 kr[UNR];
#pragma unroll
      for (int u = 0; u < UNR; ++u)
        kr[u] = pos[s0 + u] >= 0 ? ldg_stream(kb + (size_t)pos[s0 + u] * D) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        float kf[EPL];
        unpack_vec(kr[u], kf);
        float s[GM];
#pragma unroll
        for (int g = 0; g < GM; ++g) {
          s[g] = 0.f;
          if (g < G) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) s[g] = fmaf(qv[g][e], kf[e], s[g]);
          }
        }
#pragma unroll
        for (int o = L / 2; o > 0; o >>= 1) {
#pragma unroll
          for (int g = 0; g < GM; ++g) s[g] += __shfl_xor_sync(0xffffffffu, s[g], o);
        }
        if (sub == 0) {
#pragma unroll
          for (int g = 0; g < GM; ++g) sP[warp][g][(s0 + u) * TPW + grp] = pos[s0 + u] >= 0 ? s[g] : kNegInf;
        }
      }
    }
    __syncwarp();
    // pass B: chunk max, rescale, probabilities (lane = token of the chunk)
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      if (g >= G) break;
      const float s = sP[warp][g][lane];
      const float mn = fmaxf(m[g], warp_max(s));
      float alpha = 1.f, p = 0.f;
      if (mn != kNegInf) {
        alpha = exp2f(m[g] - mn);  // m = -inf gives 0
        p = exp2f(s - mn);         // s = -inf gives 0
      }
      sP[warp][g][lane] = p;
      l[g] = l[g] * alpha + warp_sum(p);
      m[g] = mn;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[g][e] *= alpha;
    }
    __syncwarp();
    // pass C: accumulate P.V
#pragma unroll
    for (int s0 = 0; s0 < STEPS; s0 += UNR) {
      uint4 vr[UNR];
#pragma unroll
      for (int u = 0; u < UNR; ++u)
        vr[u] = pos[s0 + u] >= 0 ? ldg_stream(vb + (size_t)pos[s0 + u] * D) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        if (pos[s0 + u] < 0) continue;
        float vf[EPL];
        unpack_vec(vr[u], vf);
#pragma unroll
        for (int g = 0; g < GM; ++g) {
          if (g < G) {
            const float p = sP[warp][g][(s0 + u) * TPW + grp];
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[g][e] = fmaf(p, vf[e], acc[g][e]);
          }
        }
      }
    }
    __syncwarp();
  }

  // reduce the token slots of the warp (lanes with the same sub)
#pragma unroll
  for (int o = L; o < 32; o <<= 1) {
#pragma unroll
    for (int g = 0; g < GM; ++g) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[g][e] += __shfl_xor_sync(0xffffffffu, acc[g][e], o);
    }
  }
  if (grp == 0) {
#pragma unroll
    for (int g = 0; g < GM; ++g) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) sAcc[warp][g][sub * EPL + e] = acc[g][e];
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      sM[warp][g] = m[g];
      sL[warp][g] = l[g];
    }
  }
  __syncthreads();

  // merge the warps and write the partial of every query head
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
        av += sAcc[w][g][d] * f;
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
  if (a.tickets) combine_row_if_last<T, D, NW * 32>(a, row, a.S);
}

// Stage two: one warp per (b, query head).  Lane s holds split s's max and
// normaliser; the accumulators of up to 8 splits are loaded together.
template <typename T, int D>
__global__ void __launch_bounds__(128)
combine_kernel(const float* __restrict__ o_part, const float* __restrict__ m_part,
               const float* __restrict__ l_part, int S, const float* __restrict__ sink,
               T* __restrict__ out, float* __restrict__ lse, int Hq, int total) {
  pdl_wait_then_release();
  constexpr int CPL = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int idx = blockIdx.x * 4 + warp;
  if (idx >= total) return;
  const int hq = idx % Hq;
  const float* mp = m_part + (size_t)idx * S;
  const float* lp = l_part + (size_t)idx * S;
  const float* op = o_part + (size_t)idx * S * D + lane * CPL;
  float M = kNegInf;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, mp[s]);
  M = warp_max(M);
  const float sk = sink ? sink[hq] : kNegInf;
  M = fmaxf(M, sk);
  float acc[CPL];
#pragma unroll
  for (int i = 0; i < CPL; ++i) acc[i] = 0.f;
  float Ls = 0.f;
  if (M != kNegInf) {
    for (int s0 = 0; s0 < S; s0 += 32) {
      const int s = s0 + lane;
      float w = 0.f;
      if (s < S) {
        const float ms = mp[s];
        w = ms == kNegInf ? 0.f : expf(ms - M);
        Ls += lp[s] * w;
      }
      const int n = min(32, S - s0);
      for (int j0 = 0; j0 < n; j0 += 8) {
        float v[8][CPL];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
#pragma unroll
          for (int i = 0; i < CPL; ++i) v[j][i] = j0 + j < n ? op[(size_t)(s0 + j0 + j) * D + i] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float wj = __shfl_sync(0xffffffffu, w, (j0 + j) & 31);
#pragma unroll
          for (int i = 0; i < CPL; ++i) acc[i] = fmaf(v[j][i], wj, acc[i]);
        }
      }
    }
    Ls = warp_sum(Ls);
    if (sink) Ls += expf(sk - M);
  }
  const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
  for (int i = 0; i < CPL; ++i) out[(size_t)idx * D + lane * CPL + i] = from_f32<T>(acc[i] * inv);
  if (lse && lane == 0) lse[idx] = Ls == 0.f ? kNegInf : M + logf(Ls);
}

template <typename T, int D, int GM>
static cudaError_t attend_cc(const AttendArgs& a, int rows, cudaStream_t st) {
  constexpr int NW = 4;
  cudaError_t e = launch_pdl(attend_cc_kernel<T, D, GM, NW>, dim3(rows * a.S), dim3(NW * 32), 0, st, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t attend_cc_g(const AttendArgs& a, int rows, cudaStream_t st) {
  if (a.G <= 1) return attend_cc<T, D, 1>(a, rows, st);
  if (a.G <= 2) return attend_cc<T, D, 2>(a, rows, st);
  if (a.G <= 4) return attend_cc<T, D, 4>(a, rows, st);
  return attend_cc<T, D, 8>(a, rows, st);
}

cudaError_t launch_attend_mma(const Shape& s, const AttendArgs& a, cudaStream_t st, bool* handled);
cudaError_t launch_attend_tma(const Shape& s, const AttendArgs& a, cudaStream_t st, bool* handled);
const void* attend_mma_kernel_ptr(int D);
size_t attend_mma_kernel_smem(int D);
int attend_mma_kernel_threads();

int max_auto_splits(const Shape& s) {
  // splits per row the library may choose by itself (sizes the workspace)
  const int rows = s.B * s.Hkv;
  return (4 * sm_count() + rows - 1) / rows;
}

int attend_default_splits(const Shape& s, int max_entries) {
  // one wave of attend CTAs over all rows (at most one CTA per slot), each
  // slice at least 64 tokens
  static int mma_per_sm[2] = {0, 0};  // D = 64, D = 128
  const int di = s.D == 64 ? 0 : 1;
  if (mma_per_sm[di] == 0) {
    cudaFuncSetAttribute(attend_mma_kernel_ptr(s.D), cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)attend_mma_kernel_smem(s.D));
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&mma_per_sm[di], attend_mma_kernel_ptr(s.D),
                                                      attend_mma_kernel_threads(),
                                                      attend_mma_kernel_smem(s.D)) != cudaSuccess)
      mma_per_sm[di] = 1;
  }
  if (attend_tma_eligible(s)) return attend_tma_splits(s, (int)(((long long)max_entries << s.pshift) / 16));
  const int per_sm = mma_per_sm[di];
  const int rows = s.B * s.Hkv;
  const int slots = sm_count() * (per_sm > 0 ? per_sm : 1);
  int S = slots / rows;
  const int cap = (int)(((long long)max_entries << s.pshift) / 64);
  if (S > cap) S = cap;
  if (S < 1) S = 1;
  if (S > 1024) S = 1024;
  return S;
}

cudaError_t launch_attend(const Shape& s, const void* q, const void* k, const void* v,
                          const int32_t* page_idx, int idx_stride, const int32_t* count,
                          int k_fixed, const int32_t* ctx_len, int num_splits,
                          float* o_part, float* m_part, float* l_part, cudaStream_t st,
                          const FusedCombine* fused) {
  AttendArgs a;
  a.tickets = fused ? fused->tickets : nullptr;
  a.sink = fused ? fused->sink : nullptr;
  a.out = fused ? fused->out : nullptr;
  a.lse = fused ? fused->lse : nullptr;
  a.q = q; a.k = k; a.v = v;
  a.page_idx = page_idx; a.count = count; a.ctx_len = ctx_len;
  a.o_part = o_part; a.m_part = m_part; a.l_part = l_part;
  a.idx_stride = idx_stride; a.k_fixed = k_fixed; a.S = num_splits;
  a.cluster = 0;
  a.test_wait = (s.flags & kFlagTestWaitTimeout) ? 1 : 0;
  if (num_splits == 0) {  // the library schedules (fused call only)
    const int entries = page_idx ? (count ? idx_stride : k_fixed) : (s.Cap >> s.pshift);
    a.S = attend_default_splits(s, entries > 0 ? entries : 1);
    if (a.S > max_auto_splits(s)) a.S = max_auto_splits(s);
  }
  a.Hq = s.Hq; a.Hkv = s.Hkv; a.G = s.G; a.Cap = s.Cap; a.P = s.P; a.pshift = s.pshift;
  a.qscale = s.scale * kLog2e;
  const int rows = s.B * s.Hkv;
  if (!(s.flags & kFlagCudaCores)) {
    bool handled = false;
    cudaError_t e = launch_attend_tma(s, a, st, &handled);
    if (handled) {
      stat_add(kStatAttendTma);
      return e;
    }
    e = launch_attend_mma(s, a, st, &handled);
    if (handled) {
      stat_add(kStatAttendMma);
      return e;
    }
  }
  stat_add(kStatAttendCudaCores);
  if (s.dtype == 0) {
    return s.D == 64 ? attend_cc_g<float, 64>(a, rows, st) : attend_cc_g<float, 128>(a, rows, st);
  }
  return s.D == 64 ? attend_cc_g<bf16, 64>(a, rows, st) : attend_cc_g<bf16, 128>(a, rows, st);
}

cudaError_t launch_combine(const Shape& s, const float* o_part, const float* m_part,
                           const float* l_part, int num_splits, const float* sink,
                           void* out, float* lse, cudaStream_t st) {
  const int total = s.B * s.Hq;
  const int grid = (total + 3) / 4;
  stat_add(kStatCombine);
  cudaError_t e;
  if (s.dtype == 0) {
    if (s.D == 64)
      e = launch_pdl(combine_kernel<float, 64>, dim3(grid), dim3(128), 0, st, o_part, m_part, l_part, num_splits, sink,
                     static_cast<float*>(out), lse, (int)s.Hq, total);
    else
      e = launch_pdl(combine_kernel<float, 128>, dim3(grid), dim3(128), 0, st, o_part, m_part, l_part, num_splits, sink,
                     static_cast<float*>(out), lse, (int)s.Hq, total);
  } else {
    if (s.D == 64)
      e = launch_pdl(combine_kernel<bf16, 64>, dim3(grid), dim3(128), 0, st, o_part, m_part, l_part, num_splits, sink,
                     static_cast<bf16*>(out), lse, (int)s.Hq, total);
    else
      e = launch_pdl(combine_kernel<bf16, 128>, dim3(grid), dim3(128), 0, st, o_part, m_part, l_part, num_splits, sink,
                     static_cast<bf16*>(out), lse, (int)s.Hq, total);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

DeviceStatus take_status_attend_cc() { return take_status_here(); }

}  // namespace sls
