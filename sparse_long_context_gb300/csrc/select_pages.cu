// Quest-style page selection, fused: page scores and the per-row top-k in
// one launch ("Don't read the haystack", Part two: bound every page's
// score by sum_c max(q_c*kmin_c, q_c*kmax_c), keep the top k plus the sink
// page and the last local pages).
//
// One thread-block cluster of kCluster CTAs owns one (b, kv head) row.
// Each CTA scores a contiguous chunk of the row's pages into shared memory
// as order-preserving 32-bit keys, then the cluster runs an MSB-first radix
// select (4 passes of 8-bit digits) whose histograms are summed across the
// cluster through distributed shared memory.  The k-th key T and the number
// of T-valued keys still to take come out of the passes; the chosen pages
// are then written in ascending order, each CTA at an offset it derives from
// the other CTAs' counts.  Ties on T go to the lowest page indices.
//
// Scoring of bf16 metadata runs on the tensor cores: for 16 pages at a time
// the bound is U = [kmax | kmin] . [max(q,0) ; min(q,0)], a 16 x 2D by
// 2D x 8 product (rows = pages, columns = the group's query heads) whose
// A operand comes straight from 16-byte loads of the min/max rows.  fp32
// metadata (and SLS_FLAG_CUDA_CORES) uses the CUDA-core scorer.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"
#include "mma.cuh"

namespace cg = cooperative_groups;

namespace sls {

constexpr int kCluster = 8;
constexpr int kSelThreads = 256;     // CUDA-core scorer
constexpr int kSelThreadsMma = 128;  // tensor-core scorer
constexpr uint32_t kForcedKey = 0xffffffffu;

int select_pages_cluster() { return kCluster; }
size_t select_pages_smem_limit() { return 200 * 1024; }

struct SelectArgs {
  const void* q;
  const void* kmin;
  const void* kmax;
  const int32_t* ctx_len;
  int32_t* page_idx;
  int k, n_sink, n_local;
  int Hq, Hkv, G, Cap, P, pshift;
};

// Exclusive scan of one int per thread over the CTA; `total` gets the sum.
template <int NT>
__device__ __forceinline__ int block_excl_scan(int v, int* tmp, int& total) {
  constexpr int kSelWarps = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = lane < kSelWarps ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < kSelWarps) tmp[lane] = t;
  }
  __syncthreads();
  const int before = warp > 0 ? tmp[warp - 1] : 0;
  total = tmp[kSelWarps - 1];
  __syncthreads();
  return before + x - v;
}

// Scores of pages [p0, p0 + nloc) of one row into keys[0 .. nloc).
// A page's D channels are spread over L lanes as 16-byte vectors.
template <typename T, int D, int GM>
__device__ __forceinline__ void score_chunk(const SelectArgs& a, int row, int b, int h, int p0,
                                            int nloc, int first_local, uint32_t* keys) {
  constexpr int EPL = Vec16<T>::N;
  constexpr int L = D / EPL;
  constexpr int TPW = 32 / L;
  constexpr int UNR = 4;
  constexpr int kSelWarps = kSelThreads / 32;
  constexpr int STRIDE = kSelWarps * TPW;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / L, sub = lane % L;
  const int G = a.G;
  const bool single = a.P == 1;  // a one-token page: kmin == kmax == the key

  // q split by sign: max(q*lo, q*hi) = max(q,0)*hi + min(q,0)*lo for lo <= hi
  float qp[GM][EPL], qn[GM][EPL];
  {
    const T* qb = static_cast<const T*>(a.q) + ((size_t)b * a.Hq + (size_t)h * G) * D + sub * EPL;
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      float t[EPL];
      if (g < G) load_vec(qb + (size_t)g * D, t);
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const float x = g < G ? t[e] : 0.f;
        qp[g][e] = single ? x : fmaxf(x, 0.f);
        qn[g][e] = single ? 0.f : fminf(x, 0.f);
      }
    }
  }
  const size_t base = ((size_t)row * (size_t)(a.Cap >> a.pshift) + p0) * D + sub * EPL;
  const T* lo = static_cast<const T*>(a.kmin) + base;
  const T* hi = static_cast<const T*>(a.kmax) + base;

  for (int i0 = warp * TPW; i0 < nloc; i0 += STRIDE * UNR) {
    uint4 vl[UNR], vh[UNR];
    int pi[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      pi[u] = i0 + u * STRIDE + grp;
      const bool ok = pi[u] < nloc;
      vl[u] = ok ? ldg_stream(lo + (size_t)pi[u] * D) : make_uint4(0, 0, 0, 0);
      if (!single) vh[u] = ok ? ldg_stream(hi + (size_t)pi[u] * D) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      float fl[EPL], fh[EPL];
      unpack_vec(vl[u], fl);
      if (!single) unpack_vec(vh[u], fh);
      float s[GM];
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        s[g] = 0.f;
        if (g < G) {
          if (single) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) s[g] = fmaf(qp[g][e], fl[e], s[g]);
          } else {
#pragma unroll
            for (int e = 0; e < EPL; ++e) s[g] = fmaf(qp[g][e], fh[e], fmaf(qn[g][e], fl[e], s[g]));
          }
        }
      }
#pragma unroll
      for (int o = L / 2; o > 0; o >>= 1) {
#pragma unroll
        for (int g = 0; g < GM; ++g) s[g] += __shfl_xor_sync(0xffffffffu, s[g], o);
      }
      float best = s[0];
#pragma unroll
      for (int g = 1; g < GM; ++g)
        if (g < G) best = fmaxf(best, s[g]);
      if (sub == 0 && pi[u] < nloc) {
        const int p = p0 + pi[u];
        const bool forced = p < a.n_sink || p >= first_local;
        keys[pi[u]] = forced ? kForcedKey : float_key(best);
      }
    }
  }
}

// Tensor-core scorer (bf16): 16 pages per warp step.  Lane (r, m) loads
// rows r and r+8 of the 16-page tile, chunks 4s+m of kmax and kmin (or of the
// key itself when a page is one token); the group's heads are the 8 columns.
template <int D, bool SINGLE, int NT>
__device__ __forceinline__ void score_chunk_mma(const SelectArgs& a, int row, int b, int h, int p0,
                                                int nloc, int first_local, uint32_t* keys) {
  constexpr int NS = D / 32;
  constexpr int NW = NT / 32;
  constexpr int UT = SINGLE ? 4 : 2;  // tiles in flight per warp
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, m = lane & 3;
  const int G = a.G;

  uint32_t bp[NS][4], bn[NS][4];
  {
    const bf16* qp = static_cast<const bf16*>(a.q) + ((size_t)b * a.Hq + (size_t)h * G + r) * D;
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      const uint4 c = r < G ? ldg_stream(qp + (4 * s + m) * 8) : make_uint4(0, 0, 0, 0);
      const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        bp[s][i] = SINGLE ? w[i] : bf16x2_relu(w[i]);
        bn[s][i] = SINGLE ? 0u : bf16x2_negpart(w[i]);
      }
    }
  }
  const size_t base = ((size_t)row * (size_t)(a.Cap >> a.pshift) + p0) * D;
  const bf16* lo = static_cast<const bf16*>(a.kmin) + base;
  const bf16* hi = static_cast<const bf16*>(a.kmax) + base;
  const bool h0ok = 2 * m < G, h1ok = 2 * m + 1 < G;
  const int ntiles = (nloc + 15) >> 4;

  for (int t0 = warp; t0 < ntiles; t0 += NW * UT) {
    uint4 xh[UT][2][NS], xl[UT][2][NS];
#pragma unroll
    for (int u = 0; u < UT; ++u) {
      const int pr = ((t0 + u * NW) << 4) + r;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int p = pr + 8 * half;
        const bool ok = p < nloc;
#pragma unroll
        for (int s = 0; s < NS; ++s) {
          const size_t off = (size_t)p * D + (4 * s + m) * 8;
          xh[u][half][s] = ok ? ldg_stream((SINGLE ? lo : hi) + off) : make_uint4(0, 0, 0, 0);
          if (!SINGLE) xl[u][half][s] = ok ? ldg_stream(lo + off) : make_uint4(0, 0, 0, 0);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < UT; ++u) {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        mma_bf16(c, xh[u][0][s].x, xh[u][1][s].x, xh[u][0][s].y, xh[u][1][s].y, bp[s][0], bp[s][1]);
        mma_bf16(c, xh[u][0][s].z, xh[u][1][s].z, xh[u][0][s].w, xh[u][1][s].w, bp[s][2], bp[s][3]);
        if (!SINGLE) {
          mma_bf16(c, xl[u][0][s].x, xl[u][1][s].x, xl[u][0][s].y, xl[u][1][s].y, bn[s][0], bn[s][1]);
          mma_bf16(c, xl[u][0][s].z, xl[u][1][s].z, xl[u][0][s].w, xl[u][1][s].w, bn[s][2], bn[s][3]);
        }
      }
      // page score = max over the group's heads (columns 2m, 2m+1 here)
      float v0 = kNegInf, v1 = kNegInf;
      if (h0ok) { v0 = c[0]; v1 = c[2]; }
      if (h1ok) { v0 = fmaxf(v0, c[1]); v1 = fmaxf(v1, c[3]); }
      v0 = fmaxf(v0, __shfl_xor_sync(0xffffffffu, v0, 1));
      v0 = fmaxf(v0, __shfl_xor_sync(0xffffffffu, v0, 2));
      v1 = fmaxf(v1, __shfl_xor_sync(0xffffffffu, v1, 1));
      v1 = fmaxf(v1, __shfl_xor_sync(0xffffffffu, v1, 2));
      if (m == 0) {
        const int pr = ((t0 + u * NW) << 4) + r;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int i = pr + 8 * half;
          if (i < nloc) {
            const int p = p0 + i;
            const bool forced = p < a.n_sink || p >= first_local;
            keys[i] = forced ? kForcedKey : float_key(half ? v1 : v0);
          }
        }
      }
    }
  }
}

struct TopkShared {
  uint32_t hist[2][256];
  int scan_tmp[32];
  uint32_t digit;
  int rem;
  int cnt[2];
};

// The cluster's k largest keys (ties to the lower index), written ascending
// by page index to out[0 .. k).  keys[0 .. nloc) hold pages p0 + i.
template <int NT>
__device__ __forceinline__ void cluster_topk(cg::cluster_group& cl, const uint32_t* keys, int nloc,
                                             int rank, int k, int p0, int32_t* out, TopkShared& sh) {
  constexpr int BPT = 256 / NT;  // histogram bins per thread
  const int tid = threadIdx.x, lane = tid & 31;
  uint32_t prefix = 0, mask = 0;
  int rem = k;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    uint32_t* hb = sh.hist[pass & 1];
#pragma unroll
    for (int i = 0; i < BPT; ++i) hb[tid * BPT + i] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < nloc; i0 += NT) {
      const int i = i0 + tid;
      const uint32_t kk = i < nloc ? keys[i] : 0u;
      const bool in = i < nloc && (kk & mask) == prefix;
      const unsigned act = __ballot_sync(0xffffffffu, in);
      if (in) {
        const unsigned dig = (kk >> shift) & 255u;
        const unsigned peers = __match_any_sync(act, dig);
        if (lane == __ffs(peers) - 1) atomicAdd(&hb[dig], (uint32_t)__popc(peers));
      }
    }
    cl.sync();
    // thread tid owns bins 255 - tid*BPT - i, i < BPT (descending)
    uint32_t tot[BPT];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      const int bin = 255 - tid * BPT - i;
      tot[i] = 0;
#pragma unroll
      for (int q = 0; q < kCluster; ++q) tot[i] += cl.map_shared_rank(hb, q)[bin];
      sum += (int)tot[i];
    }
    int total;
    int above = block_excl_scan<NT>(sum, sh.scan_tmp, total);  // keys with a larger digit
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      const int incl = above + (int)tot[i];
      if (incl >= rem && above < rem) {
        sh.digit = (uint32_t)(255 - tid * BPT - i);
        sh.rem = rem - above;
      }
      above = incl;
    }
    __syncthreads();
    prefix |= sh.digit << shift;
    mask |= 255u << shift;
    rem = sh.rem;
  }
  const uint32_t Tk = prefix;

  const int per_t = (nloc + NT - 1) / NT;
  const int i0 = min(tid * per_t, nloc), i1 = min(i0 + per_t, nloc);
  int gt = 0, eq = 0;
  for (int i = i0; i < i1; ++i) {
    const uint32_t kk = keys[i];
    gt += kk > Tk;
    eq += kk == Tk;
  }
  int gt_tot, eq_tot;
  block_excl_scan<NT>(gt, sh.scan_tmp, gt_tot);
  const int eq_excl = block_excl_scan<NT>(eq, sh.scan_tmp, eq_tot);
  if (tid == 0) {
    sh.cnt[0] = gt_tot;
    sh.cnt[1] = eq_tot;
  }
  cl.sync();
  int out_off = 0, take = 0, eq_seen = 0;
  for (int q = 0; q < kCluster; ++q) {
    const int* rc = cl.map_shared_rank(sh.cnt, q);
    const int g_r = rc[0], e_r = rc[1];
    const int t_r = min(max(rem - eq_seen, 0), e_r);
    if (q < rank) out_off += g_r + t_r;
    if (q == rank) take = t_r;
    eq_seen += e_r;
  }
  int nsel = 0, run = eq_excl;
  for (int i = i0; i < i1; ++i) {
    const uint32_t kk = keys[i];
    if (kk > Tk) ++nsel;
    else if (kk == Tk) nsel += (run++ < take);
  }
  int sel_tot;
  int pos = out_off + block_excl_scan<NT>(nsel, sh.scan_tmp, sel_tot);
  run = eq_excl;
  for (int i = i0; i < i1; ++i) {
    const uint32_t kk = keys[i];
    bool f = kk > Tk;
    if (kk == Tk) f = run++ < take;
    if (f && pos < k) out[pos++] = p0 + i;
  }
  cl.sync();  // peers may still read sh.cnt
}

// MODE 0: CUDA-core scorer (any dtype); 1: tensor-core scorer (bf16, P > 1);
// 2: tensor-core scorer of one-token pages (bf16, P == 1).
template <typename T, int D, int GM, int MODE>
__global__ void __cluster_dims__(kCluster, 1, 1)
__launch_bounds__(MODE == 0 ? kSelThreads : kSelThreadsMma)
select_pages_kernel(const SelectArgs a) {
  constexpr int NT = MODE == 0 ? kSelThreads : kSelThreadsMma;
  extern __shared__ uint32_t keys[];
  __shared__ TopkShared sh;

  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank();
  const int tid = threadIdx.x;
  const int row = blockIdx.x / kCluster;
  const int b = row / a.Hkv, h = row % a.Hkv;
  const int N = clamp_len(a.ctx_len[b], a.Cap);
  const int NP = (N + a.P - 1) >> a.pshift;
  int32_t* out = a.page_idx + (size_t)row * a.k;

  if (NP <= a.k) {  // the budget covers every page: no ranking needed
    for (int i = rank * NT + tid; i < a.k; i += NT * kCluster) out[i] = i < NP ? i : -1;
    return;
  }
  const int chunk = (NP + kCluster - 1) / kCluster;
  const int p0 = rank * chunk;
  const int nloc = max(min(chunk, NP - p0), 0);
  const int first_local = a.n_local > 0 ? (max(N - a.n_local, 0) >> a.pshift) : NP;
  if constexpr (MODE == 0) {
    score_chunk<T, D, GM>(a, row, b, h, p0, nloc, first_local, keys);
  } else {
    score_chunk_mma<D, MODE == 2, NT>(a, row, b, h, p0, nloc, first_local, keys);
  }
  __syncthreads();
  cluster_topk<NT>(cl, keys, nloc, rank, a.k, p0, out, sh);
}

template <typename T, int D, int GM, int MODE>
static cudaError_t select_launch(const SelectArgs& a, int rows, size_t smem, cudaStream_t st) {
  auto kern = select_pages_kernel<T, D, GM, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<rows * kCluster, MODE == 0 ? kSelThreads : kSelThreadsMma, smem, st>>>(a);
  return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t select_g(const SelectArgs& a, int rows, size_t smem, cudaStream_t st) {
  if (a.G <= 1) return select_launch<T, D, 1, 0>(a, rows, smem, st);
  if (a.G <= 2) return select_launch<T, D, 2, 0>(a, rows, smem, st);
  if (a.G <= 4) return select_launch<T, D, 4, 0>(a, rows, smem, st);
  return select_launch<T, D, 8, 0>(a, rows, smem, st);
}

template <int D>
static cudaError_t select_mma(const SelectArgs& a, int rows, size_t smem, cudaStream_t st) {
  if (a.P == 1) return select_launch<bf16, D, 8, 2>(a, rows, smem, st);
  return select_launch<bf16, D, 8, 1>(a, rows, smem, st);
}

cudaError_t launch_select_pages(const Shape& s, const void* q, const void* kmin,
                                const void* kmax, const int32_t* ctx_len, int k,
                                int n_sink_pages, int n_local_tokens, int32_t* page_idx,
                                cudaStream_t st) {
  SelectArgs a;
  a.q = q; a.kmin = kmin; a.kmax = kmax; a.ctx_len = ctx_len; a.page_idx = page_idx;
  a.k = k; a.n_sink = n_sink_pages; a.n_local = n_local_tokens;
  a.Hq = s.Hq; a.Hkv = s.Hkv; a.G = s.G; a.Cap = s.Cap; a.P = s.P; a.pshift = s.pshift;
  const int npcap = s.Cap >> s.pshift;
  const size_t chunk = (size_t)(npcap + kCluster - 1) / kCluster;
  const size_t smem = chunk * sizeof(uint32_t) < 16 ? 16 : chunk * sizeof(uint32_t);
  const int rows = s.B * s.Hkv;
  if (s.dtype == 1 && !(s.flags & 1))
    return s.D == 64 ? select_mma<64>(a, rows, smem, st) : select_mma<128>(a, rows, smem, st);
  if (s.dtype == 0)
    return s.D == 64 ? select_g<float, 64>(a, rows, smem, st) : select_g<float, 128>(a, rows, smem, st);
  return s.D == 64 ? select_g<bf16, 64>(a, rows, smem, st) : select_g<bf16, 128>(a, rows, smem, st);
}

}  // namespace sls
