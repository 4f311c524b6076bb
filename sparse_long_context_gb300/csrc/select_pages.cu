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
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"

namespace cg = cooperative_groups;

namespace sls {

constexpr int kCluster = 8;
constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
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
__device__ __forceinline__ int block_excl_scan(int v, int* tmp, int& total) {
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

template <typename T, int D, int GM>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kSelThreads)
select_pages_kernel(const SelectArgs a) {
  extern __shared__ uint32_t keys[];
  __shared__ uint32_t hist[2][256];
  __shared__ int scan_tmp[32];
  __shared__ uint32_t s_digit;
  __shared__ int s_rem;
  __shared__ int s_cnt[2];

  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank();
  const int tid = threadIdx.x, lane = tid & 31;
  const int row = blockIdx.x / kCluster;
  const int b = row / a.Hkv, h = row % a.Hkv;
  const int N = clamp_len(a.ctx_len[b], a.Cap);
  const int NP = (N + a.P - 1) >> a.pshift;
  int32_t* out = a.page_idx + (size_t)row * a.k;

  if (NP <= a.k) {  // the budget covers every page: no ranking needed
    for (int i = rank * kSelThreads + tid; i < a.k; i += kSelThreads * kCluster) out[i] = i < NP ? i : -1;
    return;
  }

  const int chunk = (NP + kCluster - 1) / kCluster;
  const int p0 = rank * chunk;
  const int nloc = max(min(chunk, NP - p0), 0);
  const int first_local = a.n_local > 0 ? (max(N - a.n_local, 0) >> a.pshift) : NP;
  score_chunk<T, D, GM>(a, row, b, h, p0, nloc, first_local, keys);
  __syncthreads();

  // radix select of the k-th largest key over the cluster
  uint32_t prefix = 0, mask = 0;
  int rem = a.k;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    uint32_t* hb = hist[pass & 1];
    hb[tid] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < nloc; i0 += kSelThreads) {
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
    const int bin = 255 - tid;  // thread tid scans bins from the top down
    uint32_t tot = 0;
#pragma unroll
    for (int r = 0; r < kCluster; ++r) tot += cl.map_shared_rank(hb, r)[bin];
    int total;
    const int incl = block_excl_scan((int)tot, scan_tmp, total) + (int)tot;  // keys with digit >= bin
    if (incl >= rem && incl - (int)tot < rem) {
      s_digit = (uint32_t)bin;
      s_rem = rem - (incl - (int)tot);
    }
    __syncthreads();
    prefix |= s_digit << shift;
    mask |= 255u << shift;
    rem = s_rem;
  }
  const uint32_t Tk = prefix;

  // counts of this CTA: keys above T and keys equal to T
  const int per_t = (nloc + kSelThreads - 1) / kSelThreads;
  const int i0 = min(tid * per_t, nloc), i1 = min(i0 + per_t, nloc);
  int gt = 0, eq = 0;
  for (int i = i0; i < i1; ++i) {
    const uint32_t kk = keys[i];
    gt += kk > Tk;
    eq += kk == Tk;
  }
  int gt_tot, eq_tot;
  block_excl_scan(gt, scan_tmp, gt_tot);
  const int eq_excl = block_excl_scan(eq, scan_tmp, eq_tot);
  if (tid == 0) {
    s_cnt[0] = gt_tot;
    s_cnt[1] = eq_tot;
  }
  cl.sync();
  int out_off = 0, take = 0, eq_seen = 0;
  for (int r = 0; r < kCluster; ++r) {
    const int* rc = cl.map_shared_rank(s_cnt, r);
    const int g_r = rc[0], e_r = rc[1];
    const int t_r = min(max(rem - eq_seen, 0), e_r);
    if (r < rank) out_off += g_r + t_r;
    if (r == rank) take = t_r;
    eq_seen += e_r;
  }
  // ascending compaction of the chosen pages of this CTA
  int nsel = 0, run = eq_excl;
  for (int i = i0; i < i1; ++i) {
    const uint32_t kk = keys[i];
    if (kk > Tk) ++nsel;
    else if (kk == Tk) nsel += (run++ < take);
  }
  int sel_tot;
  int pos = out_off + block_excl_scan(nsel, scan_tmp, sel_tot);
  run = eq_excl;
  for (int i = i0; i < i1; ++i) {
    const uint32_t kk = keys[i];
    bool f = kk > Tk;
    if (kk == Tk) f = run++ < take;
    if (f && pos < a.k) out[pos++] = p0 + i;
  }
  cl.sync();  // peers may still read s_cnt
}

template <typename T, int D, int GM>
static cudaError_t select_launch(const SelectArgs& a, int rows, size_t smem, cudaStream_t st) {
  auto kern = select_pages_kernel<T, D, GM>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<rows * kCluster, kSelThreads, smem, st>>>(a);
  return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t select_g(const SelectArgs& a, int rows, size_t smem, cudaStream_t st) {
  if (a.G <= 1) return select_launch<T, D, 1>(a, rows, smem, st);
  if (a.G <= 2) return select_launch<T, D, 2>(a, rows, smem, st);
  if (a.G <= 4) return select_launch<T, D, 4>(a, rows, smem, st);
  return select_launch<T, D, 8>(a, rows, smem, st);
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
  if (s.dtype == 0)
    return s.D == 64 ? select_g<float, 64>(a, rows, smem, st) : select_g<float, 128>(a, rows, smem, st);
  return s.D == 64 ? select_g<bf16, 64>(a, rows, smem, st) : select_g<bf16, 128>(a, rows, smem, st);
}

}  // namespace sls
