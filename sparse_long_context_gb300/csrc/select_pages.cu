// Quest-style page selection ("Don't read the haystack", Part two: bound
// every page's score by sum_c max(q_c*kmin_c, q_c*kmax_c), keep the top k
// plus the sink page and the last local pages).  Two kernels:
//
// score   streams the page min/max metadata once and writes one
//         order-preserving 32-bit key per page to a workspace.  bf16
//         metadata is scored on the tensor cores: for 16 pages at a time
//         U = [kmax | kmin] . [max(q,0) ; min(q,0)], a 16 x 2D by 2D x 8
//         product (rows = pages, columns = the GQA group's query heads) whose
//         A operand comes straight from 16-byte loads of the min/max rows;
//         fp32 metadata (and SLS_FLAG_CUDA_CORES) uses a CUDA-core scorer.
//         The grid is one wave of CTAs, each a contiguous run of one row.
// topk    one CTA per row (or a cluster of CTAs for rows longer than one
//         CTA's shared memory) loads the row's keys and runs an MSB-first
//         radix select (4 passes of 8-bit digits; cluster histograms are
//         summed through distributed shared memory).  The k-th key T and the
//         count of T-valued keys still to take come out of the passes; the
//         chosen pages are written in ascending order.  Ties on T go to the
//         lowest page indices.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"
#include "mma.cuh"

namespace cg = cooperative_groups;

namespace sls {

constexpr int kSelThreads = 256;     // CUDA-core scorer
constexpr int kSelThreadsMma = 128;  // tensor-core scorer
constexpr int kTopkThreads = 512;
constexpr int kTopkMaxKeys = 32768;  // keys per top-k CTA (128 KB of shared memory)
constexpr int kTopkMaxCluster = 8;
constexpr uint32_t kForcedKey = 0xffffffffu;

int select_pages_cluster() { return kTopkMaxCluster; }
size_t select_pages_smem_limit() { return (size_t)kTopkMaxKeys * 4; }

struct SelectArgs {
  const void* q;
  const void* kmin;
  const void* kmax;
  const int32_t* ctx_len;
  int32_t* page_idx;
  uint32_t* keys;  // workspace [rows, Cap/P]
  int k, n_sink, n_local;
  int Hq, Hkv, G, Cap, P, pshift, npcap;
  int chunk;       // pages per scoring CTA (multiple of 16)
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

// The k largest keys of a row (ties to the lower index), written ascending
// by page index to out[0 .. k).  keys[0 .. nloc) hold pages p0 + i; with
// CL > 1 the row is spread over the CTAs of a cluster.
template <int NT, int CL>
__device__ __forceinline__ void row_topk(const uint32_t* keys, int nloc, int rank, int k, int p0,
                                         int32_t* out, TopkShared& sh) {
  constexpr int BPT = NT >= 256 ? 1 : 256 / NT;  // histogram bins per owner thread
  const int tid = threadIdx.x, lane = tid & 31;
  const bool owner = tid * BPT < 256;
  auto sync_all = [] {
    if constexpr (CL > 1) cg::this_cluster().sync(); else __syncthreads();
  };
  uint32_t prefix = 0, mask = 0;
  int rem = k;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    uint32_t* hb = sh.hist[pass & 1];
    if (owner) {
#pragma unroll
      for (int i = 0; i < BPT; ++i) hb[tid * BPT + i] = 0;
    }
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
    sync_all();
    // owner thread tid holds bins 255 - tid*BPT - i, i < BPT (descending)
    uint32_t tot[BPT];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      tot[i] = 0;
      if (owner) {
        const int bin = 255 - tid * BPT - i;
        if constexpr (CL > 1) {
          cg::cluster_group cl = cg::this_cluster();
#pragma unroll
          for (int q = 0; q < CL; ++q) tot[i] += cl.map_shared_rank(hb, q)[bin];
        } else {
          tot[i] = hb[bin];
        }
      }
      sum += (int)tot[i];
    }
    int total;
    int above = block_excl_scan<NT>(sum, sh.scan_tmp, total);  // keys with a larger digit
    if (owner) {
#pragma unroll
      for (int i = 0; i < BPT; ++i) {
        const int incl = above + (int)tot[i];
        if (incl >= rem && above < rem) {
          sh.digit = (uint32_t)(255 - tid * BPT - i);
          sh.rem = rem - above;
        }
        above = incl;
      }
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
  int out_off = 0, take = min(rem, eq_tot);
  if constexpr (CL > 1) {
    if (tid == 0) {
      sh.cnt[0] = gt_tot;
      sh.cnt[1] = eq_tot;
    }
    cg::cluster_group cl = cg::this_cluster();
    cl.sync();
    int eq_seen = 0;
    for (int q = 0; q < CL; ++q) {
      const int* rc = cl.map_shared_rank(sh.cnt, q);
      const int g_r = rc[0], e_r = rc[1];
      const int t_r = min(max(rem - eq_seen, 0), e_r);
      if (q < rank) out_off += g_r + t_r;
      if (q == rank) take = t_r;
      eq_seen += e_r;
    }
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
  if constexpr (CL > 1) cg::this_cluster().sync();  // peers may still read sh.cnt
}

// Fast path for a row held by one CTA (keys[0 .. n) with n > k): one
// histogram of the keys' top 16 bits over a window of kWin values below the
// largest non-forced key locates T's 16-bit bin; the few keys in that bin
// are ranked exactly against each other; one pair scan then writes the
// chosen pages in ascending order.  Returns false (having written nothing)
// when T lies below the window or its bin holds more than kCand keys; the
// caller then runs the general radix select.
constexpr int kWin = 2048;
constexpr int kCand = 1024;

struct TopkFastShared {
  uint32_t hist[kWin];
  uint32_t cand[kCand];
  int scan_tmp[32];
  uint32_t red[32];
  int ncand;
  int bin;
  int rem;
  int take;
  uint32_t T;
  int ok;
};

template <int NT>
__device__ __forceinline__ void block_pair_excl_scan(int a, int b, int* tmp, int& ea, int& eb) {
  // scans two counts packed in one int: b in the low 16 bits, a above; the
  // callers' totals stay below 2^15 (a) and 2^16 (b), so nothing carries
  int tot;
  const int e = block_excl_scan<NT>((a << 16) | b, tmp, tot);
  ea = e >> 16;
  eb = e & 0xffff;
}

template <int NT>
__device__ __forceinline__ bool row_topk_fast(const uint32_t* keys, int n, int k, int32_t* out,
                                              TopkFastShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NWp = NT / 32;
  // 1. largest non-forced top-16 value and the number of forced keys
  uint32_t mx = 0;
  int nf = 0;
  for (int i = tid; i < n; i += NT) {
    const uint32_t kk = keys[i];
    if (kk == kForcedKey) ++nf;
    else mx = max(mx, kk >> 16);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    nf += __shfl_xor_sync(0xffffffffu, nf, o);
  }
  if (lane == 0) sh.red[warp] = mx | ((uint32_t)0);
  if (lane == 0) sh.scan_tmp[warp] = nf;
  for (int i = tid; i < kWin; i += NT) sh.hist[i] = 0;
  if (tid == 0) sh.ncand = 0;
  __syncthreads();
  uint32_t top = 0;
  int nforced = 0;
#pragma unroll
  for (int w = 0; w < NWp; ++w) {
    top = max(top, sh.red[w]);
    nforced += sh.scan_tmp[w];
  }
  __syncthreads();
  const int need = k - nforced;  // non-forced keys to take (>= 0 by validation)
  if (need <= 0) {
    if (tid == 0) {
      sh.T = kForcedKey;
      sh.take = k;
    }
  } else {
    // 2. window histogram: bin j counts keys whose top 16 bits equal top - j
    for (int i = tid; i < n; i += NT) {
      const uint32_t kk = keys[i];
      if (kk == kForcedKey) continue;
      const uint32_t j = top - (kk >> 16);
      if (j < (uint32_t)kWin) atomicAdd(&sh.hist[j], 1u);
    }
    __syncthreads();
    // 3. the bin holding the need-th largest (bins in increasing j)
    constexpr int BPT = kWin / NT;
    int c[BPT], sum = 0;
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      c[i] = (int)sh.hist[tid * BPT + i];
      sum += c[i];
    }
    int total;
    int above = block_excl_scan<NT>(sum, sh.scan_tmp, total);
    if (tid == 0) sh.ok = total >= need;
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      if (above < need && above + c[i] >= need) {
        sh.bin = tid * BPT + i;
        sh.rem = need - above;
      }
      above += c[i];
    }
    __syncthreads();
    if (!sh.ok) return false;
    // 4. collect the keys of that bin
    const uint32_t t16 = top - (uint32_t)sh.bin;
    for (int i = tid; i < n; i += NT) {
      const uint32_t kk = keys[i];
      if (kk != kForcedKey && (kk >> 16) == t16) {
        const int slot = atomicAdd(&sh.ncand, 1);
        if (slot < kCand) sh.cand[slot] = kk;
      }
    }
    __syncthreads();
    const int m = sh.ncand;
    if (m > kCand) return false;  // uniform: every thread read the same count
    // 5. exact rank inside the bin: T has fewer than rem larger keys and at
    //    least rem keys >= it
    const int rem = sh.rem;
    for (int i = tid; i < m; i += NT) {
      const uint32_t v = sh.cand[i];
      int gt = 0, ge = 0;
      for (int j = 0; j < m; ++j) {
        gt += sh.cand[j] > v;
        ge += sh.cand[j] >= v;
      }
      if (gt < rem && ge >= rem) {
        sh.T = v;            // every writer writes the same value
        sh.take = rem - gt;  // T-valued keys to take (same for all writers)
      }
    }
  }
  __syncthreads();
  const uint32_t T = sh.T;
  const int take = sh.take;
  // 6. ascending output: position = (#keys > T before) + min(#T-keys before, take)
  const int per_t = (n + NT - 1) / NT;
  const int i0 = min(tid * per_t, n), i1 = min(i0 + per_t, n);
  int gt = 0, eq = 0;
  for (int i = i0; i < i1; ++i) {
    const uint32_t kk = keys[i];
    gt += kk > T;
    eq += kk == T;
  }
  int G, E;
  block_pair_excl_scan<NT>(gt, eq, sh.scan_tmp, G, E);
  for (int i = i0; i < i1; ++i) {
    const uint32_t kk = keys[i];
    if (kk > T) {
      const int pos = G + min(E, take);
      if (pos < k) out[pos] = i;
      ++G;
    } else if (kk == T) {
      if (E < take && G + E < k) out[G + E] = i;
      ++E;
    }
  }
  return true;
}

// ---------------------------------------------------------------- kernels

// MODE 0: CUDA-core scorer (any dtype); 1: tensor-core scorer (bf16, P > 1);
// 2: tensor-core scorer of one-token pages (bf16, P == 1).
// Grid (CTAs per row, rows); CTA c scores pages [c*chunk, (c+1)*chunk).
template <typename T, int D, int GM, int MODE>
__global__ void __launch_bounds__(MODE == 0 ? kSelThreads : kSelThreadsMma)
quest_score_kernel(const SelectArgs a) {
  pdl_wait_then_release();
  constexpr int NT = MODE == 0 ? kSelThreads : kSelThreadsMma;
  const int row = blockIdx.y;
  const int b = row / a.Hkv, h = row % a.Hkv;
  const int N = clamp_len(a.ctx_len[b], a.Cap);
  const int NP = (N + a.P - 1) >> a.pshift;
  if (NP <= a.k) return;  // the top-k kernel lists every page
  const int p0 = blockIdx.x * a.chunk;
  const int nloc = min(a.chunk, NP - p0);
  if (nloc <= 0) return;
  const int first_local = a.n_local > 0 ? (max(N - a.n_local, 0) >> a.pshift) : NP;
  uint32_t* keys = a.keys + (size_t)row * a.npcap + p0;
  if constexpr (MODE == 0) {
    score_chunk<T, D, GM>(a, row, b, h, p0, nloc, first_local, keys);
  } else {
    score_chunk_mma<D, MODE == 2, NT>(a, row, b, h, p0, nloc, first_local, keys);
  }
}

template <int CL>
__global__ void __launch_bounds__(kTopkThreads)
topk_kernel(const SelectArgs a) {
  pdl_wait();  // released at exit: the attend CTAs queued behind it spread over every SM
  extern __shared__ uint32_t skeys[];
  __shared__ union {
    TopkShared radix;
    TopkFastShared fast;
  } sh;
  const int rank = CL > 1 ? (int)cg::this_cluster().block_rank() : 0;
  const int row = blockIdx.x / CL;
  const int b = row / a.Hkv;
  const int N = clamp_len(a.ctx_len[b], a.Cap);
  const int NP = (N + a.P - 1) >> a.pshift;
  int32_t* out = a.page_idx + (size_t)row * a.k;
  if (NP <= a.k) {  // the budget covers every page: no ranking needed
    for (int i = rank * kTopkThreads + threadIdx.x; i < a.k; i += kTopkThreads * CL) out[i] = i < NP ? i : -1;
    return;
  }
  const int chunk = (NP + CL - 1) / CL;
  const int p0 = rank * chunk;
  const int nloc = max(min(chunk, NP - p0), 0);
  const uint32_t* src = a.keys + (size_t)row * a.npcap + p0;
  for (int i = threadIdx.x; i < nloc; i += kTopkThreads) skeys[i] = src[i];
  __syncthreads();
  if constexpr (CL == 1) {
    if (row_topk_fast<kTopkThreads>(skeys, nloc, a.k, out, sh.fast)) return;
    __syncthreads();
  }
  row_topk<kTopkThreads, CL>(skeys, nloc, rank, a.k, p0, out, sh.radix);
}

// Rows of at most NT*KPT pages: one CTA of NT threads per row, each thread
// holding KPT consecutive keys in registers (thread t: pages t*KPT ..).
// Same algorithm as row_topk_fast (window histogram over the top 16 bits,
// exact rank inside T's bin, ascending output), but every pass is a sweep
// over registers and every scan costs two barriers.  Rows whose threshold
// leaves the window, or whose bin is too full, fall back to the radix
// select over the keys written to shared memory.
constexpr int kRegTopkThreads = 1024;
constexpr int kRegTopkKeys = 8;  // keys per thread

template <int NT>
__device__ __forceinline__ int scan2(int v, int* tmp, int& total) {
  // exclusive scan of one int per thread, two barriers (NT/32 <= 32 warps)
  constexpr int NWp = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  int t = lane < NWp ? tmp[lane] : 0;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, t, o);
    if (lane >= o) t += y;
  }
  const int before = warp > 0 ? __shfl_sync(0xffffffffu, t, warp - 1) : 0;
  total = __shfl_sync(0xffffffffu, t, NWp - 1);
  __syncthreads();  // tmp may be reused right after
  return before + x - v;
}

template <int NT, int KPT>
__global__ void __launch_bounds__(NT)
topk_reg_kernel(const SelectArgs a) {
  pdl_wait();  // released at exit: the attend CTAs queued behind it spread over every SM
  constexpr int NWp = NT / 32;
  constexpr int BPT = kWin / NT;  // window bins per thread
  __shared__ uint32_t hist[kWin];
  __shared__ uint32_t cand[kCand];
  __shared__ int tmp[32];
  __shared__ uint32_t red_max[32];
  __shared__ int red_nf[32];
  __shared__ int s_bin, s_rem, s_take, s_ncand;
  __shared__ uint32_t s_T;
  extern __shared__ uint32_t skeys[];  // only for the fallback

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;
  const int b = row / a.Hkv;
  const int N = clamp_len(a.ctx_len[b], a.Cap);
  const int n = (N + a.P - 1) >> a.pshift;
  const int k = a.k;
  int32_t* out = a.page_idx + (size_t)row * k;
  if (n <= k) {
    for (int i = tid; i < k; i += NT) out[i] = i < n ? i : -1;
    return;
  }
  const uint32_t* src = a.keys + (size_t)row * a.npcap;
  // 0 sorts below every real key (the key of -inf is 0x007fffff), so it
  // pads the slots past n without taking part in any count
  uint32_t kk[KPT];
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const int i = tid * KPT + j;
    kk[j] = i < n ? __ldcg(src + i) : 0u;
  }
  // 1. largest non-forced top-16 value, forced count; clear the window
  uint32_t mx = 0;
  int nf = 0;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    if (kk[j] == kForcedKey) ++nf;
    else mx = max(mx, kk[j] >> 16);
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  nf = __reduce_add_sync(0xffffffffu, nf);
  if (lane == 0) {
    red_max[warp] = mx;
    red_nf[warp] = nf;
  }
#pragma unroll
  for (int i = 0; i < BPT; ++i) hist[tid * BPT + i] = 0;
  if (tid == 0) s_ncand = 0;
  __syncthreads();
  const uint32_t top = __reduce_max_sync(0xffffffffu, lane < NWp ? red_max[lane] : 0u);
  const int nforced = __reduce_add_sync(0xffffffffu, lane < NWp ? red_nf[lane] : 0);
  const int need = k - nforced;
  bool fast = true;
  uint32_t T = kForcedKey;
  int take = k;
  if (need > 0) {
    // 2. window histogram: bin j counts non-forced keys whose top 16 bits are top - j
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      if (kk[j] == kForcedKey || kk[j] == 0u) continue;
      const uint32_t d = top - (kk[j] >> 16);
      if (d < (uint32_t)kWin) atomicAdd(&hist[d], 1u);
    }
    __syncthreads();
    // 3. the bin of the need-th largest (bins by increasing j)
    int c[BPT], sum = 0;
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      c[i] = (int)hist[tid * BPT + i];
      sum += c[i];
    }
    int total;
    int above = scan2<NT>(sum, tmp, total);
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      if (above < need && above + c[i] >= need) {
        s_bin = tid * BPT + i;
        s_rem = need - above;
      }
      above += c[i];
    }
    __syncthreads();
    fast = total >= need;
    if (fast) {
      // 4. the keys of that bin
      const uint32_t t16 = top - (uint32_t)s_bin;
#pragma unroll
      for (int j = 0; j < KPT; ++j) {  // one shared-memory atomic per warp and key slot
        const bool in = kk[j] != kForcedKey && kk[j] != 0u && (kk[j] >> 16) == t16;
        const unsigned bal = __ballot_sync(0xffffffffu, in);
        if (bal == 0u) continue;
        int base = 0;
        if (lane == __ffs(bal) - 1) base = atomicAdd(&s_ncand, __popc(bal));
        base = __shfl_sync(0xffffffffu, base, __ffs(bal) - 1);
        const int slot = base + __popc(bal & ((1u << lane) - 1u));
        if (in && slot < kCand) cand[slot] = kk[j];
      }
      __syncthreads();
      const int m = s_ncand;
      fast = m <= kCand;
      if (fast) {
        // 5. exact rank inside the bin: 8 threads per candidate
        const int rem = s_rem;
        const int sub = tid & 7;
        for (int i0 = 0; i0 < m; i0 += NT / 8) {
          const int i = i0 + (tid >> 3);
          const uint32_t v = i < m ? cand[i] : 0u;
          int gt = 0, ge = 0;
          for (int q = sub; q < m; q += 8) {
            const uint32_t w = cand[q];
            gt += w > v;
            ge += w >= v;
          }
#pragma unroll
          for (int o = 1; o < 8; o <<= 1) {
            gt += __shfl_xor_sync(0xffffffffu, gt, o);
            ge += __shfl_xor_sync(0xffffffffu, ge, o);
          }
          if (i < m && sub == 0 && gt < rem && ge >= rem) {
            s_T = v;
            s_take = rem - gt;
          }
        }
        __syncthreads();
        T = s_T;
        take = s_take;
      }
    }
  }
  if (!fast) {  // uniform: every thread read the same shared values
    for (int j = 0; j < KPT; ++j) {
      const int i = tid * KPT + j;
      if (i < n) skeys[i] = kk[j];
    }
    __syncthreads();
    row_topk<NT, 1>(skeys, n, 0, k, 0, out, *reinterpret_cast<TopkShared*>(hist));
    return;
  }
  // 6. ascending output: position = (#keys > T before) + min(#T-keys before, take)
  int gt = 0, eq = 0;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    gt += kk[j] > T;
    eq += kk[j] == T;
  }
  int tot;
  const int e = scan2<NT>((gt << 16) | eq, tmp, tot);  // both totals < 2^15
  int G = e >> 16, E = e & 0xffff;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const int i = tid * KPT + j;
    if (kk[j] > T) {
      const int pos = G + min(E, take);
      if (pos < k) out[pos] = i;
      ++G;
    } else if (kk[j] == T) {
      if (E < take && G + E < k) out[G + E] = i;
      ++E;
    }
  }
}

// ---------------------------------------------------------------- launches

template <typename T, int D, int GM, int MODE>
static cudaError_t score_launch(const SelectArgs& a, int rows, cudaStream_t st) {
  auto kern = quest_score_kernel<T, D, GM, MODE>;
  constexpr int NT = MODE == 0 ? kSelThreads : kSelThreadsMma;
  static int per_sm = 0;  // resident CTAs per SM of this kernel (same on every GB300)
  if (per_sm == 0) cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, 0);
  SelectArgs b = a;
  const int slots = max(1, sm_count() * max(per_sm, 1));
  const int cpr = max(1, slots / rows);  // at most one wave over all rows
  b.chunk = max(16, ((a.npcap + cpr - 1) / cpr + 15) / 16 * 16);
  dim3 grid((a.npcap + b.chunk - 1) / b.chunk, rows);
  cudaError_t e = launch_pdl(kern, grid, dim3(NT), 0, st, b);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

static cudaError_t topk_launch(const SelectArgs& a, int rows, cudaStream_t st) {
  if (a.npcap <= kRegTopkThreads * kRegTopkKeys) {
    constexpr int NT = kRegTopkThreads, KPT = kRegTopkKeys;
    const size_t smem = (size_t)a.npcap * sizeof(uint32_t);  // fallback keys
    cudaError_t e = cudaFuncSetAttribute(topk_reg_kernel<NT, KPT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(topk_reg_kernel<NT, KPT>, dim3(rows), dim3(NT), smem, st, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  int cl = 1;
  while (cl < kTopkMaxCluster && (a.npcap + cl - 1) / cl > kTopkMaxKeys) cl *= 2;
  const size_t smem = (size_t)((a.npcap + cl - 1) / cl) * sizeof(uint32_t);
  cudaError_t e;
  if (cl == 1) {
    e = cudaFuncSetAttribute(topk_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(topk_kernel<1>, dim3(rows), dim3(kTopkThreads), smem, st, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(rows * cl);
  cfg.blockDim = dim3(kTopkThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  switch (cl) {
    case 2:
      e = cudaFuncSetAttribute(topk_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, topk_kernel<2>, a);
      break;
    case 4:
      e = cudaFuncSetAttribute(topk_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, topk_kernel<4>, a);
      break;
    default:
      e = cudaFuncSetAttribute(topk_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, topk_kernel<8>, a);
      break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t score_g(const SelectArgs& a, int rows, cudaStream_t st) {
  if (a.G <= 1) return score_launch<T, D, 1, 0>(a, rows, st);
  if (a.G <= 2) return score_launch<T, D, 2, 0>(a, rows, st);
  if (a.G <= 4) return score_launch<T, D, 4, 0>(a, rows, st);
  return score_launch<T, D, 8, 0>(a, rows, st);
}

template <int D>
static cudaError_t score_mma(const SelectArgs& a, int rows, cudaStream_t st) {
  if (a.P == 1) return score_launch<bf16, D, 8, 2>(a, rows, st);
  return score_launch<bf16, D, 8, 1>(a, rows, st);
}

size_t select_pages_workspace(const Shape& s) {
  const size_t bytes = (size_t)s.B * s.Hkv * (size_t)(s.Cap >> s.pshift) * sizeof(uint32_t);
  return (bytes + 255) & ~(size_t)255;
}

cudaError_t launch_select_pages(const Shape& s, const void* q, const void* kmin,
                                const void* kmax, const int32_t* ctx_len, int k,
                                int n_sink_pages, int n_local_tokens, int32_t* page_idx,
                                void* ws, cudaStream_t st) {
  SelectArgs a;
  a.q = q; a.kmin = kmin; a.kmax = kmax; a.ctx_len = ctx_len; a.page_idx = page_idx;
  a.keys = static_cast<uint32_t*>(ws);
  a.k = k; a.n_sink = n_sink_pages; a.n_local = n_local_tokens;
  a.Hq = s.Hq; a.Hkv = s.Hkv; a.G = s.G; a.Cap = s.Cap; a.P = s.P; a.pshift = s.pshift;
  a.npcap = s.Cap >> s.pshift;
  a.chunk = 0;
  const int rows = s.B * s.Hkv;
  cudaError_t e;
  if (s.dtype == 1 && !(s.flags & 1))
    e = s.D == 64 ? score_mma<64>(a, rows, st) : score_mma<128>(a, rows, st);
  else if (s.dtype == 0)
    e = s.D == 64 ? score_g<float, 64>(a, rows, st) : score_g<float, 128>(a, rows, st);
  else
    e = s.D == 64 ? score_g<bf16, 64>(a, rows, st) : score_g<bf16, 128>(a, rows, st);
  if (e != cudaSuccess) return e;
  return topk_launch(a, rows, st);
}

}  // namespace sls
