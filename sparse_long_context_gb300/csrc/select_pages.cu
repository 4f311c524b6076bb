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

#include "common.cuh"
#include "launch.h"
#include "mma.cuh"


namespace sls {

constexpr int kSelThreads = 256;     // CUDA-core scorer
constexpr int kSelThreadsMma = 128;  // tensor-core scorer
constexpr uint32_t kForcedKey = 0xffffffffu;

int select_pages_max_pages() { return 262144; }

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
  // wide rows (more pages than one top-k CTA holds in registers): every
  // scoring CTA also sends its candidates, the keys at or above a threshold
  // of its own, and the top-k CTA ranks only those (all null otherwise)
  uint32_t* cand_key;   // [rows, npcap]: CTA c's candidates from page offset c * chunk
  int32_t* cand_page;   // [rows, npcap]: their pages
  int32_t* cand_count;  // [rows, ncmax]: candidates CTA c sent
  uint32_t* cand_tau;   // [rows, ncmax]: CTA c's threshold (0: it sent every key)
  int ncmax;            // scoring CTAs per row the arrays hold (npcap / 16)
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

// Per-thread range of the keys a scorer wrote (wide rows only): the largest
// and smallest non-forced key and the number of forced keys.
struct KeyRange {
  uint32_t top = 0, bot = 0xffffffffu;
  int nf = 0;
  __device__ __forceinline__ void add(uint32_t key) {
    if (key == kForcedKey) {
      ++nf;
    } else {
      top = max(top, key);
      bot = min(bot, key);
    }
  }
};

// Scores of pages [p0, p0 + nloc) of one row into keys[0 .. nloc).
// A page's D channels are spread over L lanes as 16-byte vectors.
template <typename T, int D, int GM, bool STAGE>
__device__ __forceinline__ void score_chunk(const SelectArgs& a, int row, int b, int h, int p0,
                                            int nloc, int first_local, uint32_t* keys, uint32_t* skeys,
                                            KeyRange& kr) {
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
        const uint32_t key = forced ? kForcedKey : float_key(best);
        keys[pi[u]] = key;
        if constexpr (STAGE) {
          if (skeys) skeys[pi[u]] = key;
          kr.add(key);
        }
      }
    }
  }
}

// Tensor-core scorer (bf16): 16 pages per warp step.  Lane (r, m) loads
// rows r and r+8 of the 16-page tile, chunks 4s+m of kmax and kmin (or of the
// key itself when a page is one token); the group's heads are the 8 columns.
template <int D, bool SINGLE, int NT, bool STAGE>
__device__ __forceinline__ void score_chunk_mma(const SelectArgs& a, int row, int b, int h, int p0,
                                                int nloc, int first_local, uint32_t* keys,
                                                uint32_t* skeys, KeyRange& kr) {
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
            const uint32_t key = forced ? kForcedKey : float_key(half ? v1 : v0);
            keys[i] = key;
            if constexpr (STAGE) {
              if (skeys) skeys[i] = key;
              kr.add(key);
            }
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
};

// The k largest keys of a row (ties to the lower index), written ascending
// by page index to out[0 .. k): an 8-bit radix select in four passes over
// keys[0 .. nloc) (pages p0 + i; shared or global memory), then one scan
// for the positions.
template <int NT>
__device__ __forceinline__ void row_topk(const uint32_t* keys, int nloc, int k, int p0, int32_t* out,
                                         TopkShared& sh) {
  constexpr int BPT = NT >= 256 ? 1 : 256 / NT;  // histogram bins per owner thread
  const int tid = threadIdx.x, lane = tid & 31;
  const bool owner = tid * BPT < 256;
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
    __syncthreads();
    // owner thread tid holds bins 255 - tid*BPT - i, i < BPT (descending)
    uint32_t tot[BPT];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      tot[i] = owner ? hb[255 - tid * BPT - i] : 0u;
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
  const int take = min(rem, eq_tot);
  int nsel = 0, run = eq_excl;
  for (int i = i0; i < i1; ++i) {
    const uint32_t kk = keys[i];
    if (kk > Tk) ++nsel;
    else if (kk == Tk) nsel += (run++ < take);
  }
  int sel_tot;
  int pos = block_excl_scan<NT>(nsel, sh.scan_tmp, sel_tot);
  run = eq_excl;
  for (int i = i0; i < i1; ++i) {
    const uint32_t kk = keys[i];
    bool f = kk > Tk;
    if (kk == Tk) f = run++ < take;
    if (f && pos < k) out[pos++] = p0 + i;
  }
}

// Window histogram constants of the register-resident top-k: kWin bins of
// the keys' top 16 bits below the largest key, at most kCand keys ranked
// exactly in the threshold bin.
constexpr int kWin = 2048;
constexpr int kCand = 1024;

template <int NT>
__device__ __forceinline__ void block_pair_excl_scan(int a, int b, int* tmp, int& ea, int& eb) {
  // scans two counts packed in one int: b in the low 16 bits, a above; the
  // callers' totals stay below 2^15 (a) and 2^16 (b), so nothing carries
  int tot;
  const int e = block_excl_scan<NT>((a << 16) | b, tmp, tot);
  ea = e >> 16;
  eb = e & 0xffff;
}


// ------------------------------------------------------ rank by range bins

// Narrows [lo, hi] to a key range that holds the rem-th largest of the
// non-forced keys keys[0 .. n) lying in [lo, hi]: a histogram of
// (hi - key) >> shift into BINS bins (shift the smallest that fits the
// range), the bin where the count from the top reaches rem, and the same
// again inside that bin while it holds more than `enough` keys and is wider
// than one value.  Order-preserving float keys are far from uniform, so one
// level of bins is often too coarse.  On return rem counts within the final
// [lo, hi] and the result is true; false (uniform) when fewer than rem keys
// lie in the first range.  keys may be in shared or global memory; hist
// holds BINS counters; every thread of the CTA calls it.
struct RankShared {
  int scan_tmp[32];
  int bin, rem, nbin, ok;
};

template <int NT, int BINS>
__device__ __forceinline__ bool narrow_to_rank(const uint32_t* keys, int n, uint32_t& lo, uint32_t& hi, int& rem,
                                               int enough, uint32_t* hist, RankShared& sh) {
  const int tid = threadIdx.x;
  if (tid == 0) sh.ok = hi >= lo;
  __syncthreads();
  while (sh.ok) {  // uniform
    const uint32_t range = hi - lo;
    int shift = 0;
    while ((range >> shift) >= (uint32_t)BINS) ++shift;
    for (int i = tid; i < BINS; i += NT) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += NT) {
      const uint32_t kk = keys[i];
      if (kk != kForcedKey && kk >= lo && kk <= hi) atomicAdd(&hist[(hi - kk) >> shift], 1u);
    }
    __syncthreads();
    constexpr int BPT = BINS / NT;
    int cnt[BPT], sum = 0;
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      cnt[i] = (int)hist[tid * BPT + i];
      sum += cnt[i];
    }
    int total;
    int above = block_excl_scan<NT>(sum, sh.scan_tmp, total);
    if (tid == 0 && total < rem) sh.ok = 0;
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      if (above < rem && above + cnt[i] >= rem) {
        sh.bin = tid * BPT + i;
        sh.rem = rem - above;
        sh.nbin = cnt[i];
      }
      above += cnt[i];
    }
    __syncthreads();
    if (!sh.ok) break;
    // the bin holds the keys in [hi - span, hi - (bin << shift)], clipped to lo
    const uint64_t top_off = (uint64_t)sh.bin << shift;
    const uint64_t span = ((uint64_t)(sh.bin + 1) << shift) - 1;
    const uint32_t nhi = hi - (uint32_t)top_off;
    const uint32_t nlo = span >= (uint64_t)(hi - lo) ? lo : hi - (uint32_t)span;
    const bool done = sh.nbin <= enough || shift == 0;
    rem = sh.rem;
    hi = nhi;
    lo = nlo;
    __syncthreads();  // every thread has read bin, rem and nbin
    if (done) break;
  }
  const bool ok = sh.ok != 0;
  __syncthreads();
  return ok;
}

// ------------------------------------------------------ wide-row candidates

// A scoring CTA of a wide row sends its forced keys and about twice its
// share of the row's top k (want = 2 k nloc / NP + 16 keys): every key whose
// score falls in the top bins of one histogram, linear in the score, between
// the CTA's smallest and largest score, down to the bin where the count from
// the top reaches want.  The bin of a score is monotone in the score, so the
// keys sent are exactly those >= tau, the smallest key sent; no exact local
// rank is needed.  The candidates are written in page order; tau = 0 means
// the CTA sent every key.  The top-k CTA later proves that its result is
// exact: its k-th key T must be >= every CTA's tau, so that no unsent key can
// reach T.  The scorer also writes the CTA's keys to shared memory when its
// chunk holds at most kCandStage pages; otherwise they are read back from
// global memory.
constexpr int kCandBins = 1024;
constexpr int kCandStage = 8192;

struct CandShared {
  uint32_t hist[kCandBins];
  int scan_tmp[32];
  uint32_t red_hi[32], red_lo[32], red_tau[32];
  int red_n[32];
  int bin;
};

// Inverse of float_key.
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

template <int NT>
__device__ __forceinline__ void emit_candidates(const SelectArgs& a, int row, int NP, int c, int p0, int nloc,
                                                const uint32_t* keys, KeyRange kr, CandShared& sh) {
  constexpr int NWp = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // 1. the CTA's key range, from the ranges the scorer's threads kept
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kr.top = max(kr.top, __shfl_xor_sync(0xffffffffu, kr.top, o));
    kr.bot = min(kr.bot, __shfl_xor_sync(0xffffffffu, kr.bot, o));
    kr.nf += __shfl_xor_sync(0xffffffffu, kr.nf, o);
  }
  if (lane == 0) {
    sh.red_hi[warp] = kr.top;
    sh.red_lo[warp] = kr.bot;
    sh.red_n[warp] = kr.nf;
  }
  for (int i = tid; i < kCandBins; i += NT) sh.hist[i] = 0;
  __syncthreads();  // also: this CTA's keys are written
  uint32_t top = 0, bot = 0xffffffffu;
  int nf = 0;
#pragma unroll
  for (int w = 0; w < NWp; ++w) {
    top = max(top, sh.red_hi[w]);
    bot = min(bot, sh.red_lo[w]);
    nf += sh.red_n[w];
  }
  const int nfree = nloc - nf;
  const int want = (int)min((long long)nfree, (2LL * a.k * nloc + NP - 1) / NP + 16);
  const float ftop = key_float(top);
  const float inv = (float)kCandBins / (ftop - key_float(bot));
  const bool cut = want < nfree && inv > 0.f && inv <= 3.0e38f;  // uniform; else every key is sent
  auto bin_of = [&](uint32_t kk) { return min(kCandBins - 1, (int)((ftop - key_float(kk)) * inv)); };
  int b = kCandBins;
  if (cut) {
    // 2. histogram of the scores; bin b is where the count from the top reaches want
#pragma unroll 4
    for (int i = tid; i < nloc; i += NT) {
      const uint32_t kk = keys[i];
      if (kk != kForcedKey) atomicAdd(&sh.hist[bin_of(kk)], 1u);
    }
    __syncthreads();
    constexpr int BPT = kCandBins / NT;
    int cnt[BPT], sum = 0;
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      cnt[i] = (int)sh.hist[tid * BPT + i];
      sum += cnt[i];
    }
    int total;
    int above = block_excl_scan<NT>(sum, sh.scan_tmp, total);
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      if (above < want && above + cnt[i] >= want) sh.bin = tid * BPT + i;
      above += cnt[i];
    }
    __syncthreads();
    b = sh.bin;
  }
  // 3. the keys sent: forced ones and those in bins 0 .. b (all when !cut).
  //    Thread t counts its run [t per, ...) and the smallest key it sends;
  //    the set is upward closed, so it is exactly the keys >= tau
  const int per = (nloc + NT - 1) / NT;
  const int i0 = min(tid * per, nloc), i1 = min(i0 + per, nloc);
  int mine = 0;
  uint32_t mn = 0xffffffffu;
#pragma unroll 4
  for (int i = i0; i < i1; ++i) {
    const uint32_t kk = keys[i];
    if (!cut || kk == kForcedKey || bin_of(kk) <= b) {
      ++mine;
      mn = min(mn, kk);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  if (lane == 0) sh.red_tau[warp] = mn;
  int total;
  int pos = block_excl_scan<NT>(mine, sh.scan_tmp, total);  // its barriers publish red_tau
  uint32_t tau = 0xffffffffu;
#pragma unroll
  for (int w = 0; w < NWp; ++w) tau = min(tau, sh.red_tau[w]);
  if (!cut) tau = 0;
  uint32_t* ck = a.cand_key + (size_t)row * a.npcap + p0;
  int32_t* cp = a.cand_page + (size_t)row * a.npcap + p0;
#pragma unroll 4
  for (int i = i0; i < i1; ++i) {
    const uint32_t kk = keys[i];
    if (kk >= tau) {
      ck[pos] = kk;
      cp[pos] = p0 + i;
      ++pos;
    }
  }
  if (tid == 0) {
    a.cand_count[(size_t)row * a.ncmax + c] = total;
    a.cand_tau[(size_t)row * a.ncmax + c] = tau;
  }
}

// ---------------------------------------------------------------- kernels

// MODE 0: CUDA-core scorer (any dtype); 1: tensor-core scorer (bf16, P > 1);
// 2: tensor-core scorer of one-token pages (bf16, P == 1).
// Grid (CTAs per row, rows); CTA c scores pages [c*chunk, (c+1)*chunk).
// CAND: the row is wide and the CTA also sends its candidates.
template <typename T, int D, int GM, int MODE, bool CAND>
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
  // wide rows with chunks of at most kCandStage pages: the keys also go to
  // shared memory (dynamic size), where the candidate selection reads them
  extern __shared__ uint32_t stage[];
  uint32_t* skeys = (CAND && a.chunk <= kCandStage) ? stage : nullptr;
  KeyRange kr;
  if constexpr (MODE == 0) {
    score_chunk<T, D, GM, CAND>(a, row, b, h, p0, nloc, first_local, keys, skeys, kr);
  } else {
    score_chunk_mma<D, MODE == 2, NT, CAND>(a, row, b, h, p0, nloc, first_local, keys, skeys, kr);
  }
  if constexpr (CAND) {
    __shared__ CandShared csh;
    emit_candidates<NT>(a, row, NP, blockIdx.x, p0, nloc, skeys ? skeys : keys, kr, csh);
  }
}

// Wide rows: one CTA per row ranks the candidates the scoring CTAs sent
// (about 2k keys plus the forced ones, in page order) in shared memory.
// The k-th largest non-forced key T is found among the candidates at or
// above tau_max (the largest threshold any scoring CTA used) by range
// histograms refined until T's bin holds few keys, then an exact rank inside
// that bin.  Every key >= T of the row is then a candidate (T >= tau_c for
// every CTA c), so the result is the row's exact top k.  When fewer than the
// needed keys lie at or above tau_max (one CTA held much more than its share
// of the row's best pages), or the candidates do not fit, the CTA selects
// from all of the row's keys instead (a radix select over the keys in global
// memory), and counts the row.
constexpr int kWideThreads = 1024;
constexpr int kWideCandMax = 16384;  // candidates held in shared memory
constexpr int kWideBins = 2048;
constexpr int kWideRank = 128;       // keys of T's bin ranked exactly

__device__ unsigned long long g_select_rows_all_keys = 0;  // wide rows selected from all keys

struct WideShared {
  uint32_t hist[kWideBins];
  uint32_t bin_keys[kWideRank];
  RankShared rank;
  int scan_tmp[32];
  uint32_t red[32];
  int red_n[32];
  uint32_t tau_max, top, T;
  int n, nforced, take, nbin, ok;
};

template <int NT>
__global__ void __launch_bounds__(NT)
topk_wide_kernel(const SelectArgs a) {
  pdl_wait();  // released at exit: the attend CTAs queued behind it spread over every SM
  constexpr int NWp = NT / 32;
  extern __shared__ uint32_t wdyn[];
  uint32_t* skey = wdyn;                                             // [kWideCandMax]
  int32_t* spage = reinterpret_cast<int32_t*>(wdyn + kWideCandMax);  // [kWideCandMax]
  int* soff = reinterpret_cast<int*>(wdyn + 2 * kWideCandMax);       // [scoring CTAs + 1]
  __shared__ union {
    WideShared w;
    TopkShared radix;
  } sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;
  const int b = row / a.Hkv;
  const int N = clamp_len(a.ctx_len[b], a.Cap);
  const int NP = (N + a.P - 1) >> a.pshift;
  int32_t* out = a.page_idx + (size_t)row * a.k;
  if (NP <= a.k) {  // the budget covers every page: no ranking needed
    for (int i = tid; i < a.k; i += NT) out[i] = i < NP ? i : -1;
    return;
  }
  const int nct = (NP + a.chunk - 1) / a.chunk;  // scoring CTAs that saw pages of this row
  const int32_t* ccount = a.cand_count + (size_t)row * a.ncmax;
  const uint32_t* ctau = a.cand_tau + (size_t)row * a.ncmax;

  // 1. offsets of every CTA's candidates, their total and tau_max
  {
    int total = 0;
    uint32_t tmax = 0;
    for (int c0 = 0; c0 < nct; c0 += NT) {
      const int c = c0 + tid;
      const int v = c < nct ? ccount[c] : 0;
      if (c < nct) tmax = max(tmax, ctau[c]);
      int tot;
      const int ex = block_excl_scan<NT>(v, sh.w.scan_tmp, tot);
      if (c < nct) soff[c] = total + ex;
      total += tot;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tmax = max(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
    if (lane == 0) sh.w.red[warp] = tmax;
    __syncthreads();
    if (tid == 0) {
      uint32_t m = 0;
      for (int w = 0; w < NWp; ++w) m = max(m, sh.w.red[w]);
      sh.w.tau_max = m;
      sh.w.n = total;
      sh.w.ok = total <= kWideCandMax;
      soff[nct] = total;
    }
    __syncthreads();
  }
  const int n = sh.w.n;
  if (sh.w.ok) {  // uniform
    // 2. the candidates in page order (warp w copies CTAs w, w + 32, ...)
    for (int c = warp; c < nct; c += NWp) {
      const int o = soff[c], cnt = soff[c + 1] - o;
      const uint32_t* ck = a.cand_key + (size_t)row * a.npcap + (size_t)c * a.chunk;
      const int32_t* cp = a.cand_page + (size_t)row * a.npcap + (size_t)c * a.chunk;
#pragma unroll 4
      for (int j = lane; j < cnt; j += 32) {  // unrolled: the loads of four rounds in flight together
        skey[o + j] = __ldcg(ck + j);
        spage[o + j] = __ldcg(cp + j);
      }
    }
    __syncthreads();
    // 3. forced keys and the largest other candidate
    uint32_t top = 0;
    int nf = 0;
    for (int i = tid; i < n; i += NT) {
      const uint32_t kk = skey[i];
      if (kk == kForcedKey) ++nf;
      else top = max(top, kk);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      top = max(top, __shfl_xor_sync(0xffffffffu, top, o));
      nf += __shfl_xor_sync(0xffffffffu, nf, o);
    }
    if (lane == 0) {
      sh.w.red[warp] = top;
      sh.w.red_n[warp] = nf;
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t t = 0;
      int f = 0;
      for (int w = 0; w < NWp; ++w) {
        t = max(t, sh.w.red[w]);
        f += sh.w.red_n[w];
      }
      sh.w.top = t;
      sh.w.nforced = f;
    }
    __syncthreads();
    const int need = a.k - sh.w.nforced;
    if (need <= 0) {
      if (tid == 0) {
        sh.w.T = kForcedKey;
        sh.w.take = a.k;
      }
    } else {
      // 4. T among the free keys in [lo, hi] (first [tau_max, top]): a range
      //    histogram, the bin where the count from the top reaches rem, and
      //    the same again inside that bin while it holds too many keys
      uint32_t hi = sh.w.top, lo = sh.w.tau_max;
      int rem = need;
      const bool found = narrow_to_rank<NT, kWideBins>(skey, n, lo, hi, rem, kWideRank, sh.w.hist, sh.w.rank);
      if (tid == 0 && !found) sh.w.ok = 0;  // fewer than `need` free keys at or above tau_max
      __syncthreads();
      if (sh.w.ok) {  // uniform
        // 5. exact rank inside [lo, hi] (every key equal when lo == hi)
        if (tid == 0) sh.w.nbin = 0;
        __syncthreads();
        for (int i = tid; i < n; i += NT) {
          const uint32_t kk = skey[i];
          if (kk != kForcedKey && kk >= lo && kk <= hi) {
            const int slot = atomicAdd(&sh.w.nbin, 1);
            if (slot < kWideRank) sh.w.bin_keys[slot] = kk;
          }
        }
        __syncthreads();
        const int m = min(sh.w.nbin, kWideRank);
        if (lo == hi) {
          if (tid == 0) {
            sh.w.T = lo;
            sh.w.take = rem;
          }
        } else {
          for (int i = tid; i < m; i += NT) {
            const uint32_t v = sh.w.bin_keys[i];
            int gt = 0, ge = 0;
            for (int j = 0; j < m; ++j) {
              gt += sh.w.bin_keys[j] > v;
              ge += sh.w.bin_keys[j] >= v;
            }
            if (gt < rem && ge >= rem) {
              sh.w.T = v;            // every writer writes the same value
              sh.w.take = rem - gt;  // T-valued keys to take
            }
          }
        }
      }
    }
    __syncthreads();
  }
  if (sh.w.ok) {  // uniform
    // 6. ascending output: position = (#keys > T before) + min(#T-keys before, take)
    const uint32_t T = sh.w.T;
    const int take = sh.w.take;
    const int per_t = (n + NT - 1) / NT;
    const int i0 = min(tid * per_t, n), i1 = min(i0 + per_t, n);
    int gt = 0, eq = 0;
    for (int i = i0; i < i1; ++i) {
      const uint32_t kk = skey[i];
      gt += kk > T;
      eq += kk == T;
    }
    int Gx, Ex;
    block_pair_excl_scan<NT>(gt, eq, sh.w.scan_tmp, Gx, Ex);
    for (int i = i0; i < i1; ++i) {
      const uint32_t kk = skey[i];
      if (kk > T) {
        const int pos = Gx + min(Ex, take);
        if (pos < a.k) out[pos] = spage[i];
        ++Gx;
      } else if (kk == T) {
        if (Ex < take && Gx + Ex < a.k) out[Gx + Ex] = spage[i];
        ++Ex;
      }
    }
    return;
  }
  // fallback: every key of the row, from global memory
  __syncthreads();
  if (tid == 0) atomicAdd(&g_select_rows_all_keys, 1ull);
  row_topk<NT>(a.keys + (size_t)row * a.npcap, NP, a.k, 0, out, sh.radix);
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
    row_topk<NT>(skeys, n, k, 0, out, *reinterpret_cast<TopkShared*>(hist));
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

// Pages per scoring CTA: one wave of scoring CTAs over all rows.
template <typename T, int D, int GM, int MODE, bool CAND>
static int score_chunk_for(int npcap, int rows) {
  auto kern = quest_score_kernel<T, D, GM, MODE, CAND>;
  constexpr int NT = MODE == 0 ? kSelThreads : kSelThreadsMma;
  static int per_sm = 0;  // resident CTAs per SM of this kernel (same on every GB300)
  if (per_sm == 0) cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, 0);
  const int slots = max(1, sm_count() * max(per_sm, 1));
  const int cpr = max(1, slots / rows);
  return max(16, ((npcap + cpr - 1) / cpr + 15) / 16 * 16);
}

template <typename T, int D, int GM, int MODE, bool CAND>
static cudaError_t score_launch_c(SelectArgs& a, int rows, cudaStream_t st) {
  auto kern = quest_score_kernel<T, D, GM, MODE, CAND>;
  constexpr int NT = MODE == 0 ? kSelThreads : kSelThreadsMma;
  a.chunk = score_chunk_for<T, D, GM, MODE, CAND>(a.npcap, rows);
  dim3 grid((a.npcap + a.chunk - 1) / a.chunk, rows);
  const size_t smem = (a.cand_key && a.chunk <= kCandStage) ? (size_t)a.chunk * 4 : 0;  // staged keys
  cudaError_t e = launch_pdl(kern, grid, dim3(NT), smem, st, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T, int D, int GM, int MODE>
static cudaError_t score_launch(SelectArgs& a, int rows, cudaStream_t st) {
  return a.cand_key ? score_launch_c<T, D, GM, MODE, true>(a, rows, st)
                    : score_launch_c<T, D, GM, MODE, false>(a, rows, st);
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
  if (a.cand_key) {  // wide rows: rank the scoring CTAs' candidates
    const int nct = (a.npcap + a.chunk - 1) / a.chunk;
    const size_t smem = (size_t)kWideCandMax * 8 + (size_t)(nct + 1) * 4;
    cudaError_t e = cudaFuncSetAttribute(topk_wide_kernel<kWideThreads>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(topk_wide_kernel<kWideThreads>, dim3(rows), dim3(kWideThreads), smem, st, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  return cudaErrorInvalidValue;  // unreachable: wide rows always carry candidate buffers
}

template <typename T, int D>
static cudaError_t score_g(SelectArgs& a, int rows, cudaStream_t st) {
  if (a.G <= 1) return score_launch<T, D, 1, 0>(a, rows, st);
  if (a.G <= 2) return score_launch<T, D, 2, 0>(a, rows, st);
  if (a.G <= 4) return score_launch<T, D, 4, 0>(a, rows, st);
  return score_launch<T, D, 8, 0>(a, rows, st);
}

template <int D>
static cudaError_t score_mma(SelectArgs& a, int rows, cudaStream_t st) {
  if (a.P == 1) return score_launch<bf16, D, 8, 2>(a, rows, st);
  return score_launch<bf16, D, 8, 1>(a, rows, st);
}

// Rows wider than one register-resident top-k CTA take the candidate path.
static bool wide_rows(const Shape& s) { return (s.Cap >> s.pshift) > kRegTopkThreads * kRegTopkKeys; }

static size_t align_256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t select_pages_workspace(const Shape& s) {
  const size_t rows = (size_t)s.B * s.Hkv, npcap = (size_t)(s.Cap >> s.pshift);
  size_t bytes = align_256(rows * npcap * sizeof(uint32_t));  // one key per page
  if (wide_rows(s))  // candidate keys and pages, per-CTA counts and thresholds
    bytes += 2 * align_256(rows * npcap * 4) + 2 * align_256(rows * ((npcap + 15) / 16) * 4);
  return bytes;
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
  a.cand_key = nullptr;
  a.cand_page = nullptr;
  a.cand_count = nullptr;
  a.cand_tau = nullptr;
  a.ncmax = (a.npcap + 15) / 16;  // >= scoring CTAs per row (chunk >= 16)
  const int rows = s.B * s.Hkv;
  if (wide_rows(s)) {
    unsigned char* w = static_cast<unsigned char*>(ws) + align_256((size_t)rows * a.npcap * 4);
    a.cand_key = reinterpret_cast<uint32_t*>(w);
    w += align_256((size_t)rows * a.npcap * 4);
    a.cand_page = reinterpret_cast<int32_t*>(w);
    w += align_256((size_t)rows * a.npcap * 4);
    a.cand_count = reinterpret_cast<int32_t*>(w);
    w += align_256((size_t)rows * a.ncmax * 4);
    a.cand_tau = reinterpret_cast<uint32_t*>(w);
  }
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

unsigned long long take_select_rows_all_keys(bool reset) {
  unsigned long long v = 0;
  if (cudaMemcpyFromSymbol(&v, g_select_rows_all_keys, sizeof(v)) != cudaSuccess) return 0;
  if (reset) {
    const unsigned long long zero = 0;
    cudaMemcpyToSymbol(g_select_rows_all_keys, &zero, sizeof(zero));
  }
  return v;
}

}  // namespace sls
