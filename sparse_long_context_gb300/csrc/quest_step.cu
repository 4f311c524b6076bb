// Fused Quest decode step for bf16 caches with pages of >= 16 tokens: page
// selection (bound, top-k) and sparse attention with the split combine in
// one launch ("Don't read the haystack", Part two: the page bound
// sum_c max(q_c * kmin_c, q_c * kmax_c), max over the GQA group, budget k
// including the sink page and the local pages; then attention over the
// chosen pages only).
//
// One thread-block cluster of C CTAs per (sequence, KV head) row; CTA c:
//   1. score   streams the page min/max of pages [c*chunk, (c+1)*chunk)
//              through a ring of shared-memory stages (tensor-map copies of
//              16 pages of kmax and of kmin) and scores them on the tensor
//              cores: U = kmax . max(q, 0) + kmin . min(q, 0), a 16-page x
//              8-head product per stage; the page score is the max over the
//              group's heads.  One order-preserving 32-bit key per page stays
//              in shared memory (forced pages get the largest key).
//   2. top-k   the cluster finds the k-th largest key T by four MSB-first
//              passes over 8-bit digits (each CTA histograms its keys, every
//              CTA sums the C histograms through distributed shared memory),
//              and how many T-valued keys to take (ties go to lower pages).
//              Each CTA writes its chosen pages, ascending, into the row's
//              list in CTA 0 (and to page_idx) at offsets from the cluster's
//              per-CTA counts.
//   3. attend  CTA c takes a contiguous 1/C of the list and runs the
//              tensor-core online-softmax attention of the split-K kernel on
//              its 16-token groups, fed by the same ring.
//   4. combine the splits' partials meet in distributed shared memory.
// Nothing of the step goes through global memory but its inputs and outputs.
#include "attend_tma.cuh"
#include "launch.h"

#include <algorithm>

namespace sls {

constexpr int kStepMinBlocks = 3;
constexpr int kStepMaxChunk = 8192;  // pages scored by one CTA (keys kept in shared memory)
constexpr int kStepMaxK = 4096;      // page budget (the row's list sits in shared memory)
constexpr uint32_t kForcedKey32 = 0xffffffffu;

__device__ unsigned long long g_step_rows_dense = 0;     // rows attended densely (sparsity gate)
__device__ unsigned long long g_step_rows_all_keys = 0;  // rows selected from all keys

struct StepArgs {
  AttendArgs a;  // q, k, v, ctx_len, sink, out, lse, shapes, qscale; S = C; cluster = 1
  const void* kmin;   // [rows, Cap / P, D] page minima
  const void* kmax;   // [rows, Cap / P, D] page maxima
  int32_t* page_idx;  // [rows, k] or null
  int k, n_sink, n_local;
  int chunk;  // pages scored per CTA (multiple of 16)
  int npcap;  // Cap / P
  size_t keys_bytes;   // shared-memory region of the keys (also the combine inbox)
  int scratch_off;     // top-k scratch in the ring, after the row's keys (all-keys selection)
  float min_sparsity;  // rows with N < min_sparsity * k * P attend densely (0: never)
  int topk_mode;       // 0: candidates of every CTA, 1: all keys to every CTA
  int cand_cap;        // candidates one CTA may send
  int cand_m;          // real keys a CTA sends (about; plus its forced keys)
};

template <int D>
struct StepLayout {
  static constexpr size_t RING = (size_t)kTmaStages * TmaLayout<D>::STAGE;
  static constexpr size_t MERGE = (size_t)kTmaConsumers * 8 * D * sizeof(float);
  static constexpr size_t RING_REGION = RING > MERGE ? RING : MERGE;
};

// Scores of the 16 pages of the stage at `stage` (kmax tile then kmin
// tile).  A = the page tile (rows = pages) from ldmatrix; lane (r, m) gives
// the row address of matrix j = lane / 8, row i = lane % 8: page
// 8 * (j % 2) + i, 8-channel chunk 2 * step + j / 2.  B = max(q, 0) for
// kmax and min(q, 0) for kmin (heads as columns).
template <int D>
__device__ __forceinline__ void score_stage(uint32_t stage, const uint32_t (&bp)[D / 16][2],
                                            const uint32_t (&bn)[D / 16][2], int G, int lane, float& v0,
                                            float& v1) {
  using L = TmaLayout<D>;
  constexpr int KS = D / 16;
  const int m = lane & 3;
  const int j = lane >> 3, i = lane & 7;
  const int page = 8 * (j & 1) + i;
  auto row_addr = [&](uint32_t base, int c16) -> uint32_t {
    const int bx = c16 >> 3, c = c16 & 7;
    return base + bx * L::BOX + page * 128 + ((c ^ i) << 4);
  };
  float ch[4] = {0.f, 0.f, 0.f, 0.f}, cl[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4(row_addr(stage, 2 * ks + (j >> 1)), a0, a1, a2, a3);
    mma_bf16(ch, a0, a1, a2, a3, bp[ks][0], bp[ks][1]);
    ldsm_x4(row_addr(stage + L::GROUP, 2 * ks + (j >> 1)), a0, a1, a2, a3);
    mma_bf16(cl, a0, a1, a2, a3, bn[ks][0], bn[ks][1]);
  }
  // C[page][head]: c0, c1 = page r, heads 2m, 2m+1; c2, c3 = page r + 8
  const bool h0 = 2 * m < G, h1 = 2 * m + 1 < G;
  v0 = kNegInf;
  v1 = kNegInf;
  if (h0) {
    v0 = ch[0] + cl[0];
    v1 = ch[2] + cl[2];
  }
  if (h1) {
    v0 = fmaxf(v0, ch[1] + cl[1]);
    v1 = fmaxf(v1, ch[3] + cl[3]);
  }
  v0 = fmaxf(v0, __shfl_xor_sync(0xffffffffu, v0, 1));
  v0 = fmaxf(v0, __shfl_xor_sync(0xffffffffu, v0, 2));
  v1 = fmaxf(v1, __shfl_xor_sync(0xffffffffu, v1, 1));
  v1 = fmaxf(v1, __shfl_xor_sync(0xffffffffu, v1, 2));
}

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive scan of one int per thread over the CTA; `total` gets the sum.
template <int NT>
__device__ __forceinline__ int block_scan_excl(int v, int* tmp, int& total) {
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
  if (warp == 0) {
    int t = lane < NWp ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < NWp) tmp[lane] = t;
  }
  __syncthreads();
  const int before = warp > 0 ? tmp[warp - 1] : 0;
  total = tmp[NWp - 1];
  __syncthreads();
  return before + x - v;
}

constexpr int kWinBins = 2048;  // window of top-16-bit values below the largest
constexpr int kRegKeys = 32;    // keys per thread when the row's keys fit in registers
constexpr int kLocalKeys = 8;   // keys per thread of a CTA's own selection (chunk <= NT * 8)
constexpr int kCandMax = 1024;  // keys of the threshold bin ranked exactly
constexpr int kTopkScratchBytes = (kWinBins + 32 + kCandMax + 256) * 4;

struct TopkScalars {
  uint32_t red_max[32];
  uint32_t red_min[32];
  int red_n[32];
  int bin, rem, ncand, digit;
  uint32_t T;
  int take;
};

// Largest digit d (descending order) where the running count of `cnt`
// (256 digits, counts of keys above in cnt order) reaches rem: warp 0.
__device__ __forceinline__ void find_digit(const uint32_t* cnt, int rem, TopkScalars& sc) {
  const int lane = threadIdx.x & 31;
  uint32_t c8[8], s = 0;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    c8[u] = cnt[255 - 8 * lane - u];
    s += c8[u];
  }
  uint32_t incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  uint32_t above = incl - s;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    if (above < (uint32_t)rem && above + c8[u] >= (uint32_t)rem) {
      sc.digit = 255 - 8 * lane - u;
      sc.rem = rem - (int)above;
    }
    above += c8[u];
  }
}

// MSB-first radix select over keys[0 .. n) restricted to keys whose bits
// above `shift0 + 8` equal `prefix`: the rem-th largest T and how many
// T-valued keys to take.  scratch: 256 words.
template <int NT>
__device__ __forceinline__ void radix_select(const uint32_t* keys, int n, uint32_t prefix, uint32_t pmask, int shift0,
                                             int rem, uint32_t* hist, TopkScalars& sc, uint32_t& T, int& take) {
  for (int shift = shift0; shift >= 0; shift -= 8) {
    for (int d = threadIdx.x; d < 256; d += NT) hist[d] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += NT) {
      const uint32_t key = keys[i];
      if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) find_digit(hist, rem, sc);
    __syncthreads();
    prefix |= (uint32_t)sc.digit << shift;
    pmask |= 255u << shift;
    rem = sc.rem;
    __syncthreads();
  }
  T = prefix;
  take = rem;
}

// The k-th largest of keys[0 .. n) (n > k) and how many keys equal to it to
// take (the lowest pages first), computed by every CTA of the cluster on its
// own copy in shared memory (rows too long for select_share_reg): the same
// range-scaled histogram, threshold bin and exact rank; a full radix select
// when the bin is crowded.  scratch: kWinBins + kCandMax + 256 words.
template <int NT>
__device__ __forceinline__ void local_topk(const uint32_t* keys, int n, int k, uint32_t* scratch, int* scan_tmp,
                                           uint32_t& T, int& take) {
  __shared__ TopkScalars sc;
  uint32_t* hist = scratch;             // [kWinBins]
  uint32_t* cand = scratch + kWinBins;  // [kCandMax]
  uint32_t* h256 = cand + kCandMax;     // [256]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int NWp = NT / 32;
  uint32_t mx = 0, mn = 0xffffffffu;
  int nf = 0;
  for (int i = threadIdx.x; i < n; i += NT) {
    const uint32_t key = keys[i];
    if (key == kForcedKey32) {
      ++nf;
    } else {
      mx = max(mx, key);
      mn = min(mn, key);
    }
  }
  for (int d = threadIdx.x; d < kWinBins; d += NT) hist[d] = 0;
  mx = __reduce_max_sync(0xffffffffu, mx);
  mn = __reduce_min_sync(0xffffffffu, mn);
  nf = __reduce_add_sync(0xffffffffu, nf);
  if (lane == 0) {
    sc.red_max[warp] = mx;
    sc.red_min[warp] = mn;
    sc.red_n[warp] = nf;
  }
  if (threadIdx.x == 0) {
    sc.ncand = 0;
    sc.bin = -1;
  }
  __syncthreads();
  const uint32_t top = __reduce_max_sync(0xffffffffu, lane < NWp ? sc.red_max[lane] : 0u);
  const uint32_t bot = __reduce_min_sync(0xffffffffu, lane < NWp ? sc.red_min[lane] : 0xffffffffu);
  const int nforced = __reduce_add_sync(0xffffffffu, lane < NWp ? sc.red_n[lane] : 0);
  const int need = k - nforced;
  if (need <= 0) {  // the first k forced pages
    T = kForcedKey32;
    take = k;
    return;
  }
  int shift = 0;
  while (((top - bot) >> shift) >= (uint32_t)kWinBins) ++shift;
  for (int i = threadIdx.x; i < n; i += NT) {
    const uint32_t key = keys[i];
    if (key != kForcedKey32) atomicAdd(&hist[(top - key) >> shift], 1u);
  }
  __syncthreads();
  constexpr int BPT = (kWinBins + NT - 1) / NT;
  const int b0 = threadIdx.x * BPT;
  int sum = 0;
  for (int i = 0; i < BPT; ++i) sum += b0 + i < kWinBins ? (int)hist[b0 + i] : 0;
  int total;
  int above = block_scan_excl<NT>(sum, scan_tmp, total);
  for (int i = 0; i < BPT; ++i) {
    const int c = b0 + i < kWinBins ? (int)hist[b0 + i] : 0;
    if (above < need && above + c >= need) {
      sc.bin = b0 + i;
      sc.rem = need - above;
    }
    above += c;
  }
  __syncthreads();
  if (sc.bin >= 0) {
    const uint32_t bin = (uint32_t)sc.bin;
    const int rem = sc.rem;
    for (int i = threadIdx.x; i < n; i += NT) {
      const uint32_t key = keys[i];
      if (key != kForcedKey32 && ((top - key) >> shift) == bin) {
        const int slot = atomicAdd(&sc.ncand, 1);
        if (slot < kCandMax) cand[slot] = key;
      }
    }
    __syncthreads();
    const int m = sc.ncand;
    if (m <= kCandMax) {
      radix_select<NT>(cand, m, 0u, 0u, 24, rem, h256, sc, T, take);
      return;
    }
  }
  __syncthreads();
  radix_select<NT>(keys, n, 0u, 0u, 24, k, h256, sc, T, take);
}

// Keys[0 .. n) into registers, thread t owning positions [t*KPT, t*KPT+KPT)
// (position order = thread order); slots past n hold 0, below every key.
template <int NT, int KPT>
__device__ __forceinline__ void load_keys_reg(const uint32_t* keys, int n, uint32_t (&kk)[KPT]) {
  const uint4* src = reinterpret_cast<const uint4*>(keys + threadIdx.x * KPT);
#pragma unroll
  for (int v = 0; v < KPT / 4; ++v) {
    const int i = threadIdx.x * KPT + 4 * v;
    uint4 x = make_uint4(0, 0, 0, 0);
    if (i + 3 < n) {
      x = src[v];
    } else if (i < n) {  // ragged end
      x.x = keys[i];
      x.y = i + 1 < n ? keys[i + 1] : 0u;
      x.z = i + 2 < n ? keys[i + 2] : 0u;
    }
    kk[4 * v] = x.x; kk[4 * v + 1] = x.y; kk[4 * v + 2] = x.z; kk[4 * v + 3] = x.w;
  }
}

// The k-th largest T of the keys held in registers (zero slots excluded;
// k <= the number of keys) and how many T-valued keys to take, the first in
// position order.  Bound scores cluster tightly, so the histogram spans the
// keys' own range: bin (top - key) >> shift, with the smallest shift that
// fits the range into kWinBins bins.  The threshold bin's keys are ranked
// exactly (by counting, or a radix select when the bin is crowded).  Forced
// keys (the largest value) are counted first.  Returns false when the bin
// holds more than kCandMax keys (T and take are then undefined).
template <int NT, int KPT, int NB = kWinBins>
__device__ __forceinline__ bool kth_largest_reg(const uint32_t (&kk)[KPT], int k, uint32_t* scratch, int* scan_tmp,
                                                uint32_t& T, int& take) {
  // Loops over the keys are branch-free (selects, a spill bin, one slot
  // reservation per warp): divergent branches per key cost far more here
  // than the work they guard.
  __shared__ TopkScalars sc;
  static_assert((NB & (NB - 1)) == 0 && NB <= kWinBins, "bins: a power of two");
  constexpr int LB = __builtin_ctz(NB);
  uint32_t* hist = scratch;            // [NB + 32]: the last 32 bins absorb excluded keys
  uint32_t* cand = scratch + NB + 32;  // [kCandMax]
  uint32_t* h256 = cand + kCandMax;          // [256]
  constexpr int NWp = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // 1. range of the non-forced keys and the forced count
  uint32_t mx = 0, mn = 0xffffffffu;
  int nf = 0;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const uint32_t x = kk[j];
    const bool forced = x == kForcedKey32, real = !forced && x != 0u;
    nf += forced;
    mx = max(mx, real ? x : 0u);
    mn = min(mn, real ? x : 0xffffffffu);
  }
  for (int d = threadIdx.x; d < NB + 32; d += NT) hist[d] = 0;
  mx = __reduce_max_sync(0xffffffffu, mx);
  mn = __reduce_min_sync(0xffffffffu, mn);
  nf = __reduce_add_sync(0xffffffffu, nf);
  if (lane == 0) {
    sc.red_max[warp] = mx;
    sc.red_min[warp] = mn;
    sc.red_n[warp] = nf;
  }
  if (threadIdx.x == 0) {
    sc.ncand = 0;
    sc.bin = -1;
  }
  __syncthreads();
  const uint32_t top = __reduce_max_sync(0xffffffffu, lane < NWp ? sc.red_max[lane] : 0u);
  const uint32_t bot = __reduce_min_sync(0xffffffffu, lane < NWp ? sc.red_min[lane] : 0xffffffffu);
  const int nforced = __reduce_add_sync(0xffffffffu, lane < NWp ? sc.red_n[lane] : 0);
  const int need = k - nforced;
  T = kForcedKey32;
  take = k;
  if (need <= 0) return true;  // the first k forced keys
  // 2. histogram of (top - key) >> shift, the smallest shift fitting the range
  const uint32_t span = top - bot;
  const int shift = span >= (uint32_t)NB ? 32 - __clz(span >> LB) : 0;  // (span >> shift) < NB
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const uint32_t x = kk[j];
    const bool real = x != kForcedKey32 && x != 0u;
    atomicAdd(&hist[real ? (top - x) >> shift : NB + lane], 1u);
  }
  __syncthreads();
  // 3. the bin of the need-th largest
  constexpr int BPT = (NB + NT - 1) / NT;
  const int b0 = threadIdx.x * BPT;
  int cnt[BPT], sum = 0;
#pragma unroll
  for (int i = 0; i < BPT; ++i) {
    cnt[i] = b0 + i < NB ? (int)hist[b0 + i] : 0;
    sum += cnt[i];
  }
  int total;
  int above = block_scan_excl<NT>(sum, scan_tmp, total);
  int mybin = -1, myrem = 0;
#pragma unroll
  for (int i = 0; i < BPT; ++i) {
    const bool hit = above < need && above + cnt[i] >= need;
    mybin = hit ? b0 + i : mybin;
    myrem = hit ? need - above : myrem;
    above += cnt[i];
  }
  if (mybin >= 0) {
    sc.bin = mybin;
    sc.rem = myrem;
  }
  __syncthreads();
  if (sc.bin < 0) return false;  // fewer non-forced keys than needed
  // 4. the bin's keys, one slot reservation per warp
  const uint32_t bin = (uint32_t)sc.bin;
  unsigned bal[KPT];
  int wcount = 0;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const uint32_t x = kk[j];
    const bool in = x != kForcedKey32 && x != 0u && ((top - x) >> shift) == bin;
    bal[j] = __ballot_sync(0xffffffffu, in);
    wcount += __popc(bal[j]);
  }
  int base = 0;
  if (lane == 0 && wcount) base = atomicAdd(&sc.ncand, wcount);
  base = __shfl_sync(0xffffffffu, base, 0);
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const int slot = base + __popc(bal[j] & ((1u << lane) - 1u));
    if (((bal[j] >> lane) & 1u) && slot < kCandMax) cand[slot] = kk[j];
    base += __popc(bal[j]);
  }
  __syncthreads();
  const int m = sc.ncand;
  const int rem = sc.rem;
  if (m > kCandMax) return false;
  if (m <= 2 * NT) {
    // 5. exact rank by counting (each candidate against all of them)
    for (int i = threadIdx.x; i < m; i += NT) {
      const uint32_t v = cand[i];
      int gt = 0, ge = 0;
      for (int q = 0; q < m; ++q) {
        const uint32_t w = cand[q];
        gt += w > v;
        ge += w >= v;
      }
      if (gt < rem && ge >= rem) {
        sc.T = v;
        sc.take = rem - gt;
      }
    }
    __syncthreads();
    T = sc.T;
    take = sc.take;
  } else {
    radix_select<NT>(cand, m, 0u, 0u, 24, rem, h256, sc, T, take);
  }
  return true;
}

// Positions in the ascending list of the keys chosen by (T, take): for the
// key at position i, (#keys > T before i) + min(#T-keys before i, take).
// Entries that land in [e0, e0 + nent) get share[pos - e0] = values[i *
// vstride] (the position i when `values` is null).
template <int NT, int KPT>
__device__ __forceinline__ void place_chosen(const uint32_t (&kk)[KPT], uint32_t T, int take, int e0, int nent,
                                             const int32_t* values, int32_t* share, int* scan_tmp,
                                             int vstride = 1) {
  int gt = 0, eq = 0;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    gt += kk[j] > T;
    eq += kk[j] == T;
  }
  int tot;
  const int excl = block_scan_excl<NT>((gt << 16) | eq, scan_tmp, tot);  // both totals < 2^15
  int Gp = excl >> 16, Ep = excl & 0xffff;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const uint32_t x = kk[j];
    const bool g = x > T, e = x == T;
    const int pos = g ? Gp + min(Ep, take) : ((e && Ep < take) ? Gp + Ep : -1);
    Gp += g;
    Ep += e;
    const int i = threadIdx.x * KPT + j;
    if (pos >= e0 && pos < e0 + nent) share[pos - e0] = values ? values[(size_t)i * vstride] : i;
  }
}

// All-keys selection of the row (keys[0 .. n) by page, n <= NT * KPT) into
// this CTA's share of the list.  False when the exact rank overflows.
template <int NT, int KPT>
__device__ __forceinline__ bool select_share_reg(const uint32_t* keys, int n, int k, uint32_t* scratch, int e0,
                                                 int nent, int32_t* share, int* scan_tmp) {
  uint32_t kk[KPT];
  load_keys_reg<NT, KPT>(keys, n, kk);
  uint32_t T;
  int take;
  if (!kth_largest_reg<NT, KPT>(kk, k, scratch, scan_tmp, T, take)) return false;
  place_chosen<NT, KPT>(kk, T, take, e0, nent, nullptr, share, scan_tmp);
  return true;
}

// A CTA's candidate threshold: the smallest key tau such that the CTA's real
// (non-forced) keys >= tau are its m largest plus the rest of their
// histogram bin (NB range-scaled bins, as in kth_largest_reg); 1 (every key)
// when the CTA holds at most m real keys.  No exact rank: the cluster's
// selection checks afterwards that the row's k-th largest is >= every CTA's
// tau, which makes the candidates a superset of the row's top k.
template <int NT, int KPT, int NB = 1024>
__device__ __forceinline__ uint32_t top_bin_threshold(const uint32_t (&kk)[KPT], int m, uint32_t* hist,
                                                      int* scan_tmp) {
  __shared__ TopkScalars sc;
  constexpr int NWp = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t mx = 0, mn = 0xffffffffu;
  int nr = 0;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const uint32_t x = kk[j];
    const bool real = x != kForcedKey32 && x != 0u;
    nr += real;
    mx = max(mx, real ? x : 0u);
    mn = min(mn, real ? x : 0xffffffffu);
  }
  static_assert((NB & (NB - 1)) == 0 && NB <= kWinBins, "bins: a power of two");
  constexpr int LB = __builtin_ctz(NB);
  for (int d = threadIdx.x; d < NB + 32; d += NT) hist[d] = 0;
  mx = __reduce_max_sync(0xffffffffu, mx);
  mn = __reduce_min_sync(0xffffffffu, mn);
  nr = __reduce_add_sync(0xffffffffu, nr);
  if (lane == 0) {
    sc.red_max[warp] = mx;
    sc.red_min[warp] = mn;
    sc.red_n[warp] = nr;
  }
  if (threadIdx.x == 0) sc.bin = -1;
  __syncthreads();
  const uint32_t top = __reduce_max_sync(0xffffffffu, lane < NWp ? sc.red_max[lane] : 0u);
  const uint32_t bot = __reduce_min_sync(0xffffffffu, lane < NWp ? sc.red_min[lane] : 0xffffffffu);
  const int nreal = __reduce_add_sync(0xffffffffu, lane < NWp ? sc.red_n[lane] : 0);
  if (nreal <= m) return 1u;  // uniform: every thread read the same totals
  const uint32_t span = top - bot;
  const int shift = span >= (uint32_t)NB ? 32 - __clz(span >> LB) : 0;  // (span >> shift) < NB
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const uint32_t x = kk[j];
    const bool real = x != kForcedKey32 && x != 0u;
    atomicAdd(&hist[real ? (top - x) >> shift : NB + lane], 1u);
  }
  __syncthreads();
  constexpr int BPT = (NB + NT - 1) / NT;
  const int b0 = threadIdx.x * BPT;
  int cnt[BPT], sum = 0;
#pragma unroll
  for (int i = 0; i < BPT; ++i) {
    cnt[i] = b0 + i < NB ? (int)hist[b0 + i] : 0;
    sum += cnt[i];
  }
  int total;
  int above = block_scan_excl<NT>(sum, scan_tmp, total);
  int mybin = -1;
#pragma unroll
  for (int i = 0; i < BPT; ++i) {
    mybin = (above < m && above + cnt[i] >= m) ? b0 + i : mybin;
    above += cnt[i];
  }
  if (mybin >= 0) sc.bin = mybin;
  __syncthreads();
  // keys x with (top - x) >> shift <= bin
  const long long lo = (long long)top - ((long long)(sc.bin + 1) << shift) + 1;
  return (uint32_t)max(lo, 1ll);
}

// Candidates of the cluster's CTAs in one array of (key, page) pairs, CTA c
// at slots [c * cap, c * cap + n[c]), slot order = page order; the other
// slots hold key 0 (below every key).  Thread t holds slots
// [t * KPT, t * KPT + KPT).
template <int NT, int KPT>
__device__ __forceinline__ void load_cand_reg(const uint2* cand, int slots, uint32_t (&kk)[KPT]) {
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const int i = threadIdx.x * KPT + j;
    kk[j] = i < slots ? cand[i].x : 0u;
  }
}

// The row's chosen pages from the cluster's candidates into this CTA's share
// of the list.  False (the same in every CTA of the cluster) when the rank
// overflows or when the row's k-th largest T falls below some CTA's
// threshold: that CTA may hold unsent keys >= T.
template <int NT, int KPT>
__device__ __forceinline__ bool select_share_cand(const uint2* cand, int slots, int C, const uint32_t* tau, int k,
                                                  uint32_t* scratch, int e0, int nent, int32_t* share,
                                                  int* scan_tmp) {
  uint32_t kk[KPT];
  load_cand_reg<NT, KPT>(cand, slots, kk);
  uint32_t T;
  int take;
  // a few hundred candidates: 512 range-scaled bins leave about one key per bin
  constexpr int NB = KPT <= 4 ? 512 : kWinBins;
  if (!kth_largest_reg<NT, KPT, NB>(kk, k, scratch, scan_tmp, T, take)) return false;
  uint32_t tmax = 0u;
  for (int c = 0; c < C; ++c) tmax = max(tmax, tau[c]);
  if (T < tmax) return false;
  place_chosen<NT, KPT>(kk, T, take, e0, nent, reinterpret_cast<const int32_t*>(cand) + 1, share, scan_tmp, 2);
  return true;
}

template <int D>
__global__ void __launch_bounds__((kTmaConsumers + 1) * 32, kStepMinBlocks)
quest_step_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                  const __grid_constant__ CUtensorMap tmin, const __grid_constant__ CUtensorMap tmax,
                  const StepArgs sa) {
  namespace cg = cooperative_groups;
  using L = TmaLayout<D>;
  constexpr int W = kTmaConsumers, NST = kTmaStages, KS = D / 16;
  constexpr int NT = (W + 1) * 32;
  const AttendArgs& a = sa.a;

  extern __shared__ unsigned char smem_raw[];
  unsigned char* ring = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint32_t* keys = reinterpret_cast<uint32_t*>(ring + StepLayout<D>::RING_REGION);
  ClusterInbox<D>* inbox = reinterpret_cast<ClusterInbox<D>*>(keys);  // after the top-k
  int32_t* list = reinterpret_cast<int32_t*>(ring + StepLayout<D>::RING_REGION + sa.keys_bytes);
  __shared__ uint64_t full[NST], empty[NST];
  __shared__ float sM[W][8], sL[W][8], sF[W][8];
  __shared__ float sHm[8], sHl[8];
  __shared__ int scan_tmp[32];
  __shared__ int s_cand_n[kMaxClusterSplits];
  __shared__ uint32_t s_cand_tau[kMaxClusterSplits];

  cg::cluster_group cl = cg::this_cluster();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_fence_init();
    tma_prefetch_map(&tk);
    tma_prefetch_map(&tv);
    tma_prefetch_map(&tmin);
    tma_prefetch_map(&tmax);
  }
  pdl_wait();

  const int C = a.S;
  const int row = blockIdx.x / C, split = blockIdx.x % C;  // split = rank in the cluster
  const int b = row / a.Hkv, h = row % a.Hkv;
  const int G = a.G, k = sa.k;
  const int N = clamp_len(a.ctx_len[b], a.Cap);
  const int NP = (N + a.P - 1) >> a.pshift;
  const int per = (k + C - 1) / C;  // list entries attended per CTA
  const int e0 = split * per;
  const int nent = max(0, min(per, k - e0));
  // sparsity gate (mlxcel, "Corrected premise 2"): a context shorter than
  // min_sparsity times the selected tokens is attended densely
  const bool dense = sa.min_sparsity > 0.f && (double)N < (double)sa.min_sparsity * k * a.P;
  __syncthreads();

  uint32_t seq = 0;  // ring position (identical in every thread)
  bool ok = true;    // this thread's waits all succeeded

  // producer's and consumers' walk of `n` stages starting at ring position seq0
  auto producer_wait = [&](uint32_t q, uint32_t tries = kWaitTries) -> bool {
    const int st = q % NST;
    const uint32_t use = q / NST;
    return use == 0 || mbar_wait(&empty[st], (use - 1) & 1, tries);
  };

  if (dense) {
    // every page of the context, no selection; page_idx stays -1
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // completes the arrive made at entry
    if (split == 0 && threadIdx.x == 0) atomicAdd(&g_step_rows_dense, 1ull);
    if (sa.page_idx)
      for (int e = threadIdx.x; e < nent; e += NT) sa.page_idx[(size_t)row * k + e0 + e] = -1;
  } else if (NP > k) {
    // ------------------------------------------------------------ 1. score
    const int p0 = split * sa.chunk;
    const int nloc = max(0, min(sa.chunk, NP - p0));
    const int n1 = (nloc + 15) >> 4;
    const int first_local = a.P > 0 && sa.n_local > 0 ? (max(N - sa.n_local, 0) >> a.pshift) : NP;
    // Every thread completes the cluster arrive made at entry while the first
    // copies are in flight (a wait on a phase long complete still takes a
    // while), before its first access to another CTA's shared memory.
    if (warp == W) {
      int issued = 0;
      auto issue = [&](int i0, int i1) {
        for (int i = i0; i < i1; ++i) {
          const uint32_t q = seq + i;
          const int st = q % NST;
          if (!producer_wait(q)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[st], L::STAGE);
          const int y = row * sa.npcap + p0 + 16 * i;
          unsigned char* dst = ring + st * L::STAGE;
          tma_load_3d(dst, &tmax, 0, y, 0, &full[st]);
          tma_load_3d(dst + L::GROUP, &tmin, 0, y, 0, &full[st]);
          issued = i + 1;
        }
      };
      if (lane == 0) issue(0, min(NST, n1));  // the ring's first round needs no free stage
      __syncwarp();
      asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
      if (lane == 0) {
        if (ok) issue(NST, n1);
        // the copies have landed before the ring turns into scratch space
        for (int i = max(0, issued - NST); i < issued; ++i) {
          const uint32_t q = seq + i;
          if (!mbar_wait(&full[q % NST], (q / NST) & 1)) ok = false;
        }
      }
    } else {
      asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
      const int r = lane >> 2, m = lane & 3;
      // q split by sign as the B operand: b0 = q[head r][16ks + 2m, +1], b1 = q[r][16ks + 8 + 2m, +1]
      uint32_t bp[KS][2], bn[KS][2];
      {
        const bf16* qp = static_cast<const bf16*>(a.q) + ((size_t)b * a.Hq + (size_t)h * G + r) * D;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const uint32_t w = r < G ? __ldg(reinterpret_cast<const uint32_t*>(qp + 16 * ks + 8 * u + 2 * m)) : 0u;
            bp[ks][u] = bf16x2_relu(w);
            bn[ks][u] = bf16x2_negpart(w);
          }
        }
      }
      const uint32_t ring_u32 = smem_u32(ring);
      for (int i = (W + warp - (int)(seq % W)) % W; i < n1; i += W) {
        const uint32_t q = seq + i;
        const int st = q % NST;
        if (!mbar_wait(&full[st], (q / NST) & 1)) {
          ok = false;
          break;
        }
        float v0, v1;
        score_stage<D>(ring_u32 + st * L::STAGE, bp, bn, G, lane, v0, v1);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        if (m == 0) {
          const int i0 = 16 * i + r, i1 = i0 + 8;
          const int pg0 = p0 + i0, pg1 = p0 + i1;
          if (i0 < nloc) keys[i0] = (pg0 < sa.n_sink || pg0 >= first_local) ? kForcedKey32 : order_key(v0);
          if (i1 < nloc) keys[i1] = (pg1 < sa.n_sink || pg1 >= first_local) ? kForcedKey32 : order_key(v1);
        }
      }
    }
    seq += n1;
    __syncthreads();  // keys complete; the ring is free

    // ------------------------------------------------------------ 2. top-k
    bool use_all = sa.topk_mode != 0;
    if (!use_all) {
      // Candidates: each CTA sends its forced keys and about its cand_m
      // largest real keys (every key >= its threshold tau, with the
      // threshold itself); every CTA then selects the row's top k among the
      // cluster's candidates.  That selection is exact when the row's k-th
      // largest is >= every CTA's tau (nothing unsent can reach it), which
      // holds unless one CTA holds far more than its share of the row's top
      // k; otherwise every CTA falls back to the all-keys selection.
      const int cap = sa.cand_cap;
      uint32_t* scratch = reinterpret_cast<uint32_t*>(ring);
      uint2* cand = reinterpret_cast<uint2*>(ring + kTopkScratchBytes);  // [C][cap] (key, page) pairs
      // empty candidate slots read as key 0; once they are zeroed (and the
      // ring is free) the CTA arrives on the cluster barrier, and the other
      // CTAs write into them only after its wait, which comes after this
      // CTA's own threshold and compaction
      for (int i = threadIdx.x; i < C * cap / 2; i += NT) reinterpret_cast<uint4*>(cand)[i] = make_uint4(0u, 0u, 0u, 0u);
      __syncthreads();
      asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
      uint32_t kk[kLocalKeys];
      load_keys_reg<NT, kLocalKeys>(keys, nloc, kk);
      const uint32_t tau = top_bin_threshold<NT, kLocalKeys>(kk, sa.cand_m, scratch, scan_tmp);
      const int j0 = threadIdx.x * kLocalKeys;
      int cnt = 0;
#pragma unroll
      for (int j = 0; j < kLocalKeys; ++j) cnt += kk[j] >= tau;  // slots past nloc hold 0 < tau
      int total;
      const int off = block_scan_excl<NT>(cnt, scan_tmp, total);
      const bool ovf = total > cap;
      // compact into this CTA's own slots (its ring is free), then copy the
      // block to the other CTAs with coalesced 16-byte stores
      uint2* mine = cand + split * cap;  // 16-byte aligned: cap is even
      if (!ovf) {
        int o = off;
#pragma unroll
        for (int j = 0; j < kLocalKeys; ++j) {
          const bool in = kk[j] >= tau;
          if (in) mine[o] = make_uint2(kk[j], (uint32_t)(sa.chunk * split + j0 + j));
          o += in;
        }
      }
      __syncthreads();  // the compacted block is complete
      asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");  // every ring is free and zeroed
      if (threadIdx.x < C) {
        cl.map_shared_rank(s_cand_n, (int)threadIdx.x)[split] = ovf ? -1 : total;
        cl.map_shared_rank(s_cand_tau, (int)threadIdx.x)[split] = tau;
      }
      if (!ovf && C > 1) {
        const int n2 = (total + 1) >> 1;  // pairs of entries (the odd tail entry is past the count)
        const uint4* src = reinterpret_cast<const uint4*>(mine);
        for (int idx = threadIdx.x; idx < (C - 1) * n2; idx += NT) {
          const int cc = idx / n2, i = idx - cc * n2;
          const int c = cc + (cc >= split);
          reinterpret_cast<uint4*>(cl.map_shared_rank(cand, c) + split * cap)[i] = src[i];
        }
      }
      cl.sync();  // the cluster's candidates are delivered
      bool any_ovf = false;
      for (int c = 0; c < C; ++c) any_ovf |= s_cand_n[c] < 0;
      if (any_ovf) {
        use_all = true;  // the same in every CTA: the counts are the cluster's
      } else {
        const int slots = C * cap;
        bool okc;
        if (slots <= NT * 2) okc = select_share_cand<NT, 2>(cand, slots, C, s_cand_tau, k, scratch, e0, nent, list, scan_tmp);
        else if (slots <= NT * 4) okc = select_share_cand<NT, 4>(cand, slots, C, s_cand_tau, k, scratch, e0, nent, list, scan_tmp);
        else if (slots <= NT * 8) okc = select_share_cand<NT, 8>(cand, slots, C, s_cand_tau, k, scratch, e0, nent, list, scan_tmp);
        else if (slots <= NT * 16) okc = select_share_cand<NT, 16>(cand, slots, C, s_cand_tau, k, scratch, e0, nent, list, scan_tmp);
        else okc = select_share_cand<NT, 32>(cand, slots, C, s_cand_tau, k, scratch, e0, nent, list, scan_tmp);
        if (!okc) use_all = true;  // identical candidates everywhere: the same in every CTA
      }
    }
    if (use_all) {
      // every CTA receives the row's keys in its ring and selects locally
      if (split == 0 && threadIdx.x == 0) atomicAdd(&g_step_rows_all_keys, 1ull);
      cl.sync();  // every ring is free (and every candidate list read)
      uint32_t* allk = reinterpret_cast<uint32_t*>(ring);  // [NP] keys of the row, by page
      {
        const int n4 = nloc >> 2;
        const uint4* src4 = reinterpret_cast<const uint4*>(keys);
        for (int c = 0; c < C; ++c) {
          uint32_t* dst = cl.map_shared_rank(allk, c) + sa.chunk * split;  // 16-byte aligned: chunk % 16 == 0
          uint4* dst4 = reinterpret_cast<uint4*>(dst);
          for (int i = threadIdx.x; i < n4; i += NT) dst4[i] = src4[i];
          for (int i = 4 * n4 + threadIdx.x; i < nloc; i += NT) dst[i] = keys[i];
        }
      }
      cl.sync();  // the row's keys are complete in every CTA
      uint32_t* scratch = reinterpret_cast<uint32_t*>(ring + sa.scratch_off);
      bool done = false;
      if (NP <= NT * kRegKeys) done = select_share_reg<NT, kRegKeys>(allk, NP, k, scratch, e0, nent, list, scan_tmp);
      __syncthreads();
      if (!done) {
        uint32_t T;
        int take;
        local_topk<NT>(allk, NP, k, scratch, scan_tmp, T, take);
        // the list positions of the chosen pages; this CTA keeps [e0, e0 + nent)
        const int RUN = (NP + NT - 1) / NT;
        const int i_beg = min(NP, threadIdx.x * RUN), i_end = min(NP, i_beg + RUN);
        int gt = 0, eq = 0;
        for (int i = i_beg; i < i_end; ++i) {
          gt += allk[i] > T;
          eq += allk[i] == T;
        }
        int tot;
        const int excl = block_scan_excl<NT>((gt << 16) | eq, scan_tmp, tot);  // both totals < 2^15
        int Gp = excl >> 16, Ep = excl & 0xffff;
        for (int i = i_beg; i < i_end; ++i) {
          const uint32_t key = allk[i];
          int pos = -1;
          if (key > T) {
            pos = Gp + min(Ep, take);
            ++Gp;
          } else if (key == T) {
            if (Ep < take) pos = Gp + Ep;
            ++Ep;
          }
          if (pos >= e0 && pos < e0 + nent) list[pos - e0] = i;
        }
      }
    }
    __syncthreads();
    if (sa.page_idx)
      for (int e = threadIdx.x; e < nent; e += NT) sa.page_idx[(size_t)row * k + e0 + e] = list[e];
  } else {
    // every page of the context is chosen: 0 .. NP-1, then -1
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // completes the arrive made at entry
    int32_t* gout = sa.page_idx ? sa.page_idx + (size_t)row * k : nullptr;
    for (int e = threadIdx.x; e < nent; e += NT) {
      const int v = e0 + e < NP ? e0 + e : -1;
      list[e] = v;
      if (gout) gout[e0 + e] = v;
    }
  }
  fence_proxy_async_smem();  // scratch writes in the ring before the copies reuse it
  __syncthreads();

  // -------------------------------------------------------------- 3. attend
  // a sparse row: the CTA's share of the list; a dense row: its share of the
  // context's 16-token groups
  const int dper = (((NP << a.pshift) >> 4) + C - 1) / C;
  const int dg0 = split * dper;
  const int ngroups = dense ? max(0, min(dper, ((NP << a.pshift) >> 4) - dg0)) : (nent << a.pshift) >> 4;
  auto group_at = [&](int gi, int& lim) -> int {
    const int j0 = gi << 4;
    const int pg = dense ? ((dg0 + gi) << 4) >> a.pshift : list[j0 >> a.pshift];
    const int jo = dense ? ((dg0 + gi) << 4) : j0;
    lim = 0;
    if ((unsigned)pg >= (unsigned)(a.Cap >> a.pshift)) return 0;
    const int base = (pg << a.pshift) + (jo & (a.P - 1));
    lim = min(N - base, 16);
    return base;
  };
  float o[KS][4];
  float m_run = kNegInf, l_run = 0.f;
#pragma unroll
  for (int t = 0; t < KS; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
  // the wait-timeout test hook: CTA 0 announces bytes for its first attend
  // stage that it never requests, and its attend waits poll briefly
  const bool plant = a.test_wait && blockIdx.x == 0;
  const uint32_t tries = plant ? kTestWaitTries : kWaitTries;
  if (warp == W) {
    if (lane == 0) {
      int issued = 0;
      for (int gi = 0; gi < ngroups; ++gi) {
        const uint32_t q = seq + gi;
        const int st = q % NST;
        if (!producer_wait(q, tries)) {
          ok = false;
          break;
        }
        int lim;
        const int base = group_at(gi, lim);
        if (plant && gi == 0) {
          mbar_arrive_expect_tx(&full[st], 16);  // no copy is issued: this phase never completes
        } else if (lim > 0) {
          mbar_arrive_expect_tx(&full[st], L::STAGE);
          const int y = row * a.Cap + base;
          unsigned char* dst = ring + st * L::STAGE;
          tma_load_3d(dst, &tk, 0, y, 0, &full[st]);
          tma_load_3d(dst + L::GROUP, &tv, 0, y, 0, &full[st]);
        } else {
          mbar_arrive(&full[st]);
        }
        issued = gi + 1;
      }
      // every copy issued has landed before the ring is reused or left
      for (int gi = max(0, issued - NST); gi < issued; ++gi) {
        const uint32_t q = seq + gi;
        if (!mbar_wait(&full[q % NST], (q / NST) & 1, tries)) ok = false;
      }
      if (!ok) note_wait_timeout();
    }
  } else {
    const int r = lane >> 2, m = lane & 3;
    uint32_t qa[KS][2];
    const bf16* qp = static_cast<const bf16*>(a.q) + ((size_t)b * a.Hq + (size_t)h * G + r) * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qa[ks][0] = r < G ? __ldg(reinterpret_cast<const uint32_t*>(qp + 16 * ks + 2 * m)) : 0u;
      qa[ks][1] = r < G ? __ldg(reinterpret_cast<const uint32_t*>(qp + 16 * ks + 8 + 2 * m)) : 0u;
    }
    const uint32_t ring_u32 = smem_u32(ring);
    for (int gi = (W + warp - (int)(seq % W)) % W; gi < ngroups; gi += W) {
      const uint32_t q = seq + gi;
      const int st = q % NST;
      if (!mbar_wait(&full[st], (q / NST) & 1, tries)) {
        ok = false;
        break;
      }
      int lim;
      group_at(gi, lim);
      if (lim > 0) tma_group<D>(ring_u32 + st * L::STAGE, lim, qa, o, m_run, l_run, a.qscale, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) note_wait_timeout();
      // an infinite running max makes this warp's merge weight inf - inf = NaN
      // at every later merge, so the row's output and lse become NaN (a NaN
      // max would be dropped by fmaxf and the partial silently ignored)
      m_run = __int_as_float(0x7f800000);
    }
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    if (m == 0) {
      sM[warp][r] = m_run;
      sL[warp][r] = l_run;
    }
  }
  __syncthreads();

  // ------------------------------------------------------------- 4. combine
  float* sO = reinterpret_cast<float*>(ring);
  merge_warps<D, W>(o, G, sO, sM, sL, sF, sHm, sHl);
  cluster_push_combine<D, W, NT>(a, row, split, sO, sF, sHm, sHl, inbox, false);
}

// ---------------------------------------------------------------- host side

// Ring bytes the top-k needs: the row's keys, then its scratch.
static size_t topk_ring_bytes(int npcap) { return ((size_t)npcap * 4 + 15) / 16 * 16 + (size_t)kTopkScratchBytes; }

bool quest_step_eligible(const Shape& s, int k) {
  const long long npcap = s.Cap >> s.pshift;
  const size_t ring = s.D == 64 ? StepLayout<64>::RING_REGION : StepLayout<128>::RING_REGION;
  return s.dtype == 1 && !(s.flags & 3) && s.G <= 8 && s.P >= 16 && (s.D == 64 || s.D == 128) &&
         k <= kStepMaxK && (long long)s.B * s.Hkv * s.Cap < (1ll << 31) &&
         (long long)s.B * s.Hkv * npcap < (1ll << 31) && topk_ring_bytes((int)npcap) <= ring &&
         attend_tma_eligible(s);
}

template <int D>
static size_t step_smem(int chunk, int k) {
  const size_t keys = std::max((size_t)chunk * 4, sizeof(ClusterInbox<D>));
  const size_t keys_al = (keys + 15) / 16 * 16;
  return StepLayout<D>::RING_REGION + keys_al + (size_t)k * 4 + 1024;
}

template <int D>
static int step_max_clusters(int C, size_t smem) {
  cudaFuncSetAttribute(quest_step_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (C > 8) cudaFuncSetAttribute(quest_step_kernel<D>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C);
  cfg.blockDim = dim3((kTmaConsumers + 1) * 32);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, quest_step_kernel<D>, &cfg) != cudaSuccess) return -1;
  return n;
}

static int chunk_for(int npcap, int C) { return ((npcap + C - 1) / C + 15) / 16 * 16; }

// Cluster size: about two CTAs per SM over all rows, at most 16, each CTA
// scoring at most kStepMaxChunk pages, all clusters resident at once when
// that is possible.
int quest_step_splits(const Shape& s, int k) {
  const int rows = s.B * s.Hkv;
  const int npcap = s.Cap >> s.pshift;
  int C = std::min((2 * sm_count()) / rows + 1, kMaxClusterSplits);
  while (C < kMaxClusterSplits && chunk_for(npcap, C) > kStepMaxChunk) ++C;
  C = std::max(C, 1);
  while (C > 1) {
    const size_t smem = s.D == 64 ? step_smem<64>(chunk_for(npcap, C), k) : step_smem<128>(chunk_for(npcap, C), k);
    const int fit = s.D == 64 ? step_max_clusters<64>(C, smem) : step_max_clusters<128>(C, smem);
    if (fit < 0 || fit >= rows || (fit > 0 && rows > fit * 4)) break;  // unknown, one wave, or many waves
    if (chunk_for(npcap, C - 1) > kStepMaxChunk) break;
    --C;
  }
  return C;
}

template <int D>
static cudaError_t step_launch(const Shape& s, const StepArgs& sa0, cudaStream_t st, bool* handled) {
  StepArgs sa = sa0;
  const int C = sa.a.S;
  sa.chunk = chunk_for(sa.npcap, C);
  if (sa.chunk > kStepMaxChunk) return cudaSuccess;
  const size_t keys = std::max((size_t)sa.chunk * 4, sizeof(ClusterInbox<D>));
  sa.keys_bytes = (keys + 15) / 16 * 16;
  sa.scratch_off = (int)(((size_t)sa.npcap * 4 + 15) / 16 * 16);
  // candidate selection when a CTA's keys fit its registers and the lists fit the ring
  // a CTA holds about k / C of the row's chosen pages: it sends about twice
  // that (plus its forced pages), room for the rest of a histogram bin
  const int forced_max = sa.n_sink + (sa.n_local + s.P - 1) / s.P + 1;
  sa.cand_m = std::min(sa.k, (2 * sa.k + C - 1) / C + 8);
  sa.cand_cap = (sa.cand_m + forced_max + 16 + 1) / 2 * 2;  // even: 16-byte aligned per-CTA blocks
  const size_t cand_bytes = (size_t)kTopkScratchBytes + (size_t)8 * C * sa.cand_cap;
  sa.topk_mode = (sa.chunk <= (kTmaConsumers + 1) * 32 * kLocalKeys && cand_bytes <= StepLayout<D>::RING_REGION &&
                  C * sa.cand_cap <= (kTmaConsumers + 1) * 32 * kRegKeys)
                     ? 0
                     : 1;
  const size_t smem = step_smem<D>(sa.chunk, sa.k);
  if (smem > 227 * 1024) return cudaSuccess;
  if (step_max_clusters<D>(C, smem) <= 0) return cudaSuccess;
  const uint64_t rows = (uint64_t)s.B * s.Hkv;
  CUtensorMap tk, tv, tmin, tmax;
  if (!encode_rows_map(&tk, sa.a.k, rows * s.Cap, D) || !encode_rows_map(&tv, sa.a.v, rows * s.Cap, D) ||
      !encode_rows_map(&tmin, sa.kmin, rows * sa.npcap, D) || !encode_rows_map(&tmax, sa.kmax, rows * sa.npcap, D))
    return cudaSuccess;
  *handled = true;
  cudaError_t e = launch_pdl_cluster(quest_step_kernel<D>, dim3((unsigned)(rows * C)), dim3((kTmaConsumers + 1) * 32),
                                     smem, C, st, tk, tv, tmin, tmax, sa);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_quest_step(const Shape& s, const void* q, const void* k_cache, const void* v_cache,
                              const void* kmin, const void* kmax, const int32_t* ctx_len, int k, int n_sink,
                              int n_local, const float* sink, int32_t* page_idx, void* out, float* lse,
                              int num_splits, float min_sparsity, cudaStream_t st, bool* handled) {
  *handled = false;
  if (!quest_step_eligible(s, k)) return cudaSuccess;
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
       reinterpret_cast<uintptr_t>(kmin) | reinterpret_cast<uintptr_t>(kmax)) & 15)
    return cudaSuccess;
  StepArgs sa = {};
  AttendArgs& a = sa.a;
  a.q = q;
  a.k = k_cache;
  a.v = v_cache;
  sa.kmin = kmin;
  sa.kmax = kmax;
  a.ctx_len = ctx_len;
  a.Hq = s.Hq; a.Hkv = s.Hkv; a.G = s.G; a.Cap = s.Cap; a.P = s.P; a.pshift = s.pshift;
  a.qscale = s.scale * kLog2e;
  a.sink = sink;
  a.out = out;
  a.lse = lse;
  a.cluster = 1;
  a.test_wait = (s.flags & kFlagTestWaitTimeout) ? 1 : 0;
  a.S = num_splits > 0 ? std::min(num_splits, kMaxClusterSplits) : quest_step_splits(s, k);
  sa.page_idx = page_idx;
  sa.k = k;
  sa.n_sink = n_sink;
  sa.n_local = n_local;
  sa.npcap = s.Cap >> s.pshift;
  sa.min_sparsity = min_sparsity;
  return s.D == 64 ? step_launch<64>(s, sa, st, handled) : step_launch<128>(s, sa, st, handled);
}

void take_step_row_stats(unsigned long long* dense, unsigned long long* all_keys, bool reset) {
  *dense = *all_keys = 0;
  if (cudaMemcpyFromSymbol(dense, g_step_rows_dense, sizeof(*dense)) != cudaSuccess ||
      cudaMemcpyFromSymbol(all_keys, g_step_rows_all_keys, sizeof(*all_keys)) != cudaSuccess) {
    *dense = *all_keys = 0;
    return;
  }
  if (reset) {
    const unsigned long long zero = 0;
    cudaMemcpyToSymbol(g_step_rows_dense, &zero, sizeof(zero));
    cudaMemcpyToSymbol(g_step_rows_all_keys, &zero, sizeof(zero));
  }
}

DeviceStatus take_status_quest_step() { return take_status_here(); }

}  // namespace sls
