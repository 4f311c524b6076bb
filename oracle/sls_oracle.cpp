// fp64 CPU oracle for sparse decode attention (select + attend), plain C++17.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the library includes, links or calls
// this file; only the test suite, the smoke check and the benchmark's CPU
// baseline do (through oracle/sls_oracle.py).  It shares no code with the
// CUDA path: it decodes bf16 itself, builds its own page summaries and
// thumbnails from the keys, and indexes the cache layout itself.  Every value
// is a double holding the exact value of a bf16/fp32 input, and every step is
// a plain loop over the definition it cites, with no blocking or reordering.
//
// Sources (web pages; cited by title and section):
//   [haystack]  "Don't read the haystack", Part one (two-stage
//               flash-decoding) and Part two (per-page min/max bound, top-k,
//               sink page and local pages); Part three (attention mass).
//   [ffd]       "Faster Than Flash: Exploiting Attention Sparsity for
//               Efficient Long-Context Decoding", Methodology 1 (2-bit
//               mid-rise thumbnails, 8-bit residuals), 2 (top-delta,
//               eqs. 1-3) and 3 (eq. 4: scaling and refined final scores).
//   [undivided] "Attention: Undivided & Uncompressed", Notation
//               (S = QK^T / sqrt(d)) and Traffic (online softmax).
//   [tsd]       "Training-free sparse attention for long-context LLM
//               decode", section 1 (learned sink as a virtual key, V = 0).
//   [mlxcel]    "perf(core): fused sparse-attention decode via page
//               indirection", "The reduction" (contiguous cache as a page
//               pool) and "Corrected premise 1" (one page list per KV head).
//
// Parity status: every function is pinned by tests/test_oracle_pins.py
// (hand-worked fixtures, brute force, closed forms, invariants) and by a
// source-mutation check (tests/test_oracle_mutations_cpp.py); none is "parity
// unpinned".
//
// Conventions: matrices are row-major doubles; q is [G, D], a key or value
// row block is [T, D]; page and token indices are int64.  Functions that
// return a variable number of indices write them into a caller buffer sized
// for the worst case and return the count.

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

typedef long long i64;

static const double kNegInf = -std::numeric_limits<double>::infinity();
static const double kPosInf = std::numeric_limits<double>::infinity();
// Residual denominator: codes -127..127 span the +-s/4 quantisation error.
static const double kResDenom = 508.0;

extern "C" {

// ---------------------------------------------------------------------------
// input decoding
// ---------------------------------------------------------------------------

// bf16 is the upper half of an IEEE binary32: widen the bit pattern, then the
// float to double (both exact).
void orc_bf16_to_f64(const uint16_t* bits, i64 n, double* out) {
  for (i64 i = 0; i < n; ++i) {
    uint32_t u = (uint32_t)bits[i] << 16;
    float f;
    std::memcpy(&f, &u, sizeof f);
    out[i] = (double)f;
  }
}

void orc_f32_to_f64(const float* x, i64 n, double* out) {
  for (i64 i = 0; i < n; ++i) out[i] = (double)x[i];
}

// ---------------------------------------------------------------------------
// attention: the plain definitions
// ---------------------------------------------------------------------------

static double dot(const double* a, const double* b, int D) {
  double s = 0.0;
  for (int c = 0; c < D; ++c) s += a[c] * b[c];
  return s;
}

// Exact softmax attention of G query rows over T keys.
// [undivided] Notation: scores x = scale * q.k (scale = 1/sqrt(d)), P the
// row softmax, O = P V.  [tsd] section 1: a learned per-head sink is a scalar
// logit that joins only the softmax denominator (a virtual key whose value is
// zero).  Reading: the sink is a raw logit, not multiplied by scale.
// q [G, Dq], K [T, Dq], V [T, Dv]; sink [G] or null.  o [G, Dv], lse [G].
// T = 0 gives o = 0 and lse = the sink (-inf without one).
void orc_softmax_attention(const double* q, int G, int Dq, const double* K, const double* V, i64 T,
                           int Dv, double scale, const double* sink, double* o, double* lse) {
  std::vector<double> x((size_t)T);
  for (int g = 0; g < G; ++g) {
    double* og = o + (i64)g * Dv;
    for (int c = 0; c < Dv; ++c) og[c] = 0.0;
    double m = kNegInf;
    for (i64 t = 0; t < T; ++t) {
      x[t] = scale * dot(q + (i64)g * Dq, K + t * Dq, Dq);
      m = std::max(m, x[t]);
    }
    if (sink) m = std::max(m, sink[g]);
    if (m == kNegInf) {
      lse[g] = kNegInf;
      continue;
    }
    double z = 0.0;
    for (i64 t = 0; t < T; ++t) {
      double w = std::exp(x[t] - m);
      z += w;
      for (int c = 0; c < Dv; ++c) og[c] += w * V[t * Dv + c];
    }
    if (sink) z += std::exp(sink[g] - m);
    for (int c = 0; c < Dv; ++c) og[c] /= z;
    lse[g] = m + std::log(z);
  }
}

// Stage one of two-stage flash-decoding ([haystack] Part one): for each slice
// [a, b) of the keys (bounds holds S pairs), the slice max m, the normaliser
// l = sum exp(x - m) and the unnormalised accumulator acc = sum exp(x - m) v.
// An empty slice gives m = -inf, l = 0, acc = 0.
// m, l [S, G]; acc [S, G, Dv].
void orc_split_partials(const double* q, int G, int Dq, const double* K, const double* V, int Dv,
                        double scale, const i64* bounds, int S, double* m, double* l, double* acc) {
  for (int s = 0; s < S; ++s) {
    i64 a = bounds[2 * s], b = bounds[2 * s + 1];
    for (int g = 0; g < G; ++g) {
      double* ms = m + (i64)s * G + g;
      double* ls = l + (i64)s * G + g;
      double* as = acc + ((i64)s * G + g) * Dv;
      for (int c = 0; c < Dv; ++c) as[c] = 0.0;
      *ms = kNegInf;
      *ls = 0.0;
      if (b <= a) continue;
      for (i64 t = a; t < b; ++t) *ms = std::max(*ms, scale * dot(q + (i64)g * Dq, K + t * Dq, Dq));
      for (i64 t = a; t < b; ++t) {
        double w = std::exp(scale * dot(q + (i64)g * Dq, K + t * Dq, Dq) - *ms);
        *ls += w;
        for (int c = 0; c < Dv; ++c) as[c] += w * V[t * Dv + c];
      }
    }
  }
}

// Stage two ([haystack] Part one; [undivided] Traffic): rescale every partial
// by exp(m_s - M), M the overall max including the sink, sum, and divide once
// at the end.  The sink joins the denominator once.  Empty partials
// (m = -inf) contribute nothing.
void orc_combine_partials(int S, int G, int D, const double* m, const double* l, const double* acc,
                          const double* sink, double* o, double* lse) {
  for (int g = 0; g < G; ++g) {
    double* og = o + (i64)g * D;
    for (int c = 0; c < D; ++c) og[c] = 0.0;
    double M = kNegInf;
    for (int s = 0; s < S; ++s) M = std::max(M, m[(i64)s * G + g]);
    if (sink) M = std::max(M, sink[g]);
    if (M == kNegInf) {
      lse[g] = kNegInf;
      continue;
    }
    double L = 0.0;
    for (int s = 0; s < S; ++s) {
      double ms = m[(i64)s * G + g];
      if (ms == kNegInf) continue;
      double f = std::exp(ms - M);
      L += l[(i64)s * G + g] * f;
      const double* as = acc + ((i64)s * G + g) * D;
      for (int c = 0; c < D; ++c) og[c] += as[c] * f;
    }
    if (sink) L += std::exp(sink[g] - M);
    for (int c = 0; c < D; ++c) og[c] /= L;
    lse[g] = M + std::log(L);
  }
}

// ---------------------------------------------------------------------------
// Quest page selection
// ---------------------------------------------------------------------------

i64 orc_num_pages(i64 n, i64 page_size) { return (n + page_size - 1) / page_size; }

// Per-page, per-channel min and max of the keys of one (b, kv head) row
// ([haystack] Part two: each page keeps the elementwise min and max of its
// keys).  Only positions < n count, so a partial last page summarises its
// valid tokens.  K [>= n, D]; kmin, kmax [NP, D].
void orc_page_minmax(const double* K, int D, i64 n, int P, double* kmin, double* kmax) {
  i64 NP = orc_num_pages(n, P);
  for (i64 p = 0; p < NP; ++p) {
    i64 t0 = p * P, t1 = std::min(t0 + P, n);
    for (int c = 0; c < D; ++c) {
      double lo = kPosInf, hi = kNegInf;
      for (i64 t = t0; t < t1; ++t) {
        lo = std::min(lo, K[t * D + c]);
        hi = std::max(hi, K[t * D + c]);
      }
      kmin[p * D + c] = lo;
      kmax[p * D + c] = hi;
    }
  }
}

// Upper bound of every page's attention score for every query head
// ([haystack] Part two): U[g, p] = sum_c max(q[g,c] * kmin[p,c],
// q[g,c] * kmax[p,c]).  Unscaled: the ranking is invariant to the positive
// softmax scale.  U [G, NP].
void orc_quest_bound(const double* q, int G, int D, const double* kmin, const double* kmax, i64 NP,
                     double* U) {
  for (int g = 0; g < G; ++g)
    for (i64 p = 0; p < NP; ++p) {
      double u = 0.0;
      for (int c = 0; c < D; ++c) {
        double a = q[(i64)g * D + c] * kmin[p * D + c];
        double b = q[(i64)g * D + c] * kmax[p * D + c];
        u += std::max(a, b);
      }
      U[(i64)g * NP + p] = u;
    }
}

// One page list per (batch, KV head), shared by the query heads of the group
// ([mlxcel] "Corrected premise 1").  Reading: the group's score of a page is
// the max over its heads, which keeps the bound admissible for every head.
void orc_group_score(const double* U, int G, i64 NP, double* score) {
  for (i64 p = 0; p < NP; ++p) {
    double s = kNegInf;
    for (int g = 0; g < G; ++g) s = std::max(s, U[(i64)g * NP + p]);
    score[p] = s;
  }
}

// Pages kept regardless of score ([haystack] Part two: the attention-sink
// page plus the last few local pages): the first n_sink_pages pages and every
// page holding one of the last n_local_tokens positions.  Ascending, unique.
// out holds up to NP entries; returns the count.
i64 orc_forced_pages(i64 n, int P, int n_sink_pages, int n_local_tokens, i64* out) {
  i64 NP = orc_num_pages(n, P);
  std::vector<char> f((size_t)NP, 0);
  for (i64 p = 0; p < std::min((i64)n_sink_pages, NP); ++p) f[p] = 1;
  if (n_local_tokens > 0 && n > 0)
    for (i64 p = std::max(n - (i64)n_local_tokens, (i64)0) / P; p < NP; ++p) f[p] = 1;
  i64 cnt = 0;
  for (i64 p = 0; p < NP; ++p)
    if (f[p]) out[cnt++] = p;
  return cnt;
}

// The non-forced pages ranked by score, descending, ties to the lower index.
static std::vector<i64> ranked_free_pages(const double* score, i64 NP, const i64* forced, i64 nf) {
  std::vector<char> isf((size_t)NP, 0);
  for (i64 i = 0; i < nf; ++i) isf[forced[i]] = 1;
  std::vector<i64> cand;
  for (i64 p = 0; p < NP; ++p)
    if (!isf[p]) cand.push_back(p);
  std::sort(cand.begin(), cand.end(), [&](i64 a, i64 b) {
    if (score[a] != score[b]) return score[a] > score[b];
    return a < b;
  });
  return cand;
}

// Top-k selection with forced pages ([haystack] Part two: rank pages by the
// bound, keep the top k together with the forced pages).  Readings: the
// budget k counts the forced pages (the list has a fixed cardinality of
// min(k, NP)); among equal scores the lower page index wins; the list is
// ascending.  Returns the count written to out (<= max(k, NP) entries), or -1
// when the forced pages exceed the budget.
i64 orc_select_topk(const double* score, i64 NP, i64 k, const i64* forced, i64 nf, i64* out) {
  if (NP <= k) {
    for (i64 p = 0; p < NP; ++p) out[p] = p;
    return NP;
  }
  if (nf > k) return -1;
  std::vector<i64> cand = ranked_free_pages(score, NP, forced, nf);
  i64 cnt = 0;
  for (i64 i = 0; i < nf; ++i) out[cnt++] = forced[i];
  for (i64 i = 0; i < k - nf && i < (i64)cand.size(); ++i) out[cnt++] = cand[i];
  std::sort(out, out + cnt);
  return cnt;
}

// Score of the last candidate admitted by orc_select_topk (the (k - nf)-th
// ranked free page), used to recognise boundary ties: -inf when every page
// fits, +inf when the forced pages fill the budget.
double orc_kth_score(const double* score, i64 NP, i64 k, const i64* forced, i64 nf) {
  if (NP <= k) return kNegInf;
  i64 kk = k - nf;
  if (kk <= 0) return kPosInf;
  std::vector<i64> cand = ranked_free_pages(score, NP, forced, nf);
  return score[cand[kk - 1]];
}

// Token positions of the given pages, in list order, restricted to positions
// < n ([mlxcel] "The reduction": token i of page p is position p * P + i);
// negative entries (padding) are skipped.  Returns the count.
i64 orc_pages_to_tokens(const i64* pages, i64 npages, i64 n, int P, i64* out) {
  i64 cnt = 0;
  for (i64 i = 0; i < npages; ++i) {
    i64 p = pages[i];
    if (p < 0) continue;
    for (i64 t = p * P; t < std::min((p + 1) * P, n); ++t) out[cnt++] = t;
  }
  return cnt;
}

// Selection of one row: page summaries -> bound -> group max -> forced
// pages -> top-k.  A one-token page (P = 1) has kmin = kmax = its key, so the
// bound is the exact score q.k.  pages_out holds max(k, NP) entries,
// score_out NP; *kth_out receives the k-th admitted score.  Returns the list
// length, or -1 when the forced pages exceed the budget.
i64 orc_quest_select_row(const double* q, int G, int D, const double* K, i64 n, int P, i64 k,
                         int n_sink_pages, int n_local_tokens, i64* pages_out, double* score_out,
                         double* kth_out) {
  i64 NP = orc_num_pages(n, P);
  std::vector<double> kmin, kmax;
  const double *lo = K, *hi = K;
  if (P != 1) {
    kmin.resize((size_t)(NP * D));
    kmax.resize((size_t)(NP * D));
    orc_page_minmax(K, D, n, P, kmin.data(), kmax.data());
    lo = kmin.data();
    hi = kmax.data();
  }
  std::vector<double> U((size_t)(G * NP));
  orc_quest_bound(q, G, D, lo, hi, NP, U.data());
  orc_group_score(U.data(), G, NP, score_out);
  std::vector<i64> forced((size_t)NP + 1);
  i64 nf = orc_forced_pages(n, P, n_sink_pages, n_local_tokens, forced.data());
  *kth_out = orc_kth_score(score_out, NP, k, forced.data(), nf);
  return orc_select_topk(score_out, NP, k, forced.data(), nf, pages_out);
}

// ---------------------------------------------------------------------------
// FFD thumbnails and top-delta
// ---------------------------------------------------------------------------

// 2-bit symmetric zero-free (mid-rise) thumbnail of one block of keys ([ffd]
// Methodology 1): s[c] = max_t |k[t,c]|; levels -0.75s, -0.25s, +0.25s,
// +0.75s (codes 0..3) with decision thresholds -s/2, 0, +s/2.  Readings: a
// value on a threshold takes the upper level (k = 0 -> +0.25s, k = s/2 ->
// +0.75s); an all-zero channel (s = 0) takes code 3, whose level is 0.
// Kb [T, D] -> codes [T, D], s [D].
void orc_thumb_quantize(const double* Kb, int T, int D, uint8_t* codes, double* s) {
  for (int c = 0; c < D; ++c) {
    double m = 0.0;
    for (int t = 0; t < T; ++t) m = std::max(m, std::fabs(Kb[(i64)t * D + c]));
    s[c] = m;
  }
  for (int t = 0; t < T; ++t)
    for (int c = 0; c < D; ++c) {
      double k = Kb[(i64)t * D + c], h = s[c] / 2.0;
      codes[(i64)t * D + c] = k >= h ? 3 : (k >= 0.0 ? 2 : (k >= -h ? 1 : 0));
    }
}

// Level of each code: (code - 1.5) * s / 2.  s holds one row of D scales
// (s_rows = 1) or one row per code row (s_rows = T).
void orc_thumb_dequant(const uint8_t* codes, const double* s, int T, int D, int s_rows, double* out) {
  for (int t = 0; t < T; ++t)
    for (int c = 0; c < D; ++c) {
      double sc = s[(s_rows == 1 ? 0 : (i64)t * D) + c];
      out[(i64)t * D + c] = ((double)codes[(i64)t * D + c] - 1.5) * (sc / 2.0);
    }
}

// Storage format of the thumbnails: four 2-bit codes per byte, channel c in
// bits 2 * (c % 4) of byte c / 4.  codes [T, D] -> packed [T, D/4].
void orc_pack_codes(const uint8_t* codes, int T, int D, uint8_t* packed) {
  for (int t = 0; t < T; ++t)
    for (int w = 0; w < D / 4; ++w) {
      unsigned b = 0;
      for (int j = 0; j < 4; ++j) b |= (unsigned)(codes[(i64)t * D + 4 * w + j] & 3) << (2 * j);
      packed[(i64)t * (D / 4) + w] = (uint8_t)b;
    }
}

void orc_unpack_codes(const uint8_t* packed, int T, int W, uint8_t* codes) {
  for (int t = 0; t < T; ++t)
    for (int w = 0; w < W; ++w)
      for (int j = 0; j < 4; ++j)
        codes[(i64)t * 4 * W + 4 * w + j] = (uint8_t)((packed[(i64)t * W + w] >> (2 * j)) & 3);
}

// Thumbnails of every complete block of one row (positions < n): codes
// [nfull * block, D] unpacked, scales [nfull, D].
void orc_thumbnails_row(const double* K, int D, i64 n, int block, uint8_t* codes, double* scales) {
  i64 nfull = n / block;
  for (i64 j = 0; j < nfull; ++j)
    orc_thumb_quantize(K + j * block * D, block, D, codes + j * block * D, scales + j * D);
}

// Blocks always kept by top-delta: block 0 (the sink tokens, S_global) and
// the block of the newest position (S_local, possibly partial).  Reading:
// [ffd] eq. 3 names S_global and S_local without sizes; here they are the
// first and the last block.  Returns the count (0, 1 or 2), ascending.
i64 orc_delta_forced_blocks(i64 n, int block, i64* out) {
  if (n <= 0) return 0;
  i64 last = (n - 1) / block;
  out[0] = 0;
  if (last == 0) return 1;
  out[1] = last;
  return 2;
}

// [ffd] eq. 3: m~ = max of the exact scores scale * q.k over the tokens of
// the sink and local blocks.  -inf for an empty context.  out [G].
void orc_pseudo_max(const double* q, int G, int D, const double* K, i64 n, int block, double scale,
                    double* out) {
  i64 fb[2];
  i64 nb = orc_delta_forced_blocks(n, block, fb);
  std::vector<i64> toks((size_t)(2 * block));
  i64 nt = orc_pages_to_tokens(fb, nb, n, block, toks.data());
  for (int g = 0; g < G; ++g) {
    double m = kNegInf;
    for (i64 i = 0; i < nt; ++i) m = std::max(m, scale * dot(q + (i64)g * D, K + toks[i] * D, D));
    out[g] = m;
  }
}

// Margin of one complete block from its thumbnail: max over heads g and
// tokens t of (s~[g,t] - m~[g]) with s~ = scale * q . k^ ([ffd] eq. 1 with the
// pseudo-max of eq. 3 in place of m; eq. 4 fixes the 1/sqrt(d) scaling).
static double block_margin(const double* q, int G, int D, const uint8_t* codes, const double* s,
                           int block, double scale, const double* mt) {
  std::vector<double> kh((size_t)block * D);
  orc_thumb_dequant(codes, s, block, D, 1, kh.data());
  double best = kNegInf;
  for (int g = 0; g < G; ++g)
    for (int t = 0; t < block; ++t)
      best = std::max(best, scale * dot(q + (i64)g * D, kh.data() + (i64)t * D, D) - mt[g]);
  return best;
}

// For every complete, non-forced block j of the row, the block margin
// (Readings: a block's score is the max over its tokens; a GQA group keeps
// the union over its heads, i.e. the max over g).  Writes the scanned blocks
// and their margins (each up to n / block entries); returns the count.
i64 orc_delta_block_margin(const double* q, int G, int D, const double* K, i64 n, int block,
                           double scale, i64* blocks, double* margins) {
  i64 nfull = n / block;
  i64 fb[2];
  i64 nb = orc_delta_forced_blocks(n, block, fb);
  std::vector<double> mt((size_t)G);
  orc_pseudo_max(q, G, D, K, n, block, scale, mt.data());
  std::vector<uint8_t> codes((size_t)block * D);
  std::vector<double> s((size_t)D);
  i64 cnt = 0;
  for (i64 j = 0; j < nfull; ++j) {
    bool forced = false;
    for (i64 i = 0; i < nb; ++i) forced = forced || fb[i] == j;
    if (forced) continue;
    orc_thumb_quantize(K + j * block * D, block, D, codes.data(), s.data());
    blocks[cnt] = j;
    margins[cnt] = block_margin(q, G, D, codes.data(), s.data(), block, scale, mt.data());
    ++cnt;
  }
  return cnt;
}

// Top-delta selection of one row ([ffd] eqs. 1-3): a complete block is kept
// when its margin is >= -delta; the forced blocks are always kept.  sel holds
// up to ceil(n / block) entries (ascending); blocks and margins receive the
// scanned blocks (count in *nscan).  Returns the list length.
i64 orc_delta_select_row(const double* q, int G, int D, const double* K, i64 n, int block, double delta,
                         double scale, i64* sel, i64* blocks, double* margins, i64* nscan) {
  i64 ns = orc_delta_block_margin(q, G, D, K, n, block, scale, blocks, margins);
  *nscan = ns;
  i64 fb[2];
  i64 nb = orc_delta_forced_blocks(n, block, fb);
  i64 cnt = 0;
  for (i64 i = 0; i < nb; ++i) sel[cnt++] = fb[i];
  for (i64 i = 0; i < ns; ++i)
    if (margins[i] >= -delta) sel[cnt++] = blocks[i];
  std::sort(sel, sel + cnt);
  return cnt;
}

// ---------------------------------------------------------------------------
// FFD 8-bit residuals and the refined scores (eq. 4)
// ---------------------------------------------------------------------------

// 8-bit residual of one complete block ([ffd] Methodology 1: the key splits
// into the 2-bit thumbnail k_quant and an 8-bit residual k_res that recovers
// the precision the thumbnail drops).  Reading (the page gives no encoding):
// the residual e = k - k^ of a mid-rise code lies in [-s/4, s/4], so it is
// stored on the thumbnail's block/channel scale s as r = the integer nearest
// to e * 508 / s (ties to even), in [-127, 127]; s = 0 gives 0.
//
// The decision is exact: for bf16 k and s the quotient is 508 k / s minus an
// integer, and k / s is a ratio of 8-bit integers times a power of two, so
// unless it sits exactly on a half-integer it lies at least 2^-19 (relative)
// away from one, far beyond the rounding of the fp64 subtraction, product and
// quotient below; an exact half-integer is computed exactly and rounds to
// even.  Kb [T, D], codes [T, D], s [D] -> r [T, D].
void orc_residual_quantize(const double* Kb, const uint8_t* codes, const double* s, int T, int D,
                           int8_t* r) {
  for (int t = 0; t < T; ++t)
    for (int c = 0; c < D; ++c) {
      i64 i = (i64)t * D + c;
      if (!(s[c] > 0.0)) {
        r[i] = 0;
        continue;
      }
      double kh = ((double)codes[i] - 1.5) * (s[c] / 2.0);
      double x = (Kb[i] - kh) * kResDenom / s[c];
      double j = std::nearbyint(x);  // round half to even (default rounding mode)
      r[i] = (int8_t)std::max(-127.0, std::min(127.0, j));
    }
}

// The key the refinement scores with: k~ = k^ + r * s / 508, so that
// q . k~ = q . k_quant + q . k_res ([ffd] eq. 4 numerator).  s as in
// orc_thumb_dequant.
void orc_refined_keys(const uint8_t* codes, const double* s, const int8_t* r, int T, int D, int s_rows,
                      double* out) {
  orc_thumb_dequant(codes, s, T, D, s_rows, out);
  for (int t = 0; t < T; ++t)
    for (int c = 0; c < D; ++c) {
      double sc = s[(s_rows == 1 ? 0 : (i64)t * D) + c];
      out[(i64)t * D + c] += (double)r[(i64)t * D + c] * (sc / kResDenom);
    }
}

// Codes, scales and residuals of every complete block of one row: codes and
// res [nfull * block, D], scales [nfull, D].
void orc_residuals_row(const double* K, int D, i64 n, int block, uint8_t* codes, double* scales,
                       int8_t* res) {
  orc_thumbnails_row(K, D, n, block, codes, scales);
  for (i64 j = 0; j < n / block; ++j)
    orc_residual_quantize(K + j * block * D, codes + j * block * D, scales + j * D, block, D,
                          res + j * block * D);
}

// Attention over the listed blocks with the refined final scores of [ffd]
// Methodology 3 step 3, eq. 4: s = (q . k_quant + q . k_res) / sqrt(d) for
// the tokens of complete blocks.  Reading: the newest block is partial and
// has no thumbnail yet, so its tokens are scored with the exact key; values
// are exact.  K, V [>= n, D].
void orc_refined_attention_row(const double* q, int G, int D, const double* K, const double* V,
                               const i64* blocks, i64 nblocks, i64 n, int block, double scale,
                               const double* sink, double* o, double* lse) {
  std::vector<i64> toks((size_t)(nblocks * block + 1));
  i64 nt = orc_pages_to_tokens(blocks, nblocks, n, block, toks.data());
  i64 nfull = n / block;
  std::vector<double> Kt((size_t)(nt * D + 1)), Vt((size_t)(nt * D + 1));
  std::vector<uint8_t> codes((size_t)block * D);
  std::vector<double> s((size_t)D), kref((size_t)block * D);
  std::vector<int8_t> r((size_t)block * D);
  i64 cached = -1;  // block whose refined keys sit in kref
  for (i64 i = 0; i < nt; ++i) {
    i64 t = toks[i], j = t / block;
    const double* src = K + t * D;
    if (j < nfull) {
      if (cached != j) {
        orc_thumb_quantize(K + j * block * D, block, D, codes.data(), s.data());
        orc_residual_quantize(K + j * block * D, codes.data(), s.data(), block, D, r.data());
        orc_refined_keys(codes.data(), s.data(), r.data(), block, D, 1, kref.data());
        cached = j;
      }
      src = kref.data() + (t - j * block) * D;
    }
    for (int c = 0; c < D; ++c) {
      Kt[i * D + c] = src[c];
      Vt[i * D + c] = V[t * D + c];
    }
  }
  orc_softmax_attention(q, G, D, Kt.data(), Vt.data(), nt, D, scale, sink, o, lse);
}

// ---------------------------------------------------------------------------
// selection quality
// ---------------------------------------------------------------------------

// Share of each query head's full-context softmax mass that falls on the
// tokens of the listed pages ([haystack] Part three, attention mass captured
// by the selection): recall_g = sum_{t in sel} exp(x_gt - M_g) /
// sum_{t < n} exp(x_gt - M_g), x = scale * q.k, M the row max.  Readings: the
// sink is not a token and takes no part; an empty context misses nothing
// (recall 1); -1 entries and positions >= n are ignored.  out [G].
void orc_attention_mass_recall(const double* q, int G, int D, const double* K, const i64* pages,
                               i64 npages, i64 n, int P, double scale, double* out) {
  if (n == 0) {
    for (int g = 0; g < G; ++g) out[g] = 1.0;
    return;
  }
  std::vector<i64> toks((size_t)(npages * P + 1));
  i64 nt = orc_pages_to_tokens(pages, npages, n, P, toks.data());
  std::vector<double> x((size_t)n);
  for (int g = 0; g < G; ++g) {
    double m = kNegInf;
    for (i64 t = 0; t < n; ++t) {
      x[t] = scale * dot(q + (i64)g * D, K + t * D, D);
      m = std::max(m, x[t]);
    }
    double all = 0.0, sel = 0.0;
    for (i64 t = 0; t < n; ++t) all += std::exp(x[t] - m);
    for (i64 i = 0; i < nt; ++i) sel += std::exp(x[toks[i]] - m);
    out[g] = sel / all;
  }
}

// ---------------------------------------------------------------------------
// one decode step of one row
// ---------------------------------------------------------------------------

// Attention restricted to the tokens of the listed pages ([haystack] Part
// two: the sparse twin attends over the selected indices only).
void orc_sparse_attention_row(const double* q, int G, int D, const double* K, const double* V,
                              const i64* pages, i64 npages, i64 n, int P, double scale,
                              const double* sink, double* o, double* lse) {
  std::vector<i64> toks((size_t)(npages * P + 1));
  i64 nt = orc_pages_to_tokens(pages, npages, n, P, toks.data());
  std::vector<double> Kt((size_t)(nt * D + 1)), Vt((size_t)(nt * D + 1));
  for (i64 i = 0; i < nt; ++i)
    for (int c = 0; c < D; ++c) {
      Kt[i * D + c] = K[toks[i] * D + c];
      Vt[i * D + c] = V[toks[i] * D + c];
    }
  orc_softmax_attention(q, G, D, Kt.data(), Vt.data(), nt, D, scale, sink, o, lse);
}

// ---------------------------------------------------------------------------
// whole decode steps over many rows (the timed CPU baseline)
// ---------------------------------------------------------------------------

}  // extern "C"

// Runs body(i) for i in [0, count) on nthreads std::threads.
template <typename F>
static void parallel_rows(int count, int nthreads, F body) {
  std::atomic<int> next(0);
  auto worker = [&]() {
    for (int i = next++; i < count; i = next++) body(i);
  };
  std::vector<std::thread> pool;
  for (int w = 1; w < std::max(nthreads, 1); ++w) pool.emplace_back(worker);
  worker();
  for (auto& th : pool) th.join();
}

static double now_s() {
  return std::chrono::duration<double>(std::chrono::steady_clock::now().time_since_epoch()).count();
}

// n elements from position off of a bf16 (bit patterns) or fp32 tensor, as doubles.
static void load(const void* base, int f32, i64 off, i64 n, double* out) {
  if (f32)
    orc_f32_to_f64((const float*)base + off, n, out);
  else
    orc_bf16_to_f64((const uint16_t*)base + off, n, out);
}

extern "C" {

// The Quest decode step on a workload, row by row: for every listed
// (b, kv head) row, decode its keys and build the page summaries (untimed
// preparation: the summaries are kept current at append time), then repeat,
// until min_busy seconds have passed, the timed select + attend: decode the
// group's queries, bound every page from the summaries, take the group max,
// the forced pages and the top k, decode the selected tokens' keys and
// values, and attend over them (with the sink, if given).
//   q [B, Hq, D], K and V [B, Hkv, Cap, D]: bf16 bit patterns, or fp32 when
//   f32 != 0; ctx_len [B];
//   sink [Hq] fp32 or null; rows: row ids b * Hkv + h.
//   pages_out [nrows, k] (-1 padded), o_out [nrows, G, D], lse_out [nrows, G].
//   stats_out: {busy seconds summed over rows, bytes (page summaries +
//   selected K and V in the input's element size, per repetition, summed),
//   repetitions}.
// Returns 0, or -1 when a row's forced pages exceed the budget.
int orc_quest_step(const void* q, const void* K, const void* V, int f32, const int32_t* ctx_len,
                        int B, int Hq, int Hkv, int D, i64 Cap, int P, int k, int n_sink_pages,
                        int n_local_tokens, double scale, const float* sink, const int32_t* rows,
                        int nrows, int nthreads, double min_busy, int32_t* pages_out, double* o_out,
                        double* lse_out, double* stats_out) {
  (void)B;
  const int G = Hq / Hkv;
  std::vector<double> busy((size_t)nrows, 0.0), bytes((size_t)nrows, 0.0), reps((size_t)nrows, 0.0);
  std::atomic<int> bad(0);
  parallel_rows(nrows, nthreads, [&](int i) {
    const int r = rows[i], b = r / Hkv, h = r % Hkv;
    const i64 n = ctx_len[b], NP = orc_num_pages(n, P);
    const i64 row0 = (i64)r * Cap * D;  // the row's first key element
    // preparation: the page summaries (for P = 1 the keys themselves)
    std::vector<double> Kd((size_t)(n * D + 1));
    load(K, f32, row0, n * D, Kd.data());
    std::vector<double> kmin, kmax;
    const double *lo = Kd.data(), *hi = Kd.data();
    if (P != 1) {
      kmin.resize((size_t)(NP * D + 1));
      kmax.resize((size_t)(NP * D + 1));
      orc_page_minmax(Kd.data(), D, n, P, kmin.data(), kmax.data());
      lo = kmin.data();
      hi = kmax.data();
    }
    std::vector<double> sk((size_t)G);
    if (sink)
      for (int g = 0; g < G; ++g) sk[g] = sink[h * G + g];
    std::vector<double> qd((size_t)G * D), U((size_t)(G * NP + 1)), score((size_t)NP + 1);
    std::vector<i64> forced((size_t)NP + 1), pages((size_t)std::max<i64>(k, NP) + 1);
    std::vector<i64> toks((size_t)(std::max<i64>(k, NP) * P + 1));
    std::vector<double> Kt, Vt;
    double* o = o_out + (i64)i * G * D;
    double* lse = lse_out + (i64)i * G;
    i64 np = 0;
    double t0 = now_s(), dt = 0.0;
    int rep = 0;
    do {
      load(q, f32, ((i64)b * Hq + (i64)h * G) * D, (i64)G * D, qd.data());
      orc_quest_bound(qd.data(), G, D, lo, hi, NP, U.data());
      orc_group_score(U.data(), G, NP, score.data());
      i64 nf = orc_forced_pages(n, P, n_sink_pages, n_local_tokens, forced.data());
      np = orc_select_topk(score.data(), NP, k, forced.data(), nf, pages.data());
      if (np < 0) {
        bad = 1;
        return;
      }
      i64 nt = orc_pages_to_tokens(pages.data(), np, n, P, toks.data());
      Kt.assign((size_t)(nt * D + 1), 0.0);
      Vt.assign((size_t)(nt * D + 1), 0.0);
      for (i64 j = 0; j < nt; ++j) {
        load(K, f32, row0 + toks[j] * D, D, Kt.data() + j * D);
        load(V, f32, row0 + toks[j] * D, D, Vt.data() + j * D);
      }
      orc_softmax_attention(qd.data(), G, D, Kt.data(), Vt.data(), nt, D, scale, sink ? sk.data() : nullptr,
                            o, lse);
      ++rep;
      const double esz = f32 ? 4.0 : 2.0;
      bytes[i] += (double)NP * (P == 1 ? 1 : 2) * D * esz + (double)nt * 2 * D * esz;
      dt = now_s() - t0;
    } while (dt < min_busy);
    busy[i] = dt;
    reps[i] = rep;
    for (i64 j = 0; j < k; ++j) pages_out[(i64)i * k + j] = j < np ? (int32_t)pages[j] : -1;
  });
  double sb = 0.0, sy = 0.0, sr = 0.0;
  for (int i = 0; i < nrows; ++i) {
    sb += busy[i];
    sy += bytes[i];
    sr += reps[i];
  }
  stats_out[0] = sb;
  stats_out[1] = sy;
  stats_out[2] = sr;
  return bad ? -1 : 0;
}

// The top-delta decode step on a bf16 workload (f32 = 0), row by row: for every listed
// row, decode its keys and build the thumbnails of its complete blocks (and,
// when refined != 0, their residuals; untimed preparation: thumbnails are
// built when a block completes), then repeat until min_busy seconds have
// passed the timed select + attend: the pseudo-max from the exact keys of
// the first and newest block, the margin of every other complete block from
// its thumbnail, the keep rule, and attention over the kept blocks (exact
// keys, or refined keys for complete blocks when refined != 0).
//   count_out [nrows], blocks_out [nrows, Cap / block] ascending, o_out and
//   lse_out as in orc_quest_step_bf16; stats_out likewise (bytes: packed
//   codes + bf16 scales of the scanned blocks + the bf16 keys of the first
//   and newest block + the kept tokens' keys (or codes, residuals and
//   scales) and values).
int orc_delta_step(const void* q, const void* K, const void* V, int f32, const int32_t* ctx_len,
                        int B, int Hq, int Hkv, int D, i64 Cap, int block, double delta, double scale,
                        const float* sink, int refined, const int32_t* rows, int nrows, int nthreads,
                        double min_busy, int32_t* count_out, int32_t* blocks_out, double* o_out,
                        double* lse_out, double* stats_out) {
  (void)B;
  const int G = Hq / Hkv;
  const i64 maxblk = Cap / block;
  std::vector<double> busy((size_t)nrows, 0.0), bytes((size_t)nrows, 0.0), reps((size_t)nrows, 0.0);
  parallel_rows(nrows, nthreads, [&](int i) {
    const int r = rows[i], b = r / Hkv, h = r % Hkv;
    const i64 n = ctx_len[b], nfull = n / block;
    const i64 row0 = (i64)r * Cap * D;  // the row's first key element
    std::vector<double> Kd((size_t)(n * D + 1));
    load(K, f32, row0, n * D, Kd.data());
    std::vector<uint8_t> codes((size_t)(nfull * block * D + 1));
    std::vector<double> scales((size_t)(nfull * D + 1));
    std::vector<int8_t> res((size_t)(nfull * block * D + 1));
    if (refined)
      orc_residuals_row(Kd.data(), D, n, block, codes.data(), scales.data(), res.data());
    else
      orc_thumbnails_row(Kd.data(), D, n, block, codes.data(), scales.data());
    std::vector<double> sk((size_t)G);
    if (sink)
      for (int g = 0; g < G; ++g) sk[g] = sink[h * G + g];
    std::vector<double> qd((size_t)G * D), mt((size_t)G), kref((size_t)block * D);
    std::vector<i64> sel((size_t)maxblk + 2), toks;
    std::vector<double> Kt, Vt;
    double* o = o_out + (i64)i * G * D;
    double* lse = lse_out + (i64)i * G;
    i64 ns = 0;
    double t0 = now_s(), dt = 0.0;
    int rep = 0;
    do {
      load(q, f32, ((i64)b * Hq + (i64)h * G) * D, (i64)G * D, qd.data());
      // the pseudo-max over the exact keys of the forced blocks (eq. 3)
      i64 fb[2];
      i64 nb = orc_delta_forced_blocks(n, block, fb);
      i64 nft = 0;
      for (int g = 0; g < G; ++g) mt[g] = kNegInf;
      for (i64 x = 0; x < nb; ++x)
        for (i64 t = fb[x] * block; t < std::min((fb[x] + 1) * block, n); ++t) {
          for (int g = 0; g < G; ++g)
            mt[g] = std::max(mt[g], scale * dot(qd.data() + (i64)g * D, Kd.data() + t * D, D));
          ++nft;
        }
      // the keep rule over every other complete block (eqs. 1-2)
      ns = 0;
      for (i64 x = 0; x < nb; ++x) sel[ns++] = fb[x];
      i64 scanned = 0;
      for (i64 j = 0; j < nfull; ++j) {
        if (j == fb[0] || (nb > 1 && j == fb[1])) continue;
        ++scanned;
        double mg = block_margin(qd.data(), G, D, codes.data() + j * block * D, scales.data() + j * D, block,
                                 scale, mt.data());
        if (mg >= -delta) sel[ns++] = j;
      }
      std::sort(sel.begin(), sel.begin() + ns);
      // attention over the kept blocks
      toks.assign((size_t)(ns * block + 1), 0);
      i64 nt = orc_pages_to_tokens(sel.data(), ns, n, block, toks.data());
      Kt.assign((size_t)(nt * D + 1), 0.0);
      Vt.assign((size_t)(nt * D + 1), 0.0);
      i64 cached = -1, ref_tok = 0, ref_blk = 0;
      for (i64 x = 0; x < nt; ++x) {
        i64 t = toks[x], j = t / block;
        if (refined && j < nfull) {
          if (cached != j) {
            orc_refined_keys(codes.data() + j * block * D, scales.data() + j * D, res.data() + j * block * D,
                             block, D, 1, kref.data());
            cached = j;
            ++ref_blk;
          }
          for (int c = 0; c < D; ++c) Kt[x * D + c] = kref[(t - j * block) * D + c];
          ++ref_tok;
        } else {
          load(K, f32, row0 + t * D, D, Kt.data() + x * D);
        }
        load(V, f32, row0 + t * D, D, Vt.data() + x * D);
      }
      orc_softmax_attention(qd.data(), G, D, Kt.data(), Vt.data(), nt, D, scale, sink ? sk.data() : nullptr,
                            o, lse);
      ++rep;
      double scan = (double)scanned * ((double)block * D / 4 + (double)D * 2) + (double)nft * D * 2;
      double kv = (double)(nt - ref_tok) * 2 * D * 2 + (double)ref_tok * ((double)D / 4 + D + D * 2) +
                  (double)ref_blk * D * 2;
      bytes[i] += scan + kv;
      dt = now_s() - t0;
    } while (dt < min_busy);
    busy[i] = dt;
    reps[i] = rep;
    count_out[i] = (int32_t)ns;
    for (i64 j = 0; j < maxblk; ++j) blocks_out[(i64)i * maxblk + j] = j < ns ? (int32_t)sel[j] : -1;
  });
  double sb = 0.0, sy = 0.0, sr = 0.0;
  for (int i = 0; i < nrows; ++i) {
    sb += busy[i];
    sy += bytes[i];
    sr += reps[i];
  }
  stats_out[0] = sb;
  stats_out[1] = sy;
  stats_out[2] = sr;
  return 0;
}

}  // extern "C"
