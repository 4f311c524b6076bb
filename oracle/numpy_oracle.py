"""Second fp64 CPU oracle for sparse decode attention, in numpy.

The primary oracle is the plain C++ one (sls_oracle.cpp, bound by
sls_oracle.py).  This numpy implementation was written independently of it
from the same pages; tests/test_oracle_cross.py checks that the two agree on
random inputs, function by function, and the mutation check plants mistakes
in both.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports, links or calls this
module; only the test suite, the smoke check and the benchmark's CPU-baseline
leg do.  It shares no code with the CUDA path: it decodes bf16 itself, builds
its own page summaries and thumbnails from the keys, and indexes the cache
layout itself.  Everything is computed in float64 from the exact values of
the bf16/fp32 inputs.

Sources (web pages; cited by title and section):

* [haystack]  "Don't read the haystack" (hareesh.pages.dev), Part one
  (two-stage flash-decoding) and Part two (per-page min/max bound, top-k,
  sink page and local pages).
* [ffd]       "Faster Than Flash: Exploiting Attention Sparsity for Efficient
  Long-Context Decoding" (picx.dev summary), Methodology 1 (2-bit mid-rise
  thumbnails and 8-bit residuals), 2 (top-delta, eqs. 1-3) and 3 (eq. 4:
  scaling and the refined final scores).
* [undivided] "Attention: Undivided & Uncompressed" (clintsebastian.com),
  Notation (S = QK^T / sqrt(d)) and Traffic (online softmax, delayed division).
* [tsd]       "Training-free sparse attention for long-context LLM decode"
  (joeddav/triton-sparse-decode), section 1 (sink as a virtual key, V=0).
* [mlxcel]    "perf(core): fused sparse-attention decode via page
  indirection" (lablup/mlxcel #1005), "The reduction" (contiguous cache as a
  page_size=1 pool) and "Corrected premise 1" (one page list per KV head).

Readings where the pages are silent are listed in the functions that take
them.  Parity status: every function here is pinned by tests under
``tests/test_oracle_*.py`` (brute force, closed forms, invariants, hand-worked
fixtures); none is "parity unpinned".
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np

NEG_INF = -math.inf


# ----------------------------------------------------------------------------
# input decoding
# ----------------------------------------------------------------------------

def to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of an fp32 array or of bf16 bit patterns (uint16)."""
    if dtype == "bf16":
        bits = np.asarray(x, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    return np.asarray(x, dtype=np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# attention: the plain definitions
# ----------------------------------------------------------------------------

def softmax_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float,
                      sink: Optional[np.ndarray] = None):
    """Exact softmax attention of G query rows over T keys.

    [undivided] Notation: scores S = q K^T * scale (scale = 1/sqrt(d)), P is
    the row softmax of S, O = P V.  [tsd] section 1: a learned per-head sink is
    a scalar logit that joins only the softmax denominator, i.e. a virtual key
    whose value is zero.  Reading: the sink is a raw logit (not multiplied by
    ``scale``).

    q [G, D], K [T, D], V [T, D] float64; sink [G] or None.
    Returns (o [G, D], lse [G]).  With T = 0 the output is 0 and the lse is
    the sink (or -inf without one).
    """
    q = np.asarray(q, np.float64)
    G = q.shape[0]
    D = V.shape[1] if V.ndim == 2 else q.shape[1]
    T = K.shape[0]
    x = scale * (q @ K.T) if T else np.zeros((G, 0))
    m = x.max(axis=1) if T else np.full(G, NEG_INF)
    if sink is not None:
        m = np.maximum(m, np.asarray(sink, np.float64))
    o = np.zeros((G, D))
    lse = np.full(G, NEG_INF)
    for g in range(G):
        if m[g] == NEG_INF:
            continue
        w = np.exp(x[g] - m[g])
        z = w.sum()
        if sink is not None:
            z += math.exp(float(sink[g]) - m[g])
        if T:
            o[g] = (w @ V) / z
        lse[g] = m[g] + math.log(z)
    return o, lse


def split_partials(q, K, V, scale, bounds):
    """Stage one of two-stage flash-decoding ([haystack] Part one): for each
    slice [a, b) of the keys, the slice max m, the normaliser l = sum
    exp(x - m) and the unnormalised accumulator acc = sum exp(x - m) v.
    Empty slices give m = -inf, l = 0, acc = 0."""
    G, D = q.shape[0], V.shape[1]
    out = []
    for a, b in bounds:
        if b <= a:
            out.append((np.full(G, NEG_INF), np.zeros(G), np.zeros((G, D))))
            continue
        x = scale * (q @ K[a:b].T)
        m = x.max(axis=1)
        w = np.exp(x - m[:, None])
        out.append((m, w.sum(axis=1), w @ V[a:b]))
    return out


def combine_partials(parts, sink=None):
    """Stage two ([haystack] Part one; [undivided] Traffic): rescale every
    partial by exp(m_s - M) with M the overall max (including the sink), sum,
    and divide once at the end.  The sink joins the denominator only, once.
    Returns (o [G, D], lse [G])."""
    G, D = parts[0][2].shape
    M = np.full(G, NEG_INF)
    for m, _, _ in parts:
        M = np.maximum(M, m)
    if sink is not None:
        M = np.maximum(M, np.asarray(sink, np.float64))
    o = np.zeros((G, D))
    lse = np.full(G, NEG_INF)
    for g in range(G):
        if M[g] == NEG_INF:
            continue
        L, acc = 0.0, np.zeros(D)
        for m, l, a in parts:
            if m[g] == NEG_INF:
                continue
            f = math.exp(m[g] - M[g])
            L += l[g] * f
            acc += a[g] * f
        if sink is not None:
            L += math.exp(float(sink[g]) - M[g])
        o[g] = acc / L
        lse[g] = M[g] + math.log(L)
    return o, lse


# ----------------------------------------------------------------------------
# Quest page selection
# ----------------------------------------------------------------------------

def num_pages(n: int, page_size: int) -> int:
    return -(-int(n) // int(page_size))


def page_minmax(K: np.ndarray, n: int, page_size: int):
    """Per-page, per-channel min and max of the keys of one (b, kv head) row
    ([haystack] Part two: "the elementwise min and max of its keys").  Only
    positions < n count, so a partial last page summarises its valid tokens.
    K [Cap, D] float64.  Returns (kmin, kmax), each [NP, D]."""
    NP = num_pages(n, page_size)
    D = K.shape[1]
    kmin = np.empty((NP, D))
    kmax = np.empty((NP, D))
    for p in range(NP):
        blk = K[p * page_size:min((p + 1) * page_size, n)]
        kmin[p] = blk.min(axis=0)
        kmax[p] = blk.max(axis=0)
    return kmin, kmax


def quest_bound(q: np.ndarray, kmin: np.ndarray, kmax: np.ndarray, chunk: int = 4096):
    """Upper bound of every page's attention score for every query head
    ([haystack] Part two): U[g, p] = sum_c max(q[g,c] * kmin[p,c],
    q[g,c] * kmax[p,c]).  Unscaled (ranking is invariant to the positive
    softmax scale).  q [G, D]; kmin, kmax [NP, D].  Returns U [G, NP]."""
    G = q.shape[0]
    NP = kmin.shape[0]
    U = np.empty((G, NP))
    for a in range(0, NP, chunk):
        lo = q[:, None, :] * kmin[None, a:a + chunk, :]
        hi = q[:, None, :] * kmax[None, a:a + chunk, :]
        U[:, a:a + chunk] = np.maximum(lo, hi).sum(axis=2)
    return U


def group_score(U: np.ndarray) -> np.ndarray:
    """One page list per (batch, KV head), shared by the query heads of the
    group ([mlxcel] "Corrected premise 1": a request shares one page list
    across the query heads under its KV head).  Reading: the group's score of
    a page is the max over its heads, which keeps the bound admissible for
    every head."""
    return U.max(axis=0)


def forced_pages(n: int, page_size: int, n_sink_pages: int, n_local_tokens: int) -> np.ndarray:
    """Pages kept regardless of score ([haystack] Part two: "plus the
    attention-sink page and the last few local pages"): the first
    ``n_sink_pages`` pages and every page holding one of the last
    ``n_local_tokens`` positions.  Sorted ascending."""
    NP = num_pages(n, page_size)
    f = set(range(min(n_sink_pages, NP)))
    if n_local_tokens > 0 and n > 0:
        first = max(n - n_local_tokens, 0) // page_size
        f.update(range(first, NP))
    return np.array(sorted(f), dtype=np.int64)


def select_topk(score: np.ndarray, k: int, forced: np.ndarray) -> np.ndarray:
    """Top-k selection with forced pages ([haystack] Part two: rank pages by
    the bound, keep the top k plus the forced pages).

    Readings: the budget k counts the forced pages (the page list has a fixed
    cardinality of min(k, NP)); among equal scores the lower page index wins;
    the result is sorted ascending.  score [NP].  Returns page indices."""
    NP = score.shape[0]
    if NP <= k:
        return np.arange(NP, dtype=np.int64)
    forced = np.asarray(forced, dtype=np.int64)
    if forced.size > k:
        raise ValueError("budget smaller than the forced pages")
    cand = np.setdiff1d(np.arange(NP), forced)
    kk = k - forced.size
    order = np.lexsort((cand, -score[cand]))   # by score desc, then index asc
    chosen = cand[order[:kk]]
    return np.sort(np.concatenate([forced, chosen]))


def kth_score(score: np.ndarray, k: int, forced: np.ndarray) -> float:
    """Score of the last candidate admitted by ``select_topk`` (the k-th
    ranked non-forced page), used to recognise boundary ties."""
    NP = score.shape[0]
    if NP <= k:
        return NEG_INF
    cand = np.setdiff1d(np.arange(NP), np.asarray(forced, dtype=np.int64))
    kk = k - len(forced)
    if kk <= 0:
        return math.inf
    order = np.lexsort((cand, -score[cand]))
    return float(score[cand[order[kk - 1]]])


def pages_to_tokens(pages: np.ndarray, n: int, page_size: int) -> np.ndarray:
    """Token positions of the given pages, restricted to positions < n
    ([mlxcel] "The reduction": a token is reached as page * page_size + i)."""
    toks = [np.arange(p * page_size, min((p + 1) * page_size, n)) for p in pages if p >= 0]
    return np.concatenate(toks) if toks else np.zeros(0, dtype=np.int64)


def quest_select_row(q, K, n, page_size, k, n_sink_pages, n_local_tokens):
    """Selection of one row: page summaries -> bound -> group max -> top-k.
    q [G, D], K [Cap, D] float64.  Returns (pages, group_score, kth)."""
    if page_size == 1:
        # A one-token page has kmin = kmax = k_t; the bound is then the exact
        # score q . k_t.
        kmin = kmax = K[:n]
    else:
        kmin, kmax = page_minmax(K, n, page_size)
    s = group_score(quest_bound(q, kmin, kmax))
    f = forced_pages(n, page_size, n_sink_pages, n_local_tokens)
    return select_topk(s, k, f), s, kth_score(s, k, f)


# ----------------------------------------------------------------------------
# FFD thumbnails and top-delta
# ----------------------------------------------------------------------------

def thumb_quantize(Kb: np.ndarray):
    """2-bit symmetric zero-free (mid-rise) thumbnail of one block of keys
    ([ffd] Methodology 1).  s[c] = max_t |k[t,c]|; levels -0.75s, -0.25s,
    +0.25s, +0.75s with decision thresholds -s/2, 0, +s/2.

    Readings: a value on a threshold takes the upper level (k = 0 maps to
    +0.25s, k = s/2 to +0.75s; an all-zero channel, s = 0, takes code 3,
    whose level is 0); codes 0..3 name the levels in increasing order.  Kb [T, D] float64.  Returns (codes [T, D] uint8, s [D])."""
    s = np.abs(Kb).max(axis=0)
    h = s / 2.0
    codes = np.where(Kb >= h, 3, np.where(Kb >= 0, 2, np.where(Kb >= -h, 1, 0)))
    return codes.astype(np.uint8), s


def thumb_dequant(codes: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Level value of each code: (code - 1.5) * s / 2."""
    return (codes.astype(np.float64) - 1.5) * (s / 2.0)


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """Storage format of the thumbnails: four 2-bit codes per byte, channel c
    in bits 2*(c % 4) of byte c // 4.  codes [T, D] -> [T, D/4] uint8."""
    T, D = codes.shape
    c = codes.reshape(T, D // 4, 4).astype(np.uint32)
    b = c[:, :, 0] | (c[:, :, 1] << 2) | (c[:, :, 2] << 4) | (c[:, :, 3] << 6)
    return b.astype(np.uint8)


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    T, W = packed.shape
    p = packed.astype(np.uint32)
    out = np.stack([(p >> (2 * j)) & 3 for j in range(4)], axis=2)
    return out.reshape(T, W * 4).astype(np.uint8)


def thumbnails_row(K: np.ndarray, n: int, block: int):
    """Thumbnails of every complete block of one row (positions < n).
    Returns (codes [nfull*block, D] uint8 unpacked, scales [nfull, D])."""
    nfull = n // block
    D = K.shape[1]
    codes = np.zeros((nfull * block, D), dtype=np.uint8)
    scales = np.zeros((nfull, D))
    for j in range(nfull):
        c, s = thumb_quantize(K[j * block:(j + 1) * block])
        codes[j * block:(j + 1) * block] = c
        scales[j] = s
    return codes, scales


def delta_forced_blocks(n: int, block: int) -> np.ndarray:
    """Blocks always kept by top-delta: block 0 (the sink tokens, S_global)
    and the block of the newest position (S_local, possibly partial).

    Reading: [ffd] eq. 3 names S_global and S_local without sizes; here they
    are the first and the last block."""
    if n <= 0:
        return np.zeros(0, dtype=np.int64)
    last = (n - 1) // block
    return np.array(sorted({0, last}), dtype=np.int64)


def pseudo_max(q: np.ndarray, K: np.ndarray, n: int, block: int, scale: float) -> np.ndarray:
    """[ffd] eq. 3: m~ = max of the exact scores s = scale * q . k over the
    sink and local tokens (blocks returned by ``delta_forced_blocks``).
    q [G, D], K [Cap, D].  Returns m~ [G]."""
    toks = pages_to_tokens(delta_forced_blocks(n, block), n, block)
    return (scale * (q @ K[toks].T)).max(axis=1)


def delta_block_margin(q, K, n, block, scale):
    """For every complete, non-forced block b of the row: the block margin
    max_g max_{t in b} (s~[g,t] - m~[g]) where s~ = scale * q . k^ uses the
    2-bit thumbnail k^ ([ffd] Methodology 2, eq. 1 with the pseudo-max of
    eq. 3 in place of m; eq. 4 fixes the 1/sqrt(d) scaling).

    Readings: a block's score is the max over its tokens; a GQA group keeps
    the union over its heads (max over g).  Returns (blocks, margin)."""
    nfull = n // block
    forced = set(delta_forced_blocks(n, block).tolist())
    mt = pseudo_max(q, K, n, block, scale)
    blocks, margins = [], []
    for j in range(nfull):
        if j in forced:
            continue
        c, s = thumb_quantize(K[j * block:(j + 1) * block])
        st = scale * (q @ thumb_dequant(c, s).T)      # [G, block]
        blocks.append(j)
        margins.append(float((st - mt[:, None]).max()))
    return np.array(blocks, dtype=np.int64), np.array(margins)


def delta_select_row(q, K, n, block, delta, scale):
    """Top-delta selection of one row ([ffd] eqs. 1-3): keep a complete block
    when its margin is >= -delta; the forced blocks are always kept.
    Returns (sorted kept blocks, (scanned blocks, margins))."""
    blocks, margins = delta_block_margin(q, K, n, block, scale)
    kept = blocks[margins >= -delta]
    sel = np.union1d(delta_forced_blocks(n, block), kept)
    return sel.astype(np.int64), (blocks, margins)


# ----------------------------------------------------------------------------
# FFD 8-bit residuals and the refined scores (eq. 4)
# ----------------------------------------------------------------------------

RES_DENOM = 508.0  # 4 * 127: residual codes -127..127 span the +-s/4 quantisation error


def residual_quantize(Kb: np.ndarray, codes: np.ndarray, s: np.ndarray) -> np.ndarray:
    """8-bit residual of one complete block ([ffd] Methodology 1: the key is
    split into the 2-bit thumbnail k_quant and an 8-bit residual k_res that
    recovers the precision the thumbnail drops).

    Readings (the page gives no encoding): the residual e = k - k^ of a
    mid-rise 2-bit code lies in [-s/4, s/4] (levels s/2 apart, thresholds
    half-way), so it is stored on the thumbnail's own block/channel scale s
    as r = the integer nearest to e * 508 / s (ties to even), in
    [-127, 127], and the refined key is k~ = k^ + r * s / 508; s = 0 (an
    all-zero channel) gives 0.  For bf16 keys and scales the float64
    quotient decides the nearest integer exactly (the exact quotient is
    either a half-integer, computed exactly, or far from one relative to
    float64 rounding).

    Kb [T, D] float64 (exact bf16 values); codes [T, D]; s [D].
    Returns r [T, D] int8."""
    Kb = np.asarray(Kb, np.float64)
    s = np.broadcast_to(np.asarray(s, np.float64), Kb.shape)
    e = Kb - thumb_dequant(codes, s)
    safe = np.where(s > 0, s, 1.0)
    x = np.where(s > 0, e * RES_DENOM / safe, 0.0)
    return np.clip(np.rint(x), -127, 127).astype(np.int8)


def refined_keys(codes: np.ndarray, s: np.ndarray, r: np.ndarray) -> np.ndarray:
    """The key the refinement scores with: k~ = k^ + r * s / 508, so that
    q . k~ = q . k_quant + q . k_res ([ffd] eq. 4 numerator).  float64."""
    return thumb_dequant(codes, s) + np.asarray(r, np.float64) * (np.asarray(s, np.float64) / RES_DENOM)


def residuals_row(K: np.ndarray, n: int, block: int):
    """Codes, scales and residuals of every complete block of one row
    (positions < n).  Returns (codes [nfull*block, D], scales [nfull, D],
    res [nfull*block, D] int8)."""
    codes, scales = thumbnails_row(K, n, block)
    res = np.zeros(codes.shape, dtype=np.int8)
    for j in range(n // block):
        rows = slice(j * block, (j + 1) * block)
        res[rows] = residual_quantize(K[rows], codes[rows], scales[j])
    return codes, scales, res


def refined_attention_row(q, K, V, blocks, n, block, scale, sink=None):
    """Attention over the selected blocks with the refined final scores of
    [ffd] Methodology 3 step 3, eq. 4: s = (q . k_quant + q . k_res) / sqrt(d)
    for the tokens of complete blocks.

    Reading: the newest block is partial and has no thumbnail yet, so its
    tokens are scored with the exact key; values are exact.
    q [G, D]; K, V [>= n, D] float64; blocks: the row's block list."""
    codes, scales, res = residuals_row(K, n, block)
    Kt = np.array(K[:n], dtype=np.float64, copy=True)
    nfull = n // block
    if nfull:
        Kt[:nfull * block] = refined_keys(codes, np.repeat(scales, block, axis=0), res)
    toks = pages_to_tokens(np.asarray(blocks), n, block)
    return softmax_attention(q, Kt[toks], V[toks], scale, sink)


# ----------------------------------------------------------------------------
# selection quality
# ----------------------------------------------------------------------------

def attention_mass_recall(q: np.ndarray, K: np.ndarray, pages, n: int, page_size: int,
                          scale: float) -> np.ndarray:
    """Share of each query head's full-context softmax mass that falls on the
    tokens of the selected pages ([haystack] Part three, "attention mass
    captured": how much of the true attention mass the selected pages hold).

    q [G, D]; K [>= n, D] float64; pages: the row's page list (-1 entries and
    positions >= n ignored).  recall_g = sum_{t in sel} exp(x_gt - M_g) /
    sum_{t < n} exp(x_gt - M_g) with x = scale * q.k and M the row max.
    Reading: the sink (a virtual key) is not a token and takes no part; an
    empty context misses nothing, so its recall is 1.
    Returns [G].
    """
    q = np.asarray(q, np.float64)
    G = q.shape[0]
    if n == 0:
        return np.ones(G)
    x = scale * (q @ K[:n].T)
    m = x.max(axis=1, keepdims=True)
    w = np.exp(x - m)
    toks = pages_to_tokens(np.asarray(pages), n, page_size)
    return w[:, toks].sum(axis=1) / w.sum(axis=1)


# ----------------------------------------------------------------------------
# one decode step of one row
# ----------------------------------------------------------------------------

def sparse_attention_row(q, K, V, pages, n, page_size, scale, sink=None):
    """Attention restricted to the tokens of the selected pages
    ([haystack] Part two: the sparse twin walks the selected indices)."""
    toks = pages_to_tokens(np.asarray(pages), n, page_size)
    return softmax_attention(q, K[toks], V[toks], scale, sink)
