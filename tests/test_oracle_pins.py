"""Pins of the fp64 oracle against things other than itself: hand-worked
fixtures (tests/golden), brute force on tiny inputs, closed forms and
invariants the pages state.  CPU only."""
import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import sls_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def rnd(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


# ----------------------------------------------------------------- attention

def brute_attention(q, K, V, scale, sink=None):
    """Explicit per-element loops with the math module (no numpy reductions)."""
    G, D = len(q), len(V[0]) if len(V) else len(q[0])
    out, lses = [], []
    for g in range(G):
        xs = [scale * sum(q[g][c] * K[t][c] for c in range(len(q[g]))) for t in range(len(K))]
        terms = list(xs) + ([float(sink[g])] if sink is not None else [])
        if not terms:
            out.append([0.0] * D)
            lses.append(-math.inf)
            continue
        m = max(terms)
        ws = [math.exp(x - m) for x in xs]
        z = sum(ws) + (math.exp(float(sink[g]) - m) if sink is not None else 0.0)
        out.append([sum(ws[t] * V[t][c] for t in range(len(K))) / z for c in range(D)])
        lses.append(m + math.log(z))
    return np.array(out), np.array(lses)


@pytest.mark.parametrize("T,with_sink", [(1, False), (5, False), (13, True), (40, True)])
def test_softmax_attention_brute_force(T, with_sink):
    G, D = 3, 6
    q, K, V = rnd(1, G, D) * 2, rnd(2, T, D), rnd(3, T, D)
    sink = rnd(4, G) if with_sink else None
    o, lse = O.softmax_attention(q, K, V, 1 / math.sqrt(D), sink)
    ob, lb = brute_attention(q.tolist(), K.tolist(), V.tolist(), 1 / math.sqrt(D), sink)
    np.testing.assert_allclose(o, ob, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lb, rtol=1e-12, atol=1e-13)


def test_attention_golden():
    d = golden("attention_sink_example.json")
    q, K, V = (np.array(d[k]) for k in ("q", "K", "V"))
    o, lse = O.softmax_attention(q, K, V, d["scale"])
    np.testing.assert_allclose(o, d["o_nosink"], atol=1e-14)
    np.testing.assert_allclose(lse, d["lse_nosink"], atol=1e-14)
    o, lse = O.softmax_attention(q, K, V, d["scale"], np.array(d["sink"]))
    np.testing.assert_allclose(o, d["o_sink"], atol=1e-14)
    np.testing.assert_allclose(lse, d["lse_sink"], atol=1e-14)


@pytest.mark.parametrize("splits", [1, 2, 3, 7])
@pytest.mark.parametrize("with_sink", [False, True])
def test_split_combine_equals_dense(splits, with_sink):
    G, D, T = 4, 8, 50
    q, K, V = rnd(5, G, D) * 3, rnd(6, T, D), rnd(7, T, D)
    sink = rnd(8, G) * 3 if with_sink else None
    cuts = np.linspace(0, T, splits + 1).astype(int)
    bounds = list(zip(cuts[:-1], cuts[1:])) + [(T, T)]   # plus one empty split
    parts = O.split_partials(q, K, V, 0.3, bounds)
    o, lse = O.combine_partials(parts, sink)
    od, ld = O.softmax_attention(q, K, V, 0.3, sink)
    np.testing.assert_allclose(o, od, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, ld, rtol=1e-12, atol=1e-13)


def test_sink_identity():
    """o_sink = o * Z / (Z + e^(sigma - M)) and lse_sink = logaddexp(lse, sigma)."""
    G, D, T = 5, 16, 33
    q, K, V = rnd(9, G, D) * 2, rnd(10, T, D), rnd(11, T, D)
    sigma = rnd(12, G) * 4
    scale = 1 / math.sqrt(D)
    o, lse = O.softmax_attention(q, K, V, scale)
    os_, ls_ = O.softmax_attention(q, K, V, scale, sigma)
    x = scale * q @ K.T
    M = x.max(axis=1)
    Z = np.exp(x - M[:, None]).sum(axis=1)
    np.testing.assert_allclose(os_, o * (Z / (Z + np.exp(sigma - M)))[:, None], rtol=1e-12)
    np.testing.assert_allclose(ls_, np.logaddexp(lse, sigma), rtol=1e-12)
    o2, _ = O.softmax_attention(q, K, V, scale, np.full(G, -1e300))
    np.testing.assert_allclose(o2, o, rtol=1e-15)


def test_empty_attention():
    q = rnd(13, 2, 4)
    o, lse = O.softmax_attention(q, np.zeros((0, 4)), np.zeros((0, 4)), 0.5)
    assert np.all(o == 0) and np.all(lse == -math.inf)
    o, lse = O.softmax_attention(q, np.zeros((0, 4)), np.zeros((0, 4)), 0.5, np.array([0.3, -1.0]))
    assert np.all(o == 0)
    np.testing.assert_allclose(lse, [0.3, -1.0])


# ---------------------------------------------------------------------- quest

def test_quest_golden():
    d = golden("quest_bound_example.json")
    q, K = np.array(d["q"]), np.array(d["K"])
    kmin, kmax = O.page_minmax(K, len(K), d["page_size"])
    np.testing.assert_array_equal(kmin, d["kmin"])
    np.testing.assert_array_equal(kmax, d["kmax"])
    U = O.quest_bound(q, kmin, kmax)
    np.testing.assert_array_equal(U, d["U"])
    sel = O.select_topk(O.group_score(U), 1, np.zeros(0, np.int64))
    assert sel.tolist() == d["top1"]


def test_page_minmax_brute_force():
    K = rnd(14, 53, 3)
    for n, P in [(53, 16), (50, 16), (1, 16), (17, 16), (16, 16), (53, 1), (40, 64)]:
        kmin, kmax = O.page_minmax(K, n, P)
        assert kmin.shape[0] == -(-n // P)
        for p in range(kmin.shape[0]):
            for c in range(3):
                vals = [K[t, c] for t in range(p * P, min(p * P + P, n))]
                assert kmin[p, c] == min(vals) and kmax[p, c] == max(vals)


@pytest.mark.parametrize("P", [1, 4, 16])
def test_quest_bound_admissible_and_identity(P):
    G, D, n = 6, 32, 203
    q, K = rnd(15, G, D) * 2, rnd(16, 256, D)
    kmin, kmax = O.page_minmax(K, n, P)
    U = O.quest_bound(q, kmin, kmax)
    true = np.array([[(q[g] @ K[p * P:min(p * P + P, n)].T).max() for p in range(kmin.shape[0])]
                     for g in range(G)])
    assert np.all(U >= true - 1e-12)
    if P == 1:
        np.testing.assert_allclose(U, true, rtol=1e-12, atol=1e-12)
    # max(q.kmin, q.kmax) = q.mid + |q|.half, summed over channels
    mid, half = (kmin + kmax) / 2, (kmax - kmin) / 2
    np.testing.assert_allclose(U, q @ mid.T + np.abs(q) @ half.T, rtol=1e-12, atol=1e-12)
    # the group score is admissible for every head of the group
    s = O.group_score(U)
    assert np.all(s[None, :] >= true - 1e-12)


def brute_topk(score, k, forced):
    """The unique subset S (|S| = min(k, NP), forced pages inside) such that
    every chosen free page beats every unchosen one by (score desc, index asc)."""
    NP = len(score)
    if NP <= k:
        return list(range(NP))
    free = [p for p in range(NP) if p not in set(forced)]
    found = []
    for comb in itertools.combinations(free, k - len(forced)):
        ok = all(score[i] > score[j] or (score[i] == score[j] and i < j)
                 for i in comb for j in free if j not in comb)
        if ok:
            found.append(sorted(list(forced) + list(comb)))
    assert len(found) == 1
    return found[0]


@pytest.mark.parametrize("seed", range(8))
def test_topk_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    NP = int(rng.integers(3, 11))
    score = rng.integers(-3, 4, NP).astype(float)   # many ties
    forced = sorted(rng.choice(NP, size=int(rng.integers(0, 3)), replace=False).tolist())
    k = int(rng.integers(len(forced) + 1, NP + 2))
    got = O.select_topk(score, k, np.array(forced, dtype=np.int64)).tolist()
    assert got == brute_topk(score.tolist(), k, forced)


def test_topk_ties_at_the_budget_boundary():
    """Ties that straddle the budget: among equal scores the lower page index
    is admitted.  A hand-worked case, then tie-heavy random rows (scores in
    {0, 1}, budgets below the page count) against the brute force."""
    assert O.select_topk(np.array([1.0, 2.0, 2.0, 2.0, 0.0]), 2, np.zeros(0, np.int64)).tolist() == [1, 2]
    assert O.select_topk(np.array([5.0, 1.0, 1.0, 1.0]), 3, np.array([0])).tolist() == [0, 1, 2]
    for seed in range(40):
        rng = np.random.default_rng(200 + seed)
        NP = int(rng.integers(6, 12))
        score = rng.integers(0, 2, NP).astype(float)
        forced = sorted(rng.choice(NP, size=int(rng.integers(0, 3)), replace=False).tolist())
        k = int(rng.integers(len(forced) + 1, NP))
        got = O.select_topk(score, k, np.array(forced, dtype=np.int64)).tolist()
        assert got == brute_topk(score.tolist(), k, forced), (seed, score, k, forced)


def test_forced_pages():
    assert O.forced_pages(32768, 16, 1, 64).tolist() == [0, 2044, 2045, 2046, 2047]
    assert O.forced_pages(1000, 16, 1, 64).tolist() == [0, 58, 59, 60, 61, 62]
    assert O.forced_pages(131072, 1, 4, 0).tolist() == [0, 1, 2, 3]
    assert O.forced_pages(20, 16, 1, 64).tolist() == [0, 1]
    assert O.forced_pages(0, 16, 1, 64).tolist() == []
    assert O.forced_pages(1024, 16, 0, 0).tolist() == []


def test_sparse_equals_dense_when_budget_covers_all():
    G, D, n, P = 4, 16, 300, 16
    q, K, V = rnd(17, G, D) * 2, rnd(18, 320, D), rnd(19, 320, D)
    sink = rnd(20, G)
    pages, _, _ = O.quest_select_row(q, K, n, P, k=100, n_sink_pages=1, n_local_tokens=64)
    assert pages.tolist() == list(range(19))
    o, lse = O.sparse_attention_row(q, K, V, pages, n, P, 0.25, sink)
    od, ld = O.softmax_attention(q, K[:n], V[:n], 0.25, sink)
    np.testing.assert_allclose(o, od, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, ld, rtol=1e-12)


@pytest.mark.parametrize("n", [1, 15, 17, 1000, 1023])
def test_partial_pages_equal_minus_inf_padding(n):
    """A partial last page behaves as if the missing positions scored -inf:
    the page summaries ignore them and attention over the selected pages
    equals attention over the valid tokens only."""
    G, D, P = 2, 8, 16
    K, V = rnd(21, 1024, D), rnd(22, 1024, D)
    K[n:] = 1e6          # garbage past the context must not leak in
    q = rnd(23, G, D)
    kmin, kmax = O.page_minmax(K, n, P)
    Kp = np.where(np.arange(1024)[:, None] < n, K, np.nan)
    for p in range(kmin.shape[0]):
        blk = Kp[p * P:(p + 1) * P]
        np.testing.assert_array_equal(kmin[p], np.nanmin(blk, axis=0))
        np.testing.assert_array_equal(kmax[p], np.nanmax(blk, axis=0))
    NP = -(-n // P)
    o, _ = O.sparse_attention_row(q, K, V, np.arange(NP), n, P, 0.3)
    x = 0.3 * q @ K[:NP * P].T
    x[:, n:] = -np.inf
    w = np.exp(x - x.max(axis=1, keepdims=True))
    ref = (w @ V[:NP * P]) / w.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-13)


def test_page_size_one_selection_is_exact_score_topk():
    G, D, n = 3, 8, 100
    q, K = rnd(24, G, D), rnd(25, 100, D)
    pages, s, _ = O.quest_select_row(q, K, n, 1, k=20, n_sink_pages=4, n_local_tokens=0)
    exact = (q @ K.T).max(axis=0)
    np.testing.assert_allclose(s, exact, rtol=1e-12)
    free = [t for t in range(n) if t >= 4]
    top = sorted(free, key=lambda t: (-exact[t], t))[:16]
    assert pages.tolist() == sorted([0, 1, 2, 3] + top)


# ------------------------------------------------------------------------ ffd

def test_thumbnail_golden():
    d = golden("ffd_thumbnail_example.json")
    k = np.array(d["k"])[:, None]
    codes, s = O.thumb_quantize(k)
    assert s.tolist() == [d["s"]]
    assert codes[:, 0].tolist() == d["codes"]
    np.testing.assert_array_equal(O.thumb_dequant(codes, s)[:, 0], d["dequant"])
    assert abs(math.exp(-d["delta"]) - d["peak_fraction_at_delta"]) < 1e-15


def test_thumbnail_error_bound_and_packing():
    """Mid-rise quantisation error is at most s/4 per element; the levels are
    exactly +-0.25s, +-0.75s; packing round-trips."""
    K = rnd(26, 64, 128) * np.exp(rnd(27, 1, 128))
    codes, s = O.thumb_quantize(K)
    kh = O.thumb_dequant(codes, s)
    assert np.all(np.abs(K - kh) <= s / 4 + 1e-15)
    lv = np.unique(np.round(kh / s, 12))
    assert set(lv.tolist()) <= {-0.75, -0.25, 0.25, 0.75}
    assert np.array_equal(O.unpack_codes(O.pack_codes(codes)), codes)
    zero = O.thumb_quantize(np.zeros((4, 8)))
    # s = 0: all three thresholds are 0, the value takes the upper level (code 3), whose value is 0
    assert np.all(zero[0] == 3) and np.all(O.thumb_dequant(*zero) == 0)


def test_pack_format_bits():
    codes = np.array([[1, 2, 3, 0, 3, 3, 3, 3]], dtype=np.uint8)
    assert O.pack_codes(codes).tolist() == [[0b00111001, 0xFF]]


def test_delta_golden():
    d = golden("delta_select_example.json")
    q, K = np.array(d["q"]), np.array(d["K"])
    mt = O.pseudo_max(q, K, d["n"], d["block"], d["scale"])
    np.testing.assert_allclose(mt, d["pseudo_max"])
    blocks, margins = O.delta_block_margin(q, K, d["n"], d["block"], d["scale"])
    assert blocks.tolist() == [1]
    np.testing.assert_allclose(margins, [d["margin_block1"]])
    assert O.delta_select_row(q, K, d["n"], d["block"], 5.0, d["scale"])[0].tolist() == d["kept_delta5"]
    assert O.delta_select_row(q, K, d["n"], d["block"], 2.0, d["scale"])[0].tolist() == d["kept_delta2"]


@pytest.mark.parametrize("n", [5, 64, 65, 640, 1000])
def test_pseudo_max_covers_sink_and_local_blocks(n):
    """FFD eq. 3: m~ is the max exact score over S_global (block 0) and
    S_local (the newest block, complete or partial), by explicit loops; a key
    planted in the newest block, and one in block 0, each set it."""
    G, D, block = 3, 8, 64
    q, K = rnd(49, G, D), rnd(50, 1100, D)
    scale = 1 / math.sqrt(D)
    last = (n - 1) // block
    toks = sorted(set(range(0, min(block, n))) | set(range(last * block, n)))
    for planted in (n - 1, 0):
        Kp = K.copy()
        Kp[planted] = 6.0 * q[1] / np.linalg.norm(q[1])
        want = [max(scale * sum(q[g, c] * Kp[t, c] for c in range(D)) for t in toks) for g in range(G)]
        np.testing.assert_allclose(O.pseudo_max(q, Kp, n, block, scale), want, rtol=1e-12)


@pytest.mark.parametrize("n", [64, 640, 1000, 1024 + 63])
def test_delta_invariants(n):
    """Pseudo-max <= true max (fail-safe); kept set contains every block the
    true max would keep; kept sets are nested in delta; delta -> inf keeps
    every complete block."""
    G, D, block = 4, 32, 64
    q, K = rnd(28, G, D) * 2, rnd(29, 1100, D)
    scale = 1 / math.sqrt(D)
    mt = O.pseudo_max(q, K, n, block, scale)
    m_true = (scale * q @ K[:n].T).max(axis=1)
    assert np.all(mt <= m_true + 1e-12)
    prev = None
    for delta in [0.5, 2.0, 5.0, 7.0]:
        sel, (blocks, margins) = O.delta_select_row(q, K, n, block, delta, scale)
        # blocks kept under the true-max threshold, same tentative scores
        true_keep = []
        for j in blocks:
            c, s = O.thumb_quantize(K[j * block:(j + 1) * block])
            st = scale * q @ O.thumb_dequant(c, s).T
            if np.max(st - m_true[:, None]) >= -delta:
                true_keep.append(int(j))
        assert set(true_keep) <= set(sel.tolist())
        if prev is not None:
            assert set(prev) <= set(sel.tolist())
        prev = sel.tolist()
    sel, _ = O.delta_select_row(q, K, n, block, 1e9, scale)
    assert sel.tolist() == list(range(-(-n // block)))
    assert set(O.delta_forced_blocks(n, block).tolist()) <= set(sel.tolist())


# ------------------------------------------------------- selection quality

@pytest.mark.parametrize("n", [1, 17, 200])
def test_recall_equals_mass_ratio_of_the_lse(n):
    """Recall of a page set = exp(lse over the set - lse over the context):
    a second route through the pinned attention routine, not the same sums."""
    rng = np.random.default_rng(11 + n)
    G, D, P = 3, 16, 8
    q, K = rng.normal(size=(G, D)), rng.normal(size=(n + 5, D))
    V = rng.normal(size=(n + 5, D))
    NP = O.num_pages(n, P)
    pages = rng.choice(NP, size=max(1, NP // 2), replace=False)
    rec = O.attention_mass_recall(q, K, pages, n, P, 0.3)
    _, lse_sel = O.sparse_attention_row(q, K, V, pages, n, P, 0.3)
    _, lse_all = O.softmax_attention(q, K[:n], V[:n], 0.3)
    np.testing.assert_allclose(rec, np.exp(lse_sel - lse_all), rtol=1e-12)


def test_recall_bounds_additivity_and_monotonicity():
    rng = np.random.default_rng(5)
    G, D, P, n = 2, 8, 4, 61
    q, K = rng.normal(size=(G, D)), rng.normal(size=(n, D))
    NP = O.num_pages(n, P)
    all_pages = np.arange(NP)
    np.testing.assert_allclose(O.attention_mass_recall(q, K, all_pages, n, P, 1.0), 1.0, rtol=0, atol=1e-15)
    assert np.all(O.attention_mass_recall(q, K, np.array([], dtype=np.int64), n, P, 1.0) == 0.0)
    a, b = all_pages[:5], all_pages[5:9]
    ra, rb = (O.attention_mass_recall(q, K, x, n, P, 1.0) for x in (a, b))
    rab = O.attention_mass_recall(q, K, np.concatenate([a, b]), n, P, 1.0)
    np.testing.assert_allclose(rab, ra + rb, rtol=1e-12)   # disjoint pages add up
    assert np.all(rab >= ra) and np.all(rab <= 1.0)
    # -1 padding and empty contexts
    np.testing.assert_allclose(O.attention_mass_recall(q, K, np.array([-1, 3, -1]), n, P, 1.0),
                               O.attention_mass_recall(q, K, np.array([3]), n, P, 1.0))
    assert np.all(O.attention_mass_recall(q, K, a, 0, P, 1.0) == 1.0)


# ------------------------------------------------------- ffd 8-bit residuals

def _bf16_exact(x):
    """Round float64 values to the nearest bf16 (ties to even), as float64."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def test_residual_golden():
    d = golden("ffd_residual_example.json")
    K = np.array(d["K"])
    codes, s = O.thumb_quantize(K)
    assert codes.tolist() == d["codes"] and s.tolist() == d["scale"]
    r = O.residual_quantize(K, codes, s)
    assert r.tolist() == d["res"]
    kt = O.refined_keys(codes, s, r)
    np.testing.assert_allclose(kt, d["refined"], rtol=0, atol=1e-15)
    assert abs(float(np.dot(d["q"], kt[1])) - d["score_token1"]) < 1e-15


def test_residual_error_bound():
    """The refined key is within s/1016 of the key (half a residual step of
    s/508; the nearest level is decided exactly); codes stay in range; an
    all-zero channel gets 0."""
    K = _bf16_exact(rnd(40, 64, 128) * np.exp(2 * rnd(41, 1, 128)))
    codes, s = O.thumb_quantize(K)
    r = O.residual_quantize(K, codes, s)
    assert r.dtype == np.int8 and np.abs(r.astype(int)).max() <= 127
    err = np.abs(K - O.refined_keys(codes, s, r))
    assert np.all(err <= s / 1016 * (1 + 1e-12) + 1e-300)
    assert np.max(err / s) > 0.9 / 1016      # the bound is met, not slack
    K[:, 5] = 0
    codes, s = O.thumb_quantize(K)
    assert np.all(O.residual_quantize(K, codes, s)[:, 5] == 0)


def test_residual_is_the_nearest_level_brute_force():
    """Exact rational arithmetic: r is the integer j in [-127, 127] nearest to
    (k - k^) * 508 / s, ties to the even j, for every element (no exclusion:
    the oracle decides it exactly).  Keys include exact half-integer
    quotients (s = 127 * 2^e, k = odd * 2^(e-3)), which must round to even."""
    from fractions import Fraction
    K = _bf16_exact(rnd(42, 64, 16) * np.exp(rnd(43, 1, 16)))
    K[3, :] = 0.0
    # channel 0: s = 127/64 (row 0), k = odd/512 on other rows: 508 k / s = odd/2
    K[:, 0] = _bf16_exact(K[:, 0] * (1.5 / np.abs(K[:, 0]).max()))
    K[0, 0] = 127.0 / 64
    K[1:9, 0] = np.array([1, 3, 5, 7, -1, -3, -9, 11]) / 512.0
    codes, s = O.thumb_quantize(K)
    r = O.residual_quantize(K, codes, s)
    halves = 0
    for t in range(K.shape[0]):
        for c in range(K.shape[1]):
            sc = Fraction(float(s[c]))
            kh = (Fraction(int(codes[t, c])) - Fraction(3, 2)) * sc / 2
            x = (Fraction(float(K[t, c])) - kh) * 508 / sc
            lo = math.floor(x)
            frac = x - lo
            j = lo + 1 if frac > Fraction(1, 2) else lo
            if frac == Fraction(1, 2):
                halves += 1
                j = lo if lo % 2 == 0 else lo + 1
            assert int(r[t, c]) == max(-127, min(127, j)), (t, c, x)
    assert halves >= 8


def test_refined_attention_brute_force():
    """Refined attention over a block list: complete blocks scored with the
    brute-force nearest-level keys, the partial newest block with the exact
    key, against explicit loops."""
    block, D, G = 64, 8, 2
    n = 3 * block + 10
    K = _bf16_exact(rnd(44, 4 * block, D) * 1.5)
    V = rnd(45, 4 * block, D)
    q = rnd(46, G, D)
    scale = 1 / math.sqrt(D)
    blocks = np.array([0, 2, 3])
    o, lse = O.refined_attention_row(q, K, V, blocks, n, block, scale)
    Kt = []
    toks = []
    for b in blocks.tolist():
        for t in range(b * block, min((b + 1) * block, n)):
            toks.append(t)
            if t >= (n // block) * block:
                Kt.append(K[t].tolist())       # partial block: exact key
                continue
            blk = K[b * block:(b + 1) * block]
            row = []
            for c in range(D):
                sc = max(abs(v) for v in blk[:, c])
                k = K[t, c]
                code = 3 if k >= sc / 2 else (2 if k >= 0 else (1 if k >= -sc / 2 else 0))
                kh = (code - 1.5) * sc / 2
                best = min(range(-127, 128), key=lambda j: (abs(k - (kh + j * sc / 508)), j % 2))
                row.append(kh + best * sc / 508 if sc > 0 else 0.0)
            Kt.append(row)
    ob, lb = brute_attention(q.tolist(), Kt, V[toks].tolist(), scale)
    np.testing.assert_allclose(o, ob, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(lse, lb, rtol=1e-12, atol=1e-12)
    # close to exact attention: k~ is within s/1016 of k
    oe, _ = O.sparse_attention_row(q, K, V, blocks, n, block, scale)
    assert np.max(np.abs(o - oe)) < 2e-2


# ------------------------------------------------------- input decoding, ties

def test_to_f64_decodes_bf16_bit_patterns():
    """bf16 is the top half of an IEEE float32: sign, 8 exponent bits, 7
    mantissa bits.  Patterns worked by hand: 0x3F80 = 1, 0xC040 = -3,
    0x4049 = 3.140625, 0x0001 = 2^-133 (smallest subnormal), 0x7F7F = the
    largest finite value (2 - 2^-7) * 2^127, 0xFF80 = -inf; fp32 input
    passes through unchanged."""
    bits = np.array([0x3F80, 0xC040, 0x4049, 0x0001, 0x7F7F, 0xFF80, 0x0000, 0x8000], dtype=np.uint16)
    got = O.to_f64(bits, "bf16")
    want = [1.0, -3.0, 3.140625, 2.0 ** -133, (2 - 2 ** -7) * 2.0 ** 127, -math.inf, 0.0, -0.0]
    assert got.dtype == np.float64
    assert got.tolist() == want
    assert math.copysign(1.0, got[7]) == -1.0
    x = np.array([0.1, -2.5, 1e-40], dtype=np.float32)
    assert O.to_f64(x, "f32").tolist() == [float(v) for v in x]


def test_kth_score_is_the_last_admitted_score():
    """The k-th ranked free page's score is the smallest score among the
    chosen free pages (brute force over the same tie rule), -inf when every
    page fits and +inf when the forced pages fill the budget."""
    for seed in range(8):
        rng = np.random.default_rng(300 + seed)
        NP = int(rng.integers(4, 12))
        score = rng.integers(-3, 4, NP).astype(float)
        forced = sorted(rng.choice(NP, size=int(rng.integers(0, 3)), replace=False).tolist())
        k = int(rng.integers(len(forced) + 1, NP))
        chosen = [p for p in brute_topk(score.tolist(), k, forced) if p not in forced]
        assert O.kth_score(score, k, np.array(forced, dtype=np.int64)) == min(score[p] for p in chosen)
    assert O.kth_score(np.zeros(3), 5, np.zeros(0, np.int64)) == -math.inf
    assert O.kth_score(np.zeros(6), 2, np.array([0, 5])) == math.inf


def test_delta_keep_rule_at_the_boundary():
    """FFD eqs. 1-2 keep a block when s~ - m~ + delta >= 0: a block whose
    margin is exactly -delta is kept, and one a hair below is not."""
    G, D, block, n = 2, 16, 64, 64 * 6 + 5
    q, K = rnd(47, G, D) * 2, rnd(48, n, D)
    scale = 1 / math.sqrt(D)
    blocks, margins = O.delta_block_margin(q, K, n, block, scale)
    i = int(np.argmin(np.abs(margins)))
    j = int(blocks[i])
    delta = -float(margins[i])
    assert j in O.delta_select_row(q, K, n, block, delta, scale)[0].tolist()
    below = float(np.nextafter(delta, -math.inf))
    assert j not in O.delta_select_row(q, K, n, block, below, scale)[0].tolist()
