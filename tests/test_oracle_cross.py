"""Cross-check of the two oracles: the plain C++ one (sls_oracle) and the
numpy one (numpy_oracle), written separately from the same pages, must agree
function by function on random inputs: bit for bit on integer results
(pages, tokens, codes, residuals), to 1e-12 relative on floating ones.  The
C++ oracle's whole-step functions (the timed CPU baseline) must agree with
its own row functions.  CPU only."""
import math

import numpy as np
import pytest

from oracle import numpy_oracle as N
from oracle import sls_oracle as C
from sparse_long_context_gb300 import workloads as W

RTOL, ATOL = 1e-12, 1e-13


def rnd(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


def close(a, b):
    np.testing.assert_allclose(a, b, rtol=RTOL, atol=ATOL)


@pytest.mark.parametrize("T,D,G,sink", [(0, 4, 2, False), (0, 4, 2, True), (1, 8, 1, False), (37, 16, 5, True),
                                        (300, 64, 8, True)])
def test_attention(T, D, G, sink):
    q, K, V = rnd(1, G, D) * 2, rnd(2, T, D), rnd(3, T, D)
    sk = rnd(4, G) * 3 if sink else None
    for a, b in zip(C.softmax_attention(q, K, V, 0.37, sk), N.softmax_attention(q, K, V, 0.37, sk)):
        close(a, b)
    if T:
        bounds = [(0, T // 3), (T // 3, T // 3), (T // 3, T)]
        pc, pn = C.split_partials(q, K, V, 0.37, bounds), N.split_partials(q, K, V, 0.37, bounds)
        for x, y in zip(pc, pn):
            for a, b in zip(x, y):
                close(a, b)
        for a, b in zip(C.combine_partials(pc, sk), N.combine_partials(pn, sk)):
            close(a, b)


@pytest.mark.parametrize("n,P", [(1, 16), (203, 16), (256, 16), (100, 1), (77, 4), (1000, 64)])
def test_quest(n, P):
    G, D = 6, 32
    q, K = rnd(5, G, D) * 2, rnd(6, 1024, D)
    a, b = C.page_minmax(K, n, P), N.page_minmax(K, n, P)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    close(C.quest_bound(q, *a), N.quest_bound(q, *b))
    assert C.num_pages(n, P) == N.num_pages(n, P)
    for k, ns, nl in [(8, 1, 64), (3, 0, 0), (5000, 4, 0), (20, 4, 0)]:
        fc, fn = C.forced_pages(n, P, ns, nl), N.forced_pages(n, P, ns, nl)
        np.testing.assert_array_equal(fc, fn)
        if len(fn) > k:
            continue
        rc = C.quest_select_row(q, K, n, P, k, ns, nl)
        rn = N.quest_select_row(q, K, n, P, k, ns, nl)
        np.testing.assert_array_equal(rc[0], rn[0])
        close(rc[1], rn[1])
        assert rc[2] == rn[2] or math.isclose(rc[2], rn[2], rel_tol=RTOL)
        np.testing.assert_array_equal(C.pages_to_tokens(rc[0], n, P), N.pages_to_tokens(rn[0], n, P))


def test_topk_with_ties():
    rng = np.random.default_rng(7)
    for _ in range(50):
        NP = int(rng.integers(1, 40))
        score = rng.integers(-2, 3, NP).astype(float)
        forced = np.sort(rng.choice(NP, size=int(rng.integers(0, min(NP, 4) + 1)), replace=False))
        k = int(rng.integers(max(len(forced), 1), NP + 3))
        np.testing.assert_array_equal(C.select_topk(score, k, forced), N.select_topk(score, k, forced))
        assert C.kth_score(score, k, forced) == N.kth_score(score, k, forced)
    with pytest.raises(ValueError):
        C.select_topk(np.zeros(10), 2, np.array([0, 1, 2]))


@pytest.mark.parametrize("n", [0, 5, 64, 65, 640, 1000, 64 * 16])
def test_thumbnails_and_delta(n):
    G, D, block = 4, 32, 64
    q = rnd(8, G, D) * 2
    K = rnd(9, 1100, D) * np.exp(rnd(10, 1, D))
    K[3, :4] = 0.0
    scale = 1 / math.sqrt(D)
    cc, sc = C.thumbnails_row(K, n, block)
    cn, sn = N.thumbnails_row(K, n, block)
    np.testing.assert_array_equal(cc, cn)
    np.testing.assert_array_equal(sc, sn)
    if cc.size:
        np.testing.assert_array_equal(C.pack_codes(cc), N.pack_codes(cn))
        np.testing.assert_array_equal(C.unpack_codes(C.pack_codes(cc)), cc)
        close(C.thumb_dequant(cc[:block], sc[0]), N.thumb_dequant(cn[:block], sn[0]))
    np.testing.assert_array_equal(C.delta_forced_blocks(n, block), N.delta_forced_blocks(n, block))
    if n == 0:
        return
    close(C.pseudo_max(q, K, n, block, scale), N.pseudo_max(q, K, n, block, scale))
    for delta in (0.5, 5.0, 1e9):
        a, (ba, ma) = C.delta_select_row(q, K, n, block, delta, scale)
        b, (bb, mb) = N.delta_select_row(q, K, n, block, delta, scale)
        np.testing.assert_array_equal(ba, bb)
        close(ma, mb)
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("n", [64, 64 * 3 + 10, 64 * 8])
def test_residuals_and_refined_attention(n):
    G, D, block = 3, 16, 64
    K = W.bf16_bits_to_f32(W.round_to_bf16_bits(rnd(11, 600, D) * np.exp(rnd(12, 1, D)))).astype(np.float64)
    V = rnd(13, 600, D)
    q = rnd(14, G, D)
    a, b = C.residuals_row(K, n, block), N.residuals_row(K, n, block)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    close(C.refined_keys(a[0][:block], a[1][0], a[2][:block]), N.refined_keys(b[0][:block], b[1][0], b[2][:block]))
    blocks = np.arange(0, -(-n // block), 2)
    sink = rnd(15, G)
    for x, y in zip(C.refined_attention_row(q, K, V, blocks, n, block, 0.25, sink),
                    N.refined_attention_row(q, K, V, blocks, n, block, 0.25, sink)):
        close(x, y)


@pytest.mark.parametrize("n", [0, 1, 17, 300])
def test_recall_and_sparse_attention(n):
    G, D, P = 3, 16, 8
    q, K, V = rnd(16, G, D), rnd(17, n + 9, D), rnd(18, n + 9, D)
    pages = np.array([-1, 0, 2, 5, 7, -1])
    close(C.attention_mass_recall(q, K, pages, n, P, 0.3), N.attention_mass_recall(q, K, pages, n, P, 0.3))
    for x, y in zip(C.sparse_attention_row(q, K, V, pages, n, P, 0.3, rnd(19, G)),
                    N.sparse_attention_row(q, K, V, pages, n, P, 0.3, rnd(19, G))):
        close(x, y)


def test_bf16_decoding():
    bits = np.random.default_rng(20).integers(0, 1 << 16, 5000, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]          # no NaN / inf patterns
    np.testing.assert_array_equal(C.to_f64(bits, "bf16"), N.to_f64(bits, "bf16"))


# ------------------------------------------------ whole steps vs row functions

def _rows_f64(s, host, r):
    b, h = divmod(r, s.num_kv_heads)
    G = s.group
    return (C.to_f64(host.q[b, h * G:(h + 1) * G], s.dtype), C.to_f64(host.K[b, h], s.dtype),
            C.to_f64(host.V[b, h], s.dtype), int(host.ctx_len[b]),
            None if host.sink is None else host.sink[h * G:(h + 1) * G].astype(np.float64))


@pytest.mark.parametrize("name,kw", [("qwen1p5b", dict(batch=2, ctx_len=[1000, 1531])), ("tiny", {}),
                                     ("gptoss", dict(batch=1, ctx_len=700)),
                                     ("qwen7b", dict(batch=1, ctx_len=40))])
def test_quest_step_equals_row_functions(name, kw):
    s = W.spec(name, **kw)
    if name == "gptoss":
        s.k_pages = 64
    host = W.generate(s)
    rows = list(range(s.rows))
    pages, o, lse, busy, nbytes, reps = C.quest_step(
        host.q, host.K, host.V, host.ctx_len, s.num_q_heads, s.page_size, s.k_pages, s.n_sink_pages,
        s.n_local_tokens, s.scale, host.sink, rows, threads=2)
    assert reps == len(rows) and busy > 0 and nbytes > 0
    for i, r in enumerate(rows):
        q, K, V, n, sink = _rows_f64(s, host, r)
        want, _, _ = C.quest_select_row(q, K, n, s.page_size, s.k_pages, s.n_sink_pages, s.n_local_tokens)
        got = pages[i][pages[i] >= 0]
        np.testing.assert_array_equal(got, want)
        ow, lw = C.sparse_attention_row(q, K, V, want, n, s.page_size, s.scale, sink)
        np.testing.assert_array_equal(o[i], ow)
        np.testing.assert_array_equal(lse[i], lw)


@pytest.mark.parametrize("refined", [False, True])
def test_delta_step_equals_row_functions(refined):
    s = W.spec("ffd", batch=1, ctx_len=64 * 20 + 9)
    host = W.generate(s)
    rows = [0, 3, 7]
    count, blocks, o, lse, busy, nbytes, reps = C.delta_step(
        host.q, host.K, host.V, host.ctx_len, s.num_q_heads, s.block, s.delta, s.scale, host.sink, rows,
        refined=refined, threads=3)
    assert reps == len(rows) and nbytes > 0
    for i, r in enumerate(rows):
        q, K, V, n, sink = _rows_f64(s, host, r)
        want, _ = C.delta_select_row(q, K, n, s.block, s.delta, s.scale)
        np.testing.assert_array_equal(blocks[i, :count[i]], want)
        if refined:
            ow, lw = C.refined_attention_row(q, K, V, want, n, s.block, s.scale, sink)
        else:
            ow, lw = C.sparse_attention_row(q, K, V, want, n, s.block, s.scale, sink)
        close(o[i], ow)
        close(lse[i], lw)
