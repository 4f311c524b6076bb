"""The seeded generators: deterministic, row-independent, shaped as stated."""
import numpy as np

from sparse_long_context_gb300 import workloads as W


def test_rows_are_independent_and_deterministic():
    s = W.spec("qwen7b", batch=2, ctx_len=[300, 257])
    full = W.generate(s)
    again = W.generate(s)
    assert np.array_equal(full.K, again.K) and np.array_equal(full.q, again.q)
    r = W.gen_row(s, 1, 2)
    assert np.array_equal(full.K[1, 2], r.K)
    assert np.array_equal(full.V[1, 2], r.V)
    G = s.group
    assert np.array_equal(full.q[1, 2 * G:3 * G], r.q)
    part = W.generate(s, rows=[(1, 2)])
    assert np.array_equal(part.K[1, 2], r.K)


def test_shapes_and_dtypes():
    for name in W.CONFIG_NAMES:
        s = W.spec(name, batch=1, ctx_len=200)
        t = W.generate(s)
        assert t.K.shape == (1, s.num_kv_heads, s.capacity, s.head_dim)
        assert t.q.shape == (1, s.num_q_heads, s.head_dim)
        assert t.K.dtype == (np.uint16 if s.dtype == "bf16" else np.float32)
        assert (t.sink is not None) == s.has_sink
        assert s.capacity % s.page_size == 0


def test_full_specs_match_the_workload_list():
    s = W.spec("qwen1p5b")
    assert (s.batch, s.num_q_heads, s.num_kv_heads, s.head_dim, s.ctx_len[0], s.page_size,
            s.k_pages * s.page_size) == (32, 12, 2, 128, 65536, 16, 2048)
    s = W.spec("gptoss")
    assert (s.batch, s.num_q_heads, s.num_kv_heads, s.head_dim, s.ctx_len[0], s.page_size,
            s.k_pages, s.n_sink_pages) == (4, 64, 8, 64, 131072, 1, 4096, 4)
    s = W.spec("ffd")
    assert (s.batch, s.num_q_heads, s.num_kv_heads, s.head_dim, s.ctx_len[0], s.block,
            s.delta) == (2, 32, 8, 128, 262144, 64, 5.0)


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0], dtype=np.float32)
    got = W.bf16_bits_to_f32(W.round_to_bf16_bits(x))
    assert got.tolist() == [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 0.0]


def test_planted_pages_are_what_the_tiny_queries_select():
    """Generator diagnostic: the tiny workload's query is the sum of its
    three planted pages' keys plus noise, so the oracle's top-8 pages hold
    all three.  On the outlier workloads the needle recall is reported by
    the diagnostics module, not asserted."""
    from oracle import sls_oracle as O
    from sparse_long_context_gb300 import diagnostics as DG
    s = W.spec("tiny")
    host = W.generate(s)
    G = s.group
    lists = []
    for b in range(s.batch):
        for h in range(s.num_kv_heads):
            q = O.to_f64(host.q[b, h * G:(h + 1) * G], s.dtype)
            K = O.to_f64(host.K[b, h], s.dtype)
            pages, _, _ = O.quest_select_row(q, K, int(host.ctx_len[b]), s.page_size, s.k_pages,
                                             s.n_sink_pages, s.n_local_tokens)
            lists.append(pages)
    nr = DG.needle_recall(np.stack(lists), None, host.needles, s.page_size, s.num_kv_heads)
    assert nr.size == s.rows and np.all(nr == 1.0)
    # the helper itself: counts bound each row's list, rows without needles are skipped
    lists = np.array([[3, 9, -1], [0, 1, 2]])
    needles = [[np.array([48, 49, 150]), None]]
    np.testing.assert_array_equal(DG.needle_recall(lists, np.array([1, 3]), needles, 16, 2), [0.5])
