"""CUDA path vs the fp64 oracle, through the C ABI, on seeded workloads.

Small cases cover every row; full-size workloads (the benchmark's launch
configuration) check sampled rows the oracle computes one by one."""
import numpy as np
import pytest
import torch

from oracle import sls_oracle as O
from sparse_long_context_gb300 import ops
from sparse_long_context_gb300 import workloads as W

from tests import parity as PT

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def small(name, **kw):
    return W.spec(name, **kw)


# The small parity cases: several tiles, ragged tails, partial last pages.
SMALL_QUEST = {
    "tiny": dict(),
    "tiny_ragged": dict(name="tiny", ctx_len=[1000]),
    "qwen7b_ragged": dict(name="qwen7b", ctx_len=[8197, 3000, 700], capacity=8208),
    "qwen1p5b_4k": dict(name="qwen1p5b", batch=3, ctx_len=4096),
    # an odd number of rows, and rows of different contexts, one within the budget
    "odd_rows": dict(name="qwen7b", batch=3, ctx_len=[6000, 300, 4100], capacity=6016, num_q_heads=12,
                     num_kv_heads=3),
    "gptoss_ragged": dict(name="gptoss", ctx_len=[20000, 5003], capacity=20000),
    # D = 64 and G = 8 with 16-token pages (the tensor-map path at its other head size)
    "gptoss_p16": dict(name="gptoss", ctx_len=[5003, 1000], capacity=5008, page_size=16, k_pages=64,
                       n_sink_pages=1),
}
SMALL_DELTA = {
    "ffd_ragged": dict(name="ffd", ctx_len=[65536 + 100, 20000], capacity=65536 + 128),
    "ffd_aligned": dict(name="ffd", batch=1, ctx_len=8192),
    # the tensor-core scan's other forms: G = 8 (one block per weight set),
    # D = 64, 16- and 32-token blocks, odd block counts per part
    "ffd_g8_d64_b16": dict(name="ffd", ctx_len=[5000, 777], num_q_heads=32, num_kv_heads=4, head_dim=64,
                           block=16, page_size=16),
    "ffd_g2_b32": dict(name="ffd", ctx_len=[12345, 64 * 37 + 1], num_q_heads=16, num_kv_heads=8, block=32,
                       page_size=32),
    "ffd_d64_b64": dict(name="ffd", ctx_len=[30000 + 64, 64 * 3 + 17], head_dim=64),
}


def make(case):
    kw = dict(case)
    name = kw.pop("name", None)
    fields = {f: kw.pop(f) for f in ("page_size", "k_pages", "n_sink_pages", "block", "num_q_heads", "num_kv_heads",
                                     "head_dim") if f in kw}
    s = W.spec(name, **kw)
    for f, v in fields.items():
        setattr(s, f, v)
    return s


def quest_case(key):
    return make(dict(SMALL_QUEST[key], name=SMALL_QUEST[key].get("name", key)))


# ----------------------------------------------------------------- metadata

@pytest.mark.parametrize("key", ["tiny_ragged", "qwen7b_ragged"])
def test_pagemeta_build_is_exact(key):
    s = quest_case(key)
    host = W.generate(s)
    dw = PT.upload(s, host)
    kmin, kmax = dw.kmin.float().cpu().numpy(), dw.kmax.float().cpu().numpy()
    for b in range(s.batch):
        for h in range(s.num_kv_heads):
            n = host.ctx_len[b]
            omin, omax = O.page_minmax(O.to_f64(host.K[b, h], s.dtype), n, s.page_size)
            np.testing.assert_array_equal(kmin[b, h, :len(omin)], omin)
            np.testing.assert_array_equal(kmax[b, h, :len(omax)], omax)


def test_pagemeta_update_matches_oracle():
    s = W.spec("qwen7b", batch=2, ctx_len=[300, 517], capacity=640)
    host = W.generate(s)
    dw = PT.upload(s, host)
    # start from summaries of shorter prefixes, then append one token at a time
    n0 = np.array([260, 490], dtype=np.int32)
    kmin, kmax = ops.pagemeta_build(dw.desc, dw.K, torch.from_numpy(n0).cuda())
    cur = n0.copy()
    while np.any(cur < host.ctx_len):
        pos = np.where(cur < host.ctx_len, cur, -1).astype(np.int32)
        ops.pagemeta_update(dw.desc, dw.K, torch.from_numpy(pos).cuda(), kmin, kmax)
        cur = np.minimum(cur + 1, host.ctx_len)
    got_min, got_max = kmin.float().cpu().numpy(), kmax.float().cpu().numpy()
    for b in range(2):
        for h in range(s.num_kv_heads):
            omin, omax = O.page_minmax(O.to_f64(host.K[b, h], s.dtype), host.ctx_len[b], 16)
            np.testing.assert_array_equal(got_min[b, h, :len(omin)], omin)
            np.testing.assert_array_equal(got_max[b, h, :len(omax)], omax)


@pytest.mark.parametrize("ctx", [[64 * 9 + 5, 64 * 3], [64 * 40]])
def test_thumbnails_are_bit_exact(ctx):
    s = W.spec("ffd", ctx_len=ctx, capacity=64 * 40)
    host = W.generate(s)
    dw = PT.upload(s, host)
    codes, scales = dw.codes.cpu().numpy(), dw.scales.float().cpu().numpy()
    for b in range(s.batch):
        for h in range(s.num_kv_heads):
            n = host.ctx_len[b]
            oc, osc = O.thumbnails_row(O.to_f64(host.K[b, h], s.dtype), n, 64)
            nfull = n // 64
            np.testing.assert_array_equal(codes[b, h, :nfull * 64], O.pack_codes(oc))
            np.testing.assert_array_equal(scales[b, h, :nfull], osc)


def test_thumb_update_completes_blocks():
    s = W.spec("ffd", batch=2, ctx_len=[64 * 5, 64 * 7], capacity=64 * 8)
    host = W.generate(s)
    dw = PT.upload(s, host)
    start = torch.tensor([64 * 3 + 10, 64 * 6 + 60], dtype=torch.int32, device="cuda")
    codes, scales = ops.thumb_build(dw.desc, dw.K, start, 64)
    cur = start.cpu().numpy().copy()
    end = host.ctx_len
    while np.any(cur < end):
        pos = np.where(cur < end, cur, -1).astype(np.int32)
        ops.thumb_update(dw.desc, dw.K, torch.from_numpy(pos).cuda(), 64, codes, scales)
        cur = np.minimum(cur + 1, end)
    codes, scales = codes.cpu().numpy(), scales.float().cpu().numpy()
    for b in range(2):
        for h in range(s.num_kv_heads):
            oc, osc = O.thumbnails_row(O.to_f64(host.K[b, h], s.dtype), end[b], 64)
            nfull = end[b] // 64
            np.testing.assert_array_equal(codes[b, h, :nfull * 64], O.pack_codes(oc))
            np.testing.assert_array_equal(scales[b, h, :nfull], osc)


# ---------------------------------------------------------- select + attend

def check_all_rows(s, host, sel, cnt, out, lse, dw=None):
    """Every row: selection parity (ties counted), output parity where the
    sets are identical, and attend parity on the oracle's own page list."""
    G = s.group
    ties = 0
    orcs = []
    exact_rows = []
    for b in range(s.batch):
        for h in range(s.num_kv_heads):
            r = b * s.num_kv_heads + h
            orc = PT.oracle_row(s, host, b, h)
            orcs.append(orc)
            if s.selector == "quest":
                t = PT.check_quest_list(sel[r], orc, int(host.ctx_len[b]), s.page_size, s.k_pages)
            else:
                t = PT.check_delta_list(int(cnt[r]), sel[r], orc, s.delta)
            ties += t
            if t == 0:
                exact_rows.append((b, h, orc))
    for b, h, orc in exact_rows:
        PT.assert_close(s, out[b, h * G:(h + 1) * G], orc.o, f"output row {(b, h)}")
        fin = np.isfinite(orc.lse)
        np.testing.assert_allclose(lse[b, h * G:(h + 1) * G][fin], orc.lse[fin], rtol=1e-4, atol=1e-4)
    if dw is not None:
        o2, _ = PT.attend_on(dw, [o.pages for o in orcs])
        for b in range(s.batch):
            for h in range(s.num_kv_heads):
                ref = orcs[b * s.num_kv_heads + h].o
                PT.assert_close(s, o2[b, h * G:(h + 1) * G], ref, f"attend on oracle set {(b, h)}")
    return ties


# kernels of a step: the one-launch Quest step (the default for bf16 pages of
# >= 16 tokens), select + the tensor-map fed attend, select + the register-fed
# attend, CUDA cores
PATHS = {"step": dict(), "tma": dict(), "registers": dict(no_tma=True), "cuda_cores": dict(cuda_cores=True)}
ONE_LAUNCH = {"step": True, "tma": False, "registers": True, "cuda_cores": True}


@pytest.mark.parametrize("key", list(SMALL_QUEST))
@pytest.mark.parametrize("path", list(PATHS))
def test_quest_step_small(key, path):
    s = quest_case(key)
    host = W.generate(s)
    dw = PT.upload(s, host, **PATHS[path])
    sel, cnt, out, lse = PT.run_step(dw, one_launch=ONE_LAUNCH[path])
    ties = check_all_rows(s, host, sel, cnt, out, lse, dw)
    print(f"{key}: boundary ties {ties}")


@pytest.mark.parametrize("key", list(SMALL_DELTA))
@pytest.mark.parametrize("path", ["step", "registers", "cuda_cores"])
def test_delta_step_small(key, path):
    s = make(SMALL_DELTA[key])
    host = W.generate(s)
    dw = PT.upload(s, host, **PATHS[path])
    sel, cnt, out, lse = PT.run_step(dw)
    ties = check_all_rows(s, host, sel, cnt, out, lse, dw)
    kept = cnt.sum() / sum((n + s.block - 1) // s.block for n in host.ctx_len for _ in range(s.num_kv_heads))
    print(f"{key}: kept fraction {kept:.3f}, boundary ties {ties}")


@pytest.mark.parametrize("key", ["qwen7b_ragged", "gptoss_ragged", "gptoss_p16"])
def test_fused_and_separate_combine_agree_and_reuse_workspace(key):
    s = quest_case(key)
    host = W.generate(s)
    dw = PT.upload(s, host)
    results = {}
    for name, kw in (("one_launch", dict(fused=True)), ("two_launch", dict(fused=True, one_launch=False))):
        step = PT.H.make_step(dw, **kw)
        outs = []
        for _ in range(3):  # reused workspaces: the arrival tickets are back at zero after every call
            o, l = step(dw.q, dw.K, dw.V, dw.kmin, dw.kmax, dw.ctx, dw.sink)
            outs.append((o.float().clone(), l.clone(), step.page_idx.clone()))
        ops.pipeline_check()
        for o, l, p in outs:
            assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1]) and torch.equal(p, outs[0][2])
        results[name] = outs[0]
    sel, _, out_sep, lse_sep = PT.run_step(dw, fused=False)
    for name, (o, l, p) in results.items():
        check_all_rows(s, host, p.cpu().numpy(), None, o.cpu().numpy().astype(np.float64),
                       l.cpu().numpy().astype(np.float64))
        assert np.abs(o.cpu().numpy() - out_sep).max() < 2e-2, name
    check_all_rows(s, host, sel, None, out_sep, lse_sep)


def test_sparsity_gate_attends_short_contexts_densely():
    """mlxcel's gate: rows with fewer than min_sparsity * k * P context tokens
    skip the selection and attend every token; longer rows stay sparse."""
    s = W.spec("qwen7b", batch=3, ctx_len=[1000, 5000, 20000], capacity=20000)
    host = W.generate(s)
    dw = PT.upload(s, host)
    step = ops.QuestDecode(dw.desc, s.k_pages, s.n_sink_pages, s.n_local_tokens, min_sparsity=4.0)
    ops.get_stats(reset=True)
    out, lse = step(dw.q, dw.K, dw.V, dw.kmin, dw.kmax, dw.ctx)
    ops.pipeline_check()
    st = ops.get_stats(reset=True)
    assert st["step_rows_dense"] == 2 * s.num_kv_heads and st["quest_step_one_launch"] == 1, st
    out = out.float().cpu().numpy().astype(np.float64)
    sel = step.page_idx.cpu().numpy()
    G, H = s.group, s.num_kv_heads
    for b in (0, 1):  # 1000 and 5000 tokens < 4 * 128 * 16: dense
        assert np.all(sel[b * H:(b + 1) * H] == -1)
        n = int(host.ctx_len[b])
        for h in range(H):
            q = O.to_f64(host.q[b, h * G:(h + 1) * G], "bf16")
            ref, _ = O.softmax_attention(q, O.to_f64(host.K[b, h, :n], "bf16"),
                                         O.to_f64(host.V[b, h, :n], "bf16"), s.scale)
            PT.assert_close(s, out[b, h * G:(h + 1) * G], ref, f"dense row {(b, h)}")
    for h in range(H):  # 20000 tokens: sparse, as without the gate
        orc = PT.oracle_row(s, host, 2, h)
        PT.check_quest_list(sel[2 * H + h], orc, 20000, 16, s.k_pages)
        PT.assert_close(s, out[2, h * G:(h + 1) * G], orc.o, f"sparse row {h}")


def test_one_launch_step_long_rows():
    """Rows of 8192 pages: the row's keys no longer fit the registers of the
    CTA, the shared-memory selection runs."""
    s = W.spec("qwen1p5b", batch=1, ctx_len=[131072], capacity=131072)
    host = W.generate(s)
    dw = PT.upload(s, host)
    sel, _, out, lse = PT.run_step(dw)
    assert ops.quest_step_splits(dw.desc, s.k_pages) > 0
    check_all_rows(s, host, sel, None, out, lse)


@pytest.mark.parametrize("ctx", [[0, 1, 17, 5000], [16, 2048, 2049, 4095]])
def test_one_launch_step_edge_contexts(ctx):
    """Empty rows, single pages, budgets covering every page and just not."""
    s = W.spec("qwen7b", batch=len(ctx), ctx_len=ctx, capacity=5008)
    host = W.generate(s)
    dw = PT.upload(s, host)
    sel, _, out, lse = PT.run_step(dw)
    rows = s.num_kv_heads
    if ctx[0] == 0:
        assert np.all(sel[:rows] == -1) and np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    check_all_rows(s, host, sel, None, out, lse)


def _bits(x):
    from sparse_long_context_gb300.workloads import round_to_bf16_bits
    return round_to_bf16_bits(np.asarray(x, dtype=np.float32))


def test_topk_exact_ties_go_to_lower_pages():
    """Pages repeat a few key patterns, so many bounds are exactly equal."""
    s = W.spec("qwen7b", batch=1, ctx_len=[8192])
    host = W.generate(s)
    pat = host.K[0, :, :4 * 16].copy()                      # 4 distinct pages per row
    for p in range(1, 512):
        host.K[0, :, p * 16:(p + 1) * 16] = pat[:, (p % 4) * 16:(p % 4 + 1) * 16]
    dw = PT.upload(s, host)
    sel, cnt, out, lse = PT.run_step(dw)
    for h in range(s.num_kv_heads):
        orc = PT.oracle_row(s, host, 0, h)
        assert np.array_equal(sel[h], orc.pages), h   # equal scores: no tolerance needed


def test_topk_scores_spanning_many_octaves():
    """Bounds spread over far more than 16 octaves: the k-th score lies below
    the fast path's window and the general radix select decides."""
    s = W.spec("qwen7b", batch=1, ctx_len=[8192])
    s.k_pages = 256
    host = W.generate(s)
    K = W.bf16_bits_to_f32(host.K[0]).copy()
    q = W.bf16_bits_to_f32(host.q[0])
    for h in range(s.num_kv_heads):
        g = np.abs(q[h * s.group:(h + 1) * s.group]).mean(axis=0)
        sgn = np.sign(q[h * s.group])                        # keys aligned with head 0's query
        base = np.abs(K[h]) * sgn[None, :]
        scale = np.exp2(-(np.arange(8192) // 16) / 8.0).astype(np.float32)[:, None]
        K[h] = base * scale
    host.K[0] = _bits(K)
    dw = PT.upload(s, host)
    sel, _, out, lse = PT.run_step(dw)
    for h in range(s.num_kv_heads):
        orc = PT.oracle_row(s, host, 0, h)
        t = PT.check_quest_list(sel[h], orc, 8192, 16, s.k_pages)
        assert t <= 2


@pytest.mark.parametrize("splits,npg", [(5, 50), (5, 100), (5, 300), (2, 128), (16, 20), (16, 128)])
def test_topk_with_the_best_pages_in_one_split(splits, npg):
    """A run of `npg` pages whose keys align with the query holds most of the
    row's top k: a split may hold more than its share of the chosen pages
    (its candidates alone then do not decide the selection)."""
    s = W.spec("qwen7b", batch=1, ctx_len=[8192])
    host = W.generate(s)
    K = W.bf16_bits_to_f32(host.K[0]).copy()
    q = W.bf16_bits_to_f32(host.q[0])
    p0 = 200
    for h in range(s.num_kv_heads):
        sgn = np.sign(q[h * s.group])
        t0, t1 = p0 * 16, (p0 + npg) * 16
        K[h, t0:t1] = np.abs(K[h, t0:t1]) * sgn[None, :] * 1.5
    host.K[0] = _bits(K)
    dw = PT.upload(s, host)
    ops.get_stats(reset=True)
    sel, cnt, out, lse = PT.run_step(dw, num_splits=splits)
    st = ops.get_stats(reset=True)
    check_all_rows(s, host, sel, cnt, out, lse)
    assert st["quest_step_one_launch"] == 1 and st["quest_step_two_launch"] == 0
    # a split holding more of the row's top k than it sends forces the all-keys selection:
    # with 5 splits of 112 pages the run 200-299 puts 76 of the top 128 into split 2 (it
    # sends about 60); with 16 splits of 32 pages, the run 200-327 fills splits 7-9 (each
    # sends about 24).  With 2 splits each sends its whole top k, so the candidates decide.
    if (splits, npg) in ((5, 100), (16, 128)):
        assert st["step_rows_all_keys"] >= 1, st
    if splits == 2:
        assert st["step_rows_all_keys"] == 0, st


def _wide_step(s, host, **kw):
    dw = PT.upload(s, host, **kw)
    ops.get_stats(reset=True)
    sel, cnt, out, lse = PT.run_step(dw, one_launch=False)
    return dw, sel, cnt, out, lse, ops.get_stats(reset=True)


@pytest.mark.parametrize("ctx", [[20000, 9000], [65536, 131072 - 5]])
def test_wide_rows_rank_the_scoring_ctas_candidates(ctx):
    """Rows of more than 8192 one-token pages: the scoring CTAs send their
    candidates and the top-k CTA ranks only those; the check T >= every
    CTA's threshold holds, so no row falls back to all keys."""
    s = W.spec("gptoss", batch=len(ctx), ctx_len=ctx, capacity=max(ctx))
    host = W.generate(s)
    dw, sel, cnt, out, lse, st = _wide_step(s, host)
    check_all_rows(s, host, sel, cnt, out, lse)
    assert st["select_rows_all_keys"] == 0, st


@pytest.mark.parametrize("run", [600, 3000])
def test_wide_rows_with_the_best_tokens_in_one_place(run):
    """A run of tokens whose keys align with the query holds most of the
    row's top 4096: a scoring CTA holds far more than twice its share, the
    check fails and the row is selected from all its keys."""
    s = W.spec("gptoss", batch=1, ctx_len=[40000], capacity=40000)
    host = W.generate(s)
    K = W.bf16_bits_to_f32(host.K[0]).copy()
    q = W.bf16_bits_to_f32(host.q[0])
    t0 = 12000
    for h in range(s.num_kv_heads):
        sgn = np.sign(q[h * s.group])
        K[h, t0:t0 + run] = np.abs(K[h, t0:t0 + run]) * sgn[None, :] * 1.5
    host.K[0] = _bits(K)
    dw, sel, cnt, out, lse, st = _wide_step(s, host)
    check_all_rows(s, host, sel, cnt, out, lse)
    if run == 3000:
        assert st["select_rows_all_keys"] >= 1, st


def test_wide_rows_exact_ties_go_to_lower_pages():
    """Sixteen-token pages repeating four key patterns over 10000 pages: the
    bounds take four values, so T's bin narrows to one value and the ties at
    the budget boundary go to the lower pages."""
    s = W.spec("qwen7b", batch=1, ctx_len=[160000], capacity=160000)
    s.k_pages = 3000
    host = W.generate(s)
    pat = host.K[0, :, :4 * 16].copy()
    for p in range(1, 10000):
        host.K[0, :, p * 16:(p + 1) * 16] = pat[:, (p % 4) * 16:(p % 4 + 1) * 16]
    dw, sel, cnt, out, lse, st = _wide_step(s, host)
    for h in range(s.num_kv_heads):
        orc = PT.oracle_row(s, host, 0, h)
        assert np.array_equal(sel[h], orc.pages), h   # equal scores: no tolerance needed


# 2..16 splits combine inside a thread-block cluster, more through global memory
@pytest.mark.parametrize("splits", [1, 2, 3, 8, 13, 16, 17, 64, 1024])
def test_split_counts_do_not_change_the_result(splits):
    s = W.spec("qwen7b", batch=2, ctx_len=[2000, 33], capacity=2048)
    host = W.generate(s)
    dw = PT.upload(s, host)
    sel, cnt, out, lse = PT.run_step(dw, num_splits=splits)
    check_all_rows(s, host, sel, cnt, out, lse)


def test_dense_attend_matches_oracle():
    s = W.spec("qwen7b", batch=2, ctx_len=[3001, 64], capacity=3008)
    host = W.generate(s)
    dw = PT.upload(s, host)
    parts = ops.sparse_decode_attend(dw.desc, dw.q, dw.K, dw.V, None, dw.ctx, 8)
    out, _ = ops.combine_splits(dw.desc, parts)
    out = out.float().cpu().numpy()
    G = s.group
    for b in range(2):
        for h in range(s.num_kv_heads):
            n = host.ctx_len[b]
            q = O.to_f64(host.q[b, h * G:(h + 1) * G], "bf16")
            K, V = O.to_f64(host.K[b, h, :n], "bf16"), O.to_f64(host.V[b, h, :n], "bf16")
            ref, _ = O.softmax_attention(q, K, V, s.scale)
            PT.assert_close(s, out[b, h * G:(h + 1) * G], ref, "dense")


def test_budget_covering_every_page_equals_dense():
    s = W.spec("qwen7b", batch=1, ctx_len=[1000], capacity=2048)
    s.k_pages = 128  # >= 63 pages
    host = W.generate(s)
    dw = PT.upload(s, host)
    sel, _, out, _ = PT.run_step(dw)
    assert np.array_equal(sel[0, :63], np.arange(63)) and np.all(sel[:, 63:] == -1)
    G = s.group
    for h in range(s.num_kv_heads):
        q = O.to_f64(host.q[0, h * G:(h + 1) * G], "bf16")
        ref, _ = O.softmax_attention(q, O.to_f64(host.K[0, h, :1000], "bf16"),
                                     O.to_f64(host.V[0, h, :1000], "bf16"), s.scale)
        PT.assert_close(s, out[0, h * G:(h + 1) * G], ref, "dense-equivalent")


def test_sparse_output_differs_from_dense():
    """A kernel that ignored the page list would return dense attention."""
    s = W.spec("qwen7b", batch=1, ctx_len=[16384])
    host = W.generate(s)
    dw = PT.upload(s, host)
    _, _, out, _ = PT.run_step(dw)
    parts = ops.sparse_decode_attend(dw.desc, dw.q, dw.K, dw.V, None, dw.ctx, 16)
    dense, _ = ops.combine_splits(dw.desc, parts)
    _, rel = PT.out_errors(out, dense.float().cpu().numpy())
    assert rel > 1e-3


def test_empty_and_single_token_rows():
    s = W.spec("gptoss", batch=3, ctx_len=[0, 1, 4100], capacity=4352)
    s.k_pages = 4096
    host = W.generate(s)
    dw = PT.upload(s, host)
    sel, _, out, lse = PT.run_step(dw)
    rows = s.num_kv_heads
    assert np.all(sel[:rows] == -1)
    assert np.all(out[0] == 0)
    np.testing.assert_allclose(lse[0], host.sink.astype(np.float64), rtol=1e-6)  # only the sink
    check_all_rows(s, host, sel, None, out, lse)
    # without a sink an empty row gives 0 and -inf
    parts = ops.sparse_decode_attend(dw.desc, dw.q, dw.K, dw.V, torch.from_numpy(sel).cuda(), dw.ctx, 4)
    out2, lse2 = ops.combine_splits(dw.desc, parts, None)
    assert torch.all(out2[0] == 0) and torch.all(torch.isinf(lse2[0]))


@pytest.mark.parametrize("path", ["tma", "registers"])
def test_cache_past_the_context_is_never_used(path):
    """Slots past each sequence's context hold NaN: the partial last page must
    be masked (scores and values), not multiplied by a zero weight."""
    s = W.spec("qwen7b", batch=2, ctx_len=[1000 + 5, 37], capacity=1024)
    host = W.generate(s)
    dw = PT.upload(s, host, **PATHS[path])
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16, device="cuda")
    for b, n in enumerate(host.ctx_len):
        dw.K[b, :, n:] = nan
        dw.V[b, :, n:] = nan
    npages = [-(-int(n) // 16) for n in host.ctx_len]
    lists = [np.arange(npages[b]) for b in range(2) for _ in range(s.num_kv_heads)]
    o, _ = PT.attend_on(dw, lists, num_splits=3)
    ops.pipeline_check()
    assert np.isfinite(o).all()
    G = s.group
    for b in range(2):
        n = int(host.ctx_len[b])
        for h in range(s.num_kv_heads):
            q = O.to_f64(host.q[b, h * G:(h + 1) * G], "bf16")
            ref, _ = O.softmax_attention(q, O.to_f64(host.K[b, h, :n], "bf16"),
                                         O.to_f64(host.V[b, h, :n], "bf16"), s.scale)
            PT.assert_close(s, o[b, h * G:(h + 1) * G], ref, f"row {(b, h)}")


def test_padded_page_lists_are_skipped():
    s = W.spec("qwen7b", batch=1, ctx_len=[640], capacity=640)
    host = W.generate(s)
    dw = PT.upload(s, host)
    lists = [np.array([3, 7, 39]), np.array([0]), np.array([], dtype=np.int64), np.array([12, 13])]
    o, lse = PT.attend_on(dw, lists, num_splits=2)
    G = s.group
    for h, pages in enumerate(lists):
        q = O.to_f64(host.q[0, h * G:(h + 1) * G], "bf16")
        ref, rl = O.sparse_attention_row(q, O.to_f64(host.K[0, h], "bf16"), O.to_f64(host.V[0, h], "bf16"),
                                         pages, 640, 16, s.scale)
        PT.assert_close(s, o[0, h * G:(h + 1) * G], ref, f"list {h}")


# ------------------------------------------------- full sizes, sampled rows

FULL = ["qwen1p5b", "qwen7b", "gptoss", "ffd"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_rows(name):
    s = W.spec(name)
    host = W.generate(s)
    dw = PT.upload(s, host)
    sel, cnt, out, lse = PT.run_step(dw)   # default launch configuration, as benchmarked
    # the first and last rows, every KV head of one sequence (the rows that share a q), and
    # seeded others: 8 rows (or all of them)
    rng = np.random.default_rng(7)
    b_mid = s.batch // 2
    picked = {0, s.rows - 1} | {b_mid * s.num_kv_heads + h for h in range(s.num_kv_heads)}
    others = [r for r in rng.permutation(s.rows).tolist() if r not in picked]
    rows = sorted(picked | set(others[:max(0, 8 - len(picked))]))
    G = s.group
    ties = 0
    for r in rows:
        b, h = divmod(r, s.num_kv_heads)
        orc = PT.oracle_row(s, host, b, h)
        if s.selector == "quest":
            t = PT.check_quest_list(sel[r], orc, int(host.ctx_len[b]), s.page_size, s.k_pages)
        else:
            t = PT.check_delta_list(int(cnt[r]), sel[r], orc, s.delta)
        ties += t
        if t == 0:
            PT.assert_close(s, out[b, h * G:(h + 1) * G], orc.o, f"{name} row {r}")
    print(f"{name}: rows {rows} boundary ties {ties}"
          + (f" kept {cnt.sum() / (s.rows * (s.ctx_len[0] // 64)):.3f}" if cnt is not None else ""))


# ------------------------------------------------------- selection quality

RECALL_ATOL = 2e-4  # ratio of fp32 sums of exp over up to 2^17 tokens, scores from bf16 inputs


@pytest.mark.parametrize("key", ["qwen7b_ragged", "gptoss_ragged", "gptoss_p16"])
def test_selection_recall_matches_oracle(key):
    s = quest_case(key)
    host = W.generate(s)
    dw = PT.upload(s, host)
    sel, _, _, _ = PT.run_step(dw)
    rec = ops.selection_recall(dw.desc, dw.q, dw.K, torch.from_numpy(sel).cuda(), dw.ctx).cpu().numpy()
    G = s.group
    for b in range(s.batch):
        n = int(host.ctx_len[b])
        for h in range(s.num_kv_heads):
            q = O.to_f64(host.q[b, h * G:(h + 1) * G], s.dtype)
            ref = O.attention_mass_recall(q, O.to_f64(host.K[b, h], s.dtype), sel[b * s.num_kv_heads + h], n,
                                          s.page_size, s.scale)
            np.testing.assert_allclose(rec[b, h * G:(h + 1) * G], ref, rtol=0, atol=RECALL_ATOL)


def test_selection_recall_of_delta_lists_and_edge_rows():
    s = make(SMALL_DELTA["ffd_ragged"])
    host = W.generate(s)
    dw = PT.upload(s, host)
    sel, cnt, _, _ = PT.run_step(dw)
    rec = ops.selection_recall(dw.desc, dw.q, dw.K, torch.from_numpy(sel).cuda(), dw.ctx,
                               count=torch.from_numpy(cnt).cuda()).cpu().numpy()
    G = s.group
    for b in range(s.batch):
        for h in range(s.num_kv_heads):
            r = b * s.num_kv_heads + h
            q = O.to_f64(host.q[b, h * G:(h + 1) * G], s.dtype)
            ref = O.attention_mass_recall(q, O.to_f64(host.K[b, h], s.dtype), sel[r, :cnt[r]],
                                          int(host.ctx_len[b]), s.block, s.scale)
            np.testing.assert_allclose(rec[b, h * G:(h + 1) * G], ref, rtol=0, atol=RECALL_ATOL)
    # every page (no list): 1; an empty context: 1
    full = ops.selection_recall(dw.desc, dw.q, dw.K, None, dw.ctx).cpu().numpy()
    np.testing.assert_allclose(full, 1.0, rtol=0, atol=1e-6)
    s2 = W.spec("qwen7b", batch=2, ctx_len=[0, 300], capacity=320)
    dw2 = PT.upload(s2, W.generate(s2))
    idx = torch.full((s2.rows, 4), -1, dtype=torch.int32, device="cuda")
    rec2 = ops.selection_recall(dw2.desc, dw2.q, dw2.K, idx, dw2.ctx).cpu().numpy()
    assert np.all(rec2[0] == 1.0) and np.all(rec2[1] == 0.0)


def test_diagnostics_report_and_bound_beats_random_pages():
    from sparse_long_context_gb300 import diagnostics as DG
    s = W.spec("qwen7b", batch=2, ctx_len=8192, capacity=8192)
    dw = PT.upload(s, W.generate(s))
    q = DG.quest_quality(dw)
    assert 0.0 <= q["recall"]["min"] <= q["recall"]["mean"] <= 1.0
    assert np.isfinite(q["rel_l2_vs_dense"]["mean"])
    # a random list of the same size holds less of the mass than the bound's top k
    rng = np.random.default_rng(0)
    NP = 8192 // 16
    rnd = np.stack([np.sort(rng.choice(NP, size=s.k_pages, replace=False)) for _ in range(s.rows)]).astype(np.int32)
    rec_rand = ops.selection_recall(dw.desc, dw.q, dw.K, torch.from_numpy(rnd).cuda(), dw.ctx).cpu().numpy()
    assert q["recall"]["mean"] > rec_rand.mean() + 0.1
    sd = make(SMALL_DELTA["ffd_aligned"])
    d = DG.delta_vs_topk(PT.upload(sd, W.generate(sd)))
    assert 0.0 < d["kept_fraction"] <= 1.0 and 0.0 <= d["recall_top_delta"]["min"] <= 1.0
    for nr in (q["needle_recall"], d["needle_recall_top_delta"]):
        assert 0.0 <= nr["min"] <= nr["mean"] <= 1.0
