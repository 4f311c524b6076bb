"""FFD 8-bit residuals and the refined attention ("Faster Than Flash",
Methodology 1 and eq. 4) through the C ABI against the fp64 oracle.

Codes and scales are bit-exact.  The oracle decides each residual integer
exactly; the kernel decides it in float32, so a residual may differ by one
only where the exact quotient lies within float32 rounding of a
half-integer (counted as a tie).
The refined step (top-delta selection, then attention whose complete blocks
are scored with k~ = thumbnail level + residual) is compared with the
oracle's refined attention on the same block sets, within the bf16 output
tolerance."""
import math

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


def _row_inputs(s, host, b, h):
    G = s.group
    q = O.to_f64(host.q[b, h * G:(h + 1) * G], s.dtype)
    K = O.to_f64(host.K[b, h], s.dtype)
    V = O.to_f64(host.V[b, h], s.dtype)
    sink = None if host.sink is None else host.sink[h * G:(h + 1) * G].astype(np.float64)
    return q, K, V, sink


def _check_residuals(s, host, codes, scales, res, ctx):
    codes, scales, res = codes.cpu().numpy(), scales.float().cpu().numpy(), res.cpu().numpy()
    for b in range(s.batch):
        for h in range(s.num_kv_heads):
            n = int(ctx[b])
            oc, osc, ores = O.residuals_row(O.to_f64(host.K[b, h], s.dtype), n, s.block)
            nfull = n // s.block
            np.testing.assert_array_equal(codes[b, h, :nfull * s.block], O.pack_codes(oc))
            np.testing.assert_array_equal(scales[b, h, :nfull], osc)
            PT.check_residuals(res[b, h], O.to_f64(host.K[b, h], s.dtype), n, s.block)


@pytest.mark.parametrize("ctx", [[64 * 9 + 5, 64 * 3], [64 * 40]])
def test_residuals_are_bit_exact(ctx):
    s = W.spec("ffd", ctx_len=ctx, capacity=64 * 40)
    host = W.generate(s)
    dw = PT.upload(s, host)
    codes, scales, res = ops.thumb_residual_build(dw.desc, dw.K, dw.ctx, s.block)
    torch.cuda.synchronize()
    _check_residuals(s, host, codes, scales, res, host.ctx_len)
    # the plain thumbnail call writes the same codes and scales
    c2, s2 = ops.thumb_build(dw.desc, dw.K, dw.ctx, s.block)
    assert torch.equal(c2, codes) and torch.equal(s2, scales)


def test_residual_update_completes_blocks():
    s = W.spec("ffd", batch=2, ctx_len=[64 * 5, 64 * 7], capacity=64 * 8)
    host = W.generate(s)
    dw = PT.upload(s, host)
    start = torch.tensor([64 * 3 + 10, 64 * 6 + 60], dtype=torch.int32, device="cuda")
    codes, scales, res = ops.thumb_residual_build(dw.desc, dw.K, start, 64)
    cur = start.cpu().numpy().copy()
    end = host.ctx_len
    while np.any(cur < end):
        pos = np.where(cur < end, cur, -1).astype(np.int32)
        ops.thumb_residual_update(dw.desc, dw.K, torch.from_numpy(pos).cuda(), 64, codes, scales, res)
        cur = np.minimum(cur + 1, end)
    torch.cuda.synchronize()
    _check_residuals(s, host, codes, scales, res, end)


SMALL = {
    "ffd_ragged": dict(ctx_len=[65536 + 100, 20000], capacity=65536 + 128),
    "ffd_aligned": dict(batch=1, ctx_len=8192),
    "ffd_short": dict(batch=3, ctx_len=[64, 100, 1], capacity=256),
}


def _refined_step(s, host, no_tma=False):
    dw = PT.upload(s, host, no_tma=no_tma)
    codes, scales, res = ops.thumb_residual_build(dw.desc, dw.K, dw.ctx, s.block)
    step = ops.DeltaDecode(dw.desc, s.block, s.delta, refined=True)
    out, lse = step(dw.q, dw.K, dw.V, codes, scales, dw.ctx, dw.sink, res=res)
    ops.pipeline_check()
    return dw, (codes, scales, res), step, out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy()


def _refined_oracle(s, host, b, h, blocks):
    q, K, V, sink = _row_inputs(s, host, b, h)
    return O.refined_attention_row(q, K, V, blocks, int(host.ctx_len[b]), s.block, s.scale, sink)


# the tensor-map fed refined attend (the default at D = 128) and the register-fed one
@pytest.mark.parametrize("no_tma", [False, True])
@pytest.mark.parametrize("key", list(SMALL))
def test_refined_step_matches_oracle(key, no_tma):
    s = W.spec("ffd", **SMALL[key])
    host = W.generate(s)
    ops.get_stats(reset=True)
    dw, (codes, scales, res), step, out, lse = _refined_step(s, host, no_tma)
    st = ops.get_stats(reset=True)
    assert st["attend_refined"] == 1 and st["attend_refined_tma"] == (0 if no_tma else 1), st
    sel, cnt = step.block_idx.cpu().numpy(), step.count.cpu().numpy()
    G = s.group
    ties = 0
    sets = []
    for b in range(s.batch):
        for h in range(s.num_kv_heads):
            r = b * s.num_kv_heads + h
            orc = PT.oracle_row(s, host, b, h)
            sets.append(orc.pages)
            t = PT.check_delta_list(int(cnt[r]), sel[r], orc, s.delta)
            ties += t
            if t:
                continue
            o_ref, lse_ref = _refined_oracle(s, host, b, h, orc.pages)
            PT.assert_close(s, out[b, h * G:(h + 1) * G], o_ref, f"refined row {(b, h)}")
            fin = np.isfinite(lse_ref)
            np.testing.assert_allclose(lse[b, h * G:(h + 1) * G][fin], lse_ref[fin], rtol=1e-4, atol=1e-4)
    # the attend alone on the oracle's own block sets
    width = max(1, max(len(p) for p in sets))
    idx = np.full((s.rows, width), -1, dtype=np.int32)
    count = np.array([len(p) for p in sets], dtype=np.int32)
    for r, p in enumerate(sets):
        idx[r, :len(p)] = p
    o2, _ = ops.refined_decode_attend_combine(dw.desc, dw.q, dw.K, dw.V, codes, scales, res,
                                              torch.from_numpy(idx).cuda(), torch.from_numpy(count).cuda(),
                                              dw.ctx, sink=dw.sink)
    o2 = o2.float().cpu().numpy().astype(np.float64)
    for b in range(s.batch):
        for h in range(s.num_kv_heads):
            o_ref, _ = _refined_oracle(s, host, b, h, sets[b * s.num_kv_heads + h])
            PT.assert_close(s, o2[b, h * G:(h + 1) * G], o_ref, f"refined attend on oracle set {(b, h)}")
    print(f"{key}: boundary ties {ties}")


@pytest.mark.parametrize("refined", [False, True])
def test_stream_k_with_more_rows_than_ctas(refined):
    """192 rows of 7-8 blocks against one CTA per SM: most CTA ranges hold
    several whole rows and start or end inside others, and the row-start
    cost the partition charges outweighs the real entries (every partition
    boundary case at once).  Lists: empty, one block, every block, or a
    random subset; outputs against the oracle's attention on the same sets
    (refined keys: the oracle's refined attention)."""
    s = W.spec("ffd", batch=24, ctx_len=[64 * 7 + 5 + 13 * (b % 5) for b in range(24)], capacity=64 * 8)
    assert s.rows > 152
    host = W.generate(s)
    dw = PT.upload(s, host)
    codes = scales = res = None
    if refined:
        codes, scales, res = ops.thumb_residual_build(dw.desc, dw.K, dw.ctx, s.block)
    rng = np.random.default_rng(11)
    width = s.capacity // s.block
    idx = np.full((s.rows, width), -1, dtype=np.int32)
    count = np.zeros(s.rows, dtype=np.int32)
    lists = []
    for r in range(s.rows):
        nb = -(-int(host.ctx_len[r // s.num_kv_heads]) // s.block)
        kind = r % 5
        if kind == 0:
            blocks = np.zeros(0, dtype=np.int64)
        elif kind == 1:
            blocks = np.array([nb - 1])
        elif kind == 2:
            blocks = np.arange(nb)
        else:
            blocks = np.sort(rng.choice(nb, size=int(rng.integers(1, nb + 1)), replace=False))
        lists.append(blocks)
        idx[r, :len(blocks)] = blocks
        count[r] = len(blocks)
    ops.get_stats(reset=True)
    out, lse = ops.refined_decode_attend_combine(dw.desc, dw.q, dw.K, dw.V, codes, scales, res,
                                                 torch.from_numpy(idx).cuda(), torch.from_numpy(count).cuda(),
                                                 dw.ctx, sink=dw.sink)
    ops.pipeline_check()
    st = ops.get_stats(reset=True)
    assert st["attend_refined_tma" if refined else "attend_stream_k_tma"] == 1, st
    out = out.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy()
    G = s.group
    for b in range(s.batch):
        for h in range(s.num_kv_heads):
            r = b * s.num_kv_heads + h
            if refined:
                o_ref, l_ref = _refined_oracle(s, host, b, h, lists[r])
            else:
                q, K, V, sink = _row_inputs(s, host, b, h)
                o_ref, l_ref = O.sparse_attention_row(q, K, V, lists[r], int(host.ctx_len[b]), s.page_size,
                                                      s.scale, sink)
            PT.assert_close(s, out[b, h * G:(h + 1) * G], o_ref, f"row {r}")
            fin = np.isfinite(l_ref)
            np.testing.assert_allclose(lse[b, h * G:(h + 1) * G][fin], l_ref[fin], rtol=1e-4, atol=1e-4)


def test_refined_scores_differ_from_exact_ones():
    """The refined path really scores with k~: against the exact-key step on
    the same selection the outputs differ (slightly), and both stay within
    tolerance of their own oracle; the path counters name the kernels."""
    s = W.spec("ffd", **SMALL["ffd_aligned"])
    host = W.generate(s)
    ops.get_stats(reset=True)
    dw, _, step, out_ref, _ = _refined_step(s, host)
    exact = ops.DeltaDecode(dw.desc, s.block, s.delta)
    out_ex, _ = exact(dw.q, dw.K, dw.V, dw.codes, dw.scales, dw.ctx, dw.sink)
    st = ops.get_stats(reset=True)
    assert st["attend_refined"] == 1 and st["attend_stream_k"] == 1, st
    assert st["attend_refined_tma"] == 1 and st["attend_stream_k_tma"] == 1, st
    assert st["select_delta_tensor_cores"] == 2 and st["select_delta_cuda_cores"] == 0, st
    out_ex = out_ex.float().cpu().numpy().astype(np.float64)
    assert np.abs(out_ref - out_ex).max() > 0
    q, K, V, sink = _row_inputs(s, host, 0, 0)
    blocks = step.block_idx.cpu().numpy()[0, :int(step.count.cpu().numpy()[0])]
    o_ex, _ = O.sparse_attention_row(q, K, V, blocks, int(host.ctx_len[0]), s.block, s.scale, sink)
    o_rf, _ = O.refined_attention_row(q, K, V, blocks, int(host.ctx_len[0]), s.block, s.scale, sink)
    assert np.abs(o_ex - o_rf).max() > 0


def test_refined_full_size_sampled_rows():
    """The full-size top-delta workload (2 sequences of 256k tokens), in the
    launch configuration of the step, on two sampled rows."""
    s = W.spec("ffd")
    host = W.generate(s)
    _, _, step, out, lse = _refined_step(s, host)
    sel, cnt = step.block_idx.cpu().numpy(), step.count.cpu().numpy()
    G = s.group
    for b, h in [(0, 0), (s.batch - 1, s.num_kv_heads - 1)]:
        r = b * s.num_kv_heads + h
        orc = PT.oracle_row(s, host, b, h)
        if PT.check_delta_list(int(cnt[r]), sel[r], orc, s.delta):
            continue
        o_ref, _ = _refined_oracle(s, host, b, h, orc.pages)
        PT.assert_close(s, out[b, h * G:(h + 1) * G], o_ref, f"full-size refined row {(b, h)}")
    assert math.isfinite(float(np.abs(out).max()))


@pytest.mark.parametrize("ctx", [[5000, 3000, 10], [100, 37, 16]])
def test_balanced_attend_uneven_lists_and_sink(ctx):
    """The stream-K attend (bf16 keys) on lists of very different lengths:
    empty rows, one page, every page, padded entries, a sink, against the
    oracle's attention over the same pages; with few entries in all (the
    second case) most CTAs get an empty range."""
    s = W.spec("qwen7b", batch=3, ctx_len=ctx, capacity=5008)
    host = W.generate(s)
    dw = PT.upload(s, host)
    rng = np.random.default_rng(7)
    npg = [-(-int(n) // s.page_size) for n in host.ctx_len]
    width = max(npg) + 3
    idx = np.full((s.rows, width), -1, dtype=np.int32)
    count = np.zeros(s.rows, dtype=np.int32)
    lists = []
    for r in range(s.rows):
        n = npg[r // s.num_kv_heads]
        kind = r % 4
        if kind == 0:
            pages = np.zeros(0, dtype=np.int64)
        elif kind == 1:
            pages = np.array([n - 1])
        elif kind == 2:
            pages = np.arange(n)
        else:
            pages = np.sort(rng.choice(n, size=min(n, 37), replace=False))
        lists.append(pages)
        idx[r, :len(pages)] = pages
        count[r] = len(pages) + (2 if kind == 3 else 0)  # two -1 entries counted in: skipped
    sink = torch.from_numpy(rng.standard_normal(s.num_q_heads).astype(np.float32)).cuda()
    out, lse = ops.refined_decode_attend_combine(dw.desc, dw.q, dw.K, dw.V, None, None, None,
                                                 torch.from_numpy(idx).cuda(), torch.from_numpy(count).cuda(),
                                                 dw.ctx, sink=sink)
    ops.pipeline_check()
    out = out.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy()
    G = s.group
    for b in range(s.batch):
        for h in range(s.num_kv_heads):
            r = b * s.num_kv_heads + h
            q = O.to_f64(host.q[b, h * G:(h + 1) * G], s.dtype)
            K = O.to_f64(host.K[b, h], s.dtype)
            V = O.to_f64(host.V[b, h], s.dtype)
            sk = sink.cpu().numpy()[h * G:(h + 1) * G].astype(np.float64)
            o_ref, l_ref = O.sparse_attention_row(q, K, V, lists[r], int(host.ctx_len[b]), s.page_size,
                                                  s.scale, sk)
            PT.assert_close(s, out[b, h * G:(h + 1) * G], o_ref, f"row {r}")
            np.testing.assert_allclose(lse[b, h * G:(h + 1) * G], l_ref, rtol=1e-4, atol=1e-4)


@pytest.mark.parametrize("D,Hq,Hkv,sink", [(64, 16, 2, True), (128, 4, 4, False), (64, 3, 1, True)])
def test_refined_other_head_shapes(D, Hq, Hkv, sink):
    """The refined step at D = 64 and at group sizes 8, 1 and 3 (padded head
    rows), with and without a sink, against the oracle's refined attention."""
    s = W.spec("ffd", batch=2, ctx_len=[64 * 37 + 5, 64 * 12], capacity=64 * 38)
    s.head_dim, s.num_q_heads, s.num_kv_heads, s.has_sink = D, Hq, Hkv, sink
    host = W.generate(s)
    dw, _, step, out, lse = _refined_step(s, host)
    sel, cnt = step.block_idx.cpu().numpy(), step.count.cpu().numpy()
    G = s.group
    for b in range(s.batch):
        for h in range(s.num_kv_heads):
            r = b * s.num_kv_heads + h
            orc = PT.oracle_row(s, host, b, h)
            if PT.check_delta_list(int(cnt[r]), sel[r], orc, s.delta):
                continue
            o_ref, lse_ref = _refined_oracle(s, host, b, h, orc.pages)
            PT.assert_close(s, out[b, h * G:(h + 1) * G], o_ref, f"row {(b, h)}")
            np.testing.assert_allclose(lse[b, h * G:(h + 1) * G], lse_ref, rtol=1e-4, atol=1e-4)


@pytest.mark.parametrize("block", [16, 32, 128])
def test_refined_other_block_sizes(block):
    """The refined step with thumbnail blocks of 16, 32 and 128 tokens (one,
    two and eight 16-token groups per block: the attend scores a block's
    groups in one warp and reuses the block's q s parts) against the oracle's
    refined attention."""
    s = W.spec("ffd", batch=2, ctx_len=[block * 45 + 7, block * 20], capacity=block * 46)
    s.block = s.page_size = block
    host = W.generate(s)
    dw, _, step, out, lse = _refined_step(s, host)
    sel, cnt = step.block_idx.cpu().numpy(), step.count.cpu().numpy()
    G = s.group
    checked = 0
    for b in range(s.batch):
        for h in range(s.num_kv_heads):
            r = b * s.num_kv_heads + h
            orc = PT.oracle_row(s, host, b, h)
            if PT.check_delta_list(int(cnt[r]), sel[r], orc, s.delta):
                continue
            o_ref, lse_ref = _refined_oracle(s, host, b, h, orc.pages)
            PT.assert_close(s, out[b, h * G:(h + 1) * G], o_ref, f"block {block} row {(b, h)}")
            np.testing.assert_allclose(lse[b, h * G:(h + 1) * G], lse_ref, rtol=1e-4, atol=1e-4)
            checked += 1
    assert checked >= s.rows // 2
