"""Device status through the C ABI: bad page-list entries and bounded waits
that give up are counted on the device and reported by sls_pipeline_check.

Both failures are made without a GPU fault.  A bad page id is an integer in
the caller's list that the kernels check before any load and skip.  A wait
that gives up is planted with the test hook SLS_FLAG_TEST_WAIT_TIMEOUT: the
first CTA announces copy bytes on one pipeline stage and requests none, so
that stage's waits run out of polls; no copy is in flight for it.  After each
failure the context stays usable, which the next, clean call shows."""
import numpy as np
import pytest
import torch

from oracle import sls_oracle as O
from sparse_long_context_gb300 import _lib as L
from sparse_long_context_gb300 import ops
from sparse_long_context_gb300 import workloads as W

from tests import parity as PT

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _check_status():
    """Status code of sls_pipeline_check (0 when clean)."""
    try:
        ops.pipeline_check()
        return L.SLS_OK
    except L.SlsError as e:
        return e.code


def _workload(**kw):
    s = W.spec("qwen1p5b", batch=2, ctx_len=[1000, 1531], **kw)
    return s, W.generate(s)


def _oracle_lists(s, host):
    width = s.k_pages
    idx = np.full((s.rows, width), -1, dtype=np.int32)
    for r in range(s.rows):
        b, h = divmod(r, s.num_kv_heads)
        p = PT.oracle_row(s, host, b, h).pages
        idx[r, :len(p)] = p
    return idx


def _plant_bad(idx, npool):
    """Bad entries in three rows: just past the pool, far past it, and a
    negative id other than the -1 padding.  Returns (bad list, the same list
    with those entries as -1, the number planted)."""
    bad = idx.copy()
    spots = [(0, 3, npool), (1, 5, 1 << 30), (2, 0, -7), (3, 7, npool + 1)]
    for r, e, v in spots:
        bad[r % idx.shape[0], e] = v
    clean = bad.copy()
    clean[(clean < -1) | (clean >= npool)] = -1
    return bad, clean, len(spots)


@pytest.mark.parametrize("path", ["tma", "registers", "cuda_cores"])
def test_bad_page_ids_are_skipped_and_reported(path):
    s, host = _workload()
    dw = PT.upload(s, host, cuda_cores=path == "cuda_cores", no_tma=path == "registers")
    npool = s.capacity // s.page_size
    bad, clean, _ = _plant_bad(_oracle_lists(s, host), npool)
    assert _check_status() == L.SLS_OK
    ops.get_stats(reset=True)
    outs = {}
    for name, lst in (("bad", bad), ("clean", clean)):
        idx = torch.from_numpy(lst).cuda()
        out, lse = ops.sparse_decode_attend_combine(dw.desc, dw.q, dw.K, dw.V, idx, dw.ctx, 4, sink=dw.sink)
        outs[name] = (out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy())
        code = _check_status()
        assert code == (L.SLS_EDEVICE if name == "bad" else L.SLS_OK), (name, code, L.load().sls_last_error())
    stats = ops.get_stats(reset=True)
    want = {"tma": "attend_tma", "registers": "attend_mma", "cuda_cores": "attend_cuda_cores"}[path]
    assert stats[want] >= 2, stats
    # a bad entry is skipped: the output is the clean list's, which matches the oracle
    np.testing.assert_allclose(outs["bad"][0], outs["clean"][0], rtol=1e-5, atol=1e-6)
    for r in range(s.rows):
        b, h = divmod(r, s.num_kv_heads)
        G, n = s.group, int(host.ctx_len[b])
        q = O.to_f64(host.q[b, h * G:(h + 1) * G], s.dtype)
        K, V = O.to_f64(host.K[b, h], s.dtype), O.to_f64(host.V[b, h], s.dtype)
        ref, _ = O.sparse_attention_row(q, K, V, clean[r], n, s.page_size, s.scale)
        PT.assert_close(s, outs["bad"][0][b, h * G:(h + 1) * G], ref, f"row {r}")


@pytest.mark.parametrize("refined", [False, True])
def test_bad_block_ids_in_the_stream_k_attend_and_recall_are_reported(refined):
    s = W.spec("ffd", batch=1, ctx_len=64 * 40 + 9, capacity=64 * 48)
    host = W.generate(s)
    dw = PT.upload(s, host)
    codes = scales = res = None
    if refined:  # the refined (2-bit + 8-bit) keys on the tensor-map fed kernel
        codes, scales, res = ops.thumb_residual_build(dw.desc, dw.K, dw.ctx, s.block)
    npool = s.capacity // s.block
    lists = np.full((s.rows, npool), -1, dtype=np.int32)
    count = np.zeros(s.rows, dtype=np.int32)
    for r in range(s.rows):
        p = np.arange(0, 41, 3)
        lists[r, :len(p)] = p
        count[r] = len(p)
    bad = lists.copy()
    bad[1, 2] = npool + 5
    bad[4, 0] = -3
    clean = bad.copy()
    clean[(clean < -1) | (clean >= npool)] = -1
    cnt = torch.from_numpy(count).cuda()
    assert _check_status() == L.SLS_OK
    outs = {}
    for name, lst in (("bad", bad), ("clean", clean)):
        idx = torch.from_numpy(lst).cuda()
        out, _ = ops.refined_decode_attend_combine(dw.desc, dw.q, dw.K, dw.V, codes, scales, res, idx, cnt, dw.ctx)
        outs[name] = out.float().cpu().numpy()
        assert _check_status() == (L.SLS_EDEVICE if name == "bad" else L.SLS_OK), name
        rec = ops.selection_recall(dw.desc, dw.q, dw.K, idx, dw.ctx, count=cnt)
        torch.cuda.synchronize()
        assert _check_status() == (L.SLS_EDEVICE if name == "bad" else L.SLS_OK), ("recall", name)
        outs[name + "_recall"] = rec.cpu().numpy()
    np.testing.assert_allclose(outs["bad"], outs["clean"], rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(outs["bad_recall"], outs["clean_recall"], rtol=1e-6)


@pytest.mark.parametrize("entry", ["attend_combine", "quest_step"])
def test_a_wait_that_gives_up_is_reported(entry):
    s = W.spec("qwen1p5b", batch=2, ctx_len=[4096, 3001])
    host = W.generate(s)
    dw = PT.upload(s, host)
    G = s.group
    idx = torch.from_numpy(_oracle_lists(s, host)).cuda()
    hooked = ops.make_desc(s.batch, s.num_q_heads, s.num_kv_heads, s.head_dim, s.page_size, s.capacity,
                           dw.K.dtype, test_wait_timeout=True)

    def run(desc):
        if entry == "attend_combine":
            out, lse = ops.sparse_decode_attend_combine(desc, dw.q, dw.K, dw.V, idx, dw.ctx, 4)
        else:
            out, lse = ops.quest_decode_step(desc, dw.q, dw.K, dw.V, dw.kmin, dw.kmax, dw.ctx, s.k_pages,
                                             s.n_sink_pages, s.n_local_tokens)
        return out.float().cpu().numpy(), lse.cpu().numpy()

    assert _check_status() == L.SLS_OK
    ops.get_stats(reset=True)
    ok_out, ok_lse = run(dw.desc)
    assert _check_status() == L.SLS_OK
    t_out, t_lse = run(hooked)
    code = _check_status()
    assert code == L.SLS_ETIMEOUT, (code, L.load().sls_last_error())
    stats = ops.get_stats(reset=True)
    assert stats["attend_tma" if entry == "attend_combine" else "quest_step_one_launch"] >= 2, stats
    # the first row (sequence 0, KV head 0) is NaN, every other row is unchanged
    assert np.isnan(t_out[0, :G]).all() and np.isnan(t_lse[0, :G]).all()
    np.testing.assert_array_equal(t_out[0, G:], ok_out[0, G:])
    np.testing.assert_array_equal(t_out[1:], ok_out[1:])
    np.testing.assert_array_equal(t_lse[1:], ok_lse[1:])
    # the context stays usable: the next clean call is correct and reports nothing
    again, _ = run(dw.desc)
    assert _check_status() == L.SLS_OK
    np.testing.assert_array_equal(again, ok_out)


@pytest.mark.parametrize("refined", [False, True])
def test_a_stream_k_wait_that_gives_up_is_reported(refined):
    """The tensor-map fed stream-K attends (bf16 keys, or the refined keys,
    over block lists): under the hook the first CTA's first stage never
    fills.  Every row keeps all 41 blocks (328 entries, more than one per
    CTA), so the first CTA's range holds entries of row 0 only: row 0 becomes
    NaN, every other row is unchanged, and the next clean call is correct
    again."""
    s = W.spec("ffd", batch=1, ctx_len=64 * 40 + 9, capacity=64 * 48)
    host = W.generate(s)
    dw = PT.upload(s, host)
    codes = scales = res = None
    if refined:
        codes, scales, res = ops.thumb_residual_build(dw.desc, dw.K, dw.ctx, s.block)
    npool = s.capacity // s.block
    lists = np.full((s.rows, npool), -1, dtype=np.int32)
    count = np.zeros(s.rows, dtype=np.int32)
    for r in range(s.rows):
        p = np.arange(0, 41)
        lists[r, :len(p)] = p
        count[r] = len(p)
    idx, cnt = torch.from_numpy(lists).cuda(), torch.from_numpy(count).cuda()
    hooked = ops.make_desc(s.batch, s.num_q_heads, s.num_kv_heads, s.head_dim, s.page_size, s.capacity,
                           dw.K.dtype, test_wait_timeout=True)

    def run(desc):
        out, lse = ops.refined_decode_attend_combine(desc, dw.q, dw.K, dw.V, codes, scales, res, idx, cnt, dw.ctx)
        return out.float().cpu().numpy(), lse.cpu().numpy()

    G = s.group
    assert _check_status() == L.SLS_OK
    ops.get_stats(reset=True)
    ok_out, ok_lse = run(dw.desc)
    assert _check_status() == L.SLS_OK
    t_out, t_lse = run(hooked)
    code = _check_status()
    assert code == L.SLS_ETIMEOUT, (code, L.load().sls_last_error())
    assert ops.get_stats(reset=True)["attend_refined_tma" if refined else "attend_stream_k_tma"] >= 2
    assert np.isnan(t_out[0, :G]).all() and np.isnan(t_lse[0, :G]).all()
    np.testing.assert_array_equal(t_out[0, G:], ok_out[0, G:])
    np.testing.assert_array_equal(t_lse[0, G:], ok_lse[0, G:])
    again, _ = run(dw.desc)
    assert _check_status() == L.SLS_OK
    np.testing.assert_array_equal(again, ok_out)
