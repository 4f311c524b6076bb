"""The device-resident decode loop: append + select + attend + combine per
token, eager and replayed from a CUDA graph, against the fp64 oracle.

Each case starts L tokens short of the workload's context with the cache
past that point cleared, then decodes the remaining tokens one at a time
feeding the workload's own keys and values as the new tokens.  After the
last step the cache, the selector's summaries and ctx_len must equal what
the oracle builds on the full context (bit-exact), and the last step's
output must match the oracle's decode of the full context."""
import numpy as np
import pytest
import torch

from oracle import sls_oracle as O
from sparse_long_context_gb300 import harness as H
from sparse_long_context_gb300 import ops
from sparse_long_context_gb300 import workloads as W

from tests import parity as PT
from tests.test_gpu_parity import check_all_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


CASES = {
    # 16-token pages, bf16: the one-launch step; L crosses several pages
    "qwen7b": (dict(name="qwen7b", batch=2, ctx_len=[2300, 517], capacity=2304), 40),
    # page size 1 (the key cache is its own metadata): select + attend
    "gptoss": (dict(name="gptoss", batch=2, ctx_len=[4500, 1203], capacity=4608), 20),
    # top-delta: thumbnails of the blocks the new tokens complete
    "ffd": (dict(name="ffd", batch=2, ctx_len=[64 * 5 + 3, 64 * 7], capacity=64 * 8), 70),
}


def _spec(key):
    kw = dict(CASES[key][0])
    return W.spec(kw.pop("name"), **kw), CASES[key][1]


def _rewind(dw, n0):
    """Clears the cache past n0 and rebuilds the summaries at n0."""
    s = dw.spec
    for b in range(s.batch):
        dw.K[b, :, int(n0[b]):] = 0
        dw.V[b, :, int(n0[b]):] = 0
    ctx0 = torch.from_numpy(n0.astype(np.int32)).cuda()
    dw.ctx.copy_(ctx0)
    if s.selector == "quest":
        if s.page_size > 1:
            ops.pagemeta_build(dw.desc, dw.K, dw.ctx, dw.kmin, dw.kmax)
    else:
        ops.thumb_build(dw.desc, dw.K, dw.ctx, s.block, dw.codes, dw.scales)
    torch.cuda.synchronize()


def _token(host, s, t):
    """New key/value of step t: the workload's own token at position t[b]."""
    kb = np.stack([host.K[b, :, int(t[b])] for b in range(s.batch)])
    vb = np.stack([host.V[b, :, int(t[b])] for b in range(s.batch)])
    return PT.to_device(kb, s.dtype), PT.to_device(vb, s.dtype)


def _check_state(dw, host):
    s = dw.spec
    np.testing.assert_array_equal(dw.ctx.cpu().numpy(), host.ctx_len)
    K = dw.K.cpu()
    V = dw.V.cpu()
    Kh, Vh = PT.to_device(host.K, s.dtype, "cpu"), PT.to_device(host.V, s.dtype, "cpu")
    for b in range(s.batch):
        n = int(host.ctx_len[b])
        assert torch.equal(K[b, :, :n], Kh[b, :, :n]), f"key cache of sequence {b}"
        assert torch.equal(V[b, :, :n], Vh[b, :, :n]), f"value cache of sequence {b}"
    if s.selector == "quest" and s.page_size > 1:
        kmin, kmax = dw.kmin.float().cpu().numpy(), dw.kmax.float().cpu().numpy()
        for b in range(s.batch):
            for h in range(s.num_kv_heads):
                omin, omax = O.page_minmax(O.to_f64(host.K[b, h], s.dtype), int(host.ctx_len[b]), s.page_size)
                np.testing.assert_array_equal(kmin[b, h, :len(omin)], omin)
                np.testing.assert_array_equal(kmax[b, h, :len(omax)], omax)
    if s.selector != "quest":
        codes, scales = dw.codes.cpu().numpy(), dw.scales.float().cpu().numpy()
        for b in range(s.batch):
            for h in range(s.num_kv_heads):
                n = int(host.ctx_len[b])
                oc, osc = O.thumbnails_row(O.to_f64(host.K[b, h], s.dtype), n, s.block)
                nfull = n // s.block
                np.testing.assert_array_equal(codes[b, h, :nfull * s.block], O.pack_codes(oc))
                np.testing.assert_array_equal(scales[b, h, :nfull], osc)


def _selection(loop):
    st = loop.step
    if isinstance(st, ops.QuestDecode):
        return st.page_idx.cpu().numpy(), None
    return st.block_idx.cpu().numpy(), st.count.cpu().numpy()


def _host_out(out, lse):
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("key", list(CASES))
def test_eager_decode_loop_matches_oracle(key):
    s, L = _spec(key)
    host = W.generate(s)
    dw = PT.upload(s, host)
    n0 = host.ctx_len - L
    _rewind(dw, n0)
    loop = H.DecodeLoop(dw)
    for i in range(L):
        k_new, v_new = _token(host, s, n0 + i)
        loop.k_new.copy_(k_new)
        loop.v_new.copy_(v_new)
        out, lse = loop.run_once()
        np.testing.assert_array_equal(loop.pos.cpu().numpy(), n0 + i)
    ops.pipeline_check()
    _check_state(dw, host)
    sel, cnt = _selection(loop)
    check_all_rows(s, host, sel, cnt, *_host_out(out, lse), dw)


@pytest.mark.parametrize("key", list(CASES))
def test_graph_replays_equal_eager_steps(key):
    s, L = _spec(key)
    host = W.generate(s)
    n0 = host.ctx_len - L
    # eager reference run
    dw = PT.upload(s, host)
    _rewind(dw, n0)
    loop = H.DecodeLoop(dw)
    eager = []
    for i in range(L):
        k_new, v_new = _token(host, s, n0 + i)
        loop.k_new.copy_(k_new)
        loop.v_new.copy_(v_new)
        out, lse = loop.run_once()
        eager.append((out.clone(), lse.clone()))
    ops.pipeline_check()
    # the same steps as graph replays
    dg = PT.upload(s, host)
    _rewind(dg, n0)
    gl = H.DecodeLoop(dg)
    gl.capture()
    for i in range(L):
        k_new, v_new = _token(host, s, n0 + i)
        gl.k_new.copy_(k_new)
        gl.v_new.copy_(v_new)
        out, lse = gl.replay()
        assert torch.equal(out, eager[i][0]), f"output of step {i}"
        assert torch.equal(lse, eager[i][1]), f"lse of step {i}"
    ops.pipeline_check()
    _check_state(dg, host)


def test_refined_decode_loop_matches_oracle():
    """The top-delta loop with 8-bit residuals kept current (f2 inside f3):
    after the appends the codes, scales and residuals equal the oracle's on
    the full context, graph replays equal eager steps, and the last step's
    output matches the oracle's refined attention."""
    s, L = _spec("ffd")
    host = W.generate(s)
    n0 = host.ctx_len - L
    outs = []
    for graph in (False, True):
        dw = PT.upload(s, host)
        _rewind(dw, n0)
        _, _, res = ops.thumb_residual_build(dw.desc, dw.K, dw.ctx, s.block, dw.codes, dw.scales)
        loop = H.DecodeLoop(dw, refined=True, res=res)
        if graph:
            loop.capture()
        for i in range(L):
            k_new, v_new = _token(host, s, n0 + i)
            loop.k_new.copy_(k_new)
            loop.v_new.copy_(v_new)
            out, lse = loop.replay() if graph else loop.run_once()
            outs.append((graph, i, out.clone(), lse.clone()))
        ops.pipeline_check()
        _check_state(dw, host)
        rr = res.cpu().numpy()
        for b in range(s.batch):
            for h in range(s.num_kv_heads):
                n = int(host.ctx_len[b])
                PT.check_residuals(rr[b, h], O.to_f64(host.K[b, h], s.dtype), n, s.block)
    eager = {i: (o, l) for g, i, o, l in outs if not g}
    for g, i, o, l in outs:
        if g:
            assert torch.equal(o, eager[i][0]) and torch.equal(l, eager[i][1]), f"step {i}"
    sel, cnt = _selection(loop)
    out = outs[-1][2].float().cpu().numpy().astype(np.float64)
    G = s.group
    for b in range(s.batch):
        for h in range(s.num_kv_heads):
            r = b * s.num_kv_heads + h
            orc = PT.oracle_row(s, host, b, h)
            if PT.check_delta_list(int(cnt[r]), sel[r], orc, s.delta):
                continue
            q = O.to_f64(host.q[b, h * G:(h + 1) * G], s.dtype)
            K = O.to_f64(host.K[b, h], s.dtype)
            V = O.to_f64(host.V[b, h], s.dtype)
            o_ref, _ = O.refined_attention_row(q, K, V, orc.pages, int(host.ctx_len[b]), s.block, s.scale)
            PT.assert_close(s, out[b, h * G:(h + 1) * G], o_ref, f"refined loop row {(b, h)}")


def test_append_at_capacity_changes_nothing():
    s = W.spec("qwen7b", batch=2, ctx_len=[2304, 2288], capacity=2304)
    host = W.generate(s)
    dw = PT.upload(s, host)
    loop = H.DecodeLoop(dw)
    K0, V0 = dw.K.clone(), dw.V.clone()
    kmin0, kmax0 = dw.kmin.clone(), dw.kmax.clone()
    loop.k_new.fill_(3.0)
    loop.v_new.fill_(-3.0)
    ops.decode_append(dw.desc, loop.k_new, loop.v_new, dw.K, dw.V, dw.ctx, dw.kmin, dw.kmax, pos_out=loop.pos)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(loop.pos.cpu().numpy(), [-1, 2288])
    np.testing.assert_array_equal(dw.ctx.cpu().numpy(), [2304, 2289])
    assert torch.equal(dw.K[0], K0[0]) and torch.equal(dw.V[0], V0[0])
    assert torch.equal(dw.kmin[0], kmin0[0]) and torch.equal(dw.kmax[0], kmax0[0])
    # sequence 1 took the token at 2288, the first of page 143: min = max = the key
    assert torch.all(dw.K[1, :, 2288] == 3.0) and torch.all(dw.V[1, :, 2288] == -3.0)
    assert torch.all(dw.kmin[1, :, 143] == 3.0) and torch.all(dw.kmax[1, :, 143] == 3.0)
    assert torch.equal(dw.K[1, :, :2288], K0[1, :, :2288])
