"""sls_select_pages_static: the page selection entry point that takes its
scratch from an array inside the library instead of a caller workspace,
for callers that cannot allocate device memory.  Its page lists must equal
those of sls_select_pages on the same inputs, call after call (the array
keeps the previous call's contents), and shapes too large for the array
must be refused before anything is launched.

This file is collected last on purpose: if it fails, a run that stops at
the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from sparse_long_context_gb300 import _lib as L
from sparse_long_context_gb300 import harness as H
from sparse_long_context_gb300 import ops
from sparse_long_context_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _select_static(dw, out):
    s = dw.spec
    L.call("sls_select_pages_static", ctypes.byref(dw.desc), ops._ptr(dw.q), ops._ptr(dw.kmin),
           ops._ptr(dw.kmax), ops._ptr(dw.ctx), s.k_pages, s.n_sink_pages, s.n_local_tokens,
           ops._ptr(out), ops._stream())
    return out


@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
def test_static_scratch_matches_workspace_version_on_consecutive_calls():
    L.load()
    cases = [W.spec("qwen1p5b", batch=4, ctx_len=[16384, 9000, 4099, 700]),
             W.spec("qwen7b", batch=2, ctx_len=[32768, 20000])]
    for s in cases:  # two calls in a row, different shapes, shared array
        dw = H.upload(s, W.generate(s))
        rows = s.rows
        ref = ops.select_pages(dw.desc, dw.q, dw.kmin, dw.kmax, dw.ctx, s.k_pages, s.n_sink_pages,
                               s.n_local_tokens)
        got = _select_static(dw, torch.full((rows, s.k_pages), -7, dtype=torch.int32, device="cuda"))
        torch.cuda.synchronize()
        assert torch.equal(got, ref)
        # the same inputs again: stale keys in the array must not matter
        again = _select_static(dw, torch.full((rows, s.k_pages), -7, dtype=torch.int32, device="cuda"))
        torch.cuda.synchronize()
        assert torch.equal(again, ref)


@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
def test_static_scratch_refuses_shapes_beyond_its_size():
    lib = L.load()
    # token-level selection over 131072-token rows needs 16 MiB of keys
    d = ops.make_desc(4, 64, 8, 64, 1, 131072, torch.bfloat16)
    assert lib.sls_select_pages_workspace_size(ctypes.byref(d)) > (4 << 20)
    bad = ctypes.c_void_p(0x1000)  # never dereferenced: the call is refused first
    st = lib.sls_select_pages_static(ctypes.byref(d), bad, bad, bad, bad, 4096, 4, 0, bad, None)
    assert st == L.SLS_EWORKSPACE
    assert "built-in scratch" in lib.sls_last_error().decode()
