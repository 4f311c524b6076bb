"""Host-side checks of the C ABI: the library loads without a GPU, exports
every symbol include/sls.h declares, and rejects bad arguments before it
launches anything.  Every call here fails validation, so no kernel runs."""
import ctypes
import os
import re

import pytest

from sparse_long_context_gb300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sls.h")
BAD = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:sls_status|size_t|const char\*|int32_t)\s+(sls_\w+)\(",
                                 text, re.M)))


def desc(**kw):
    d = dict(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
             capacity=1024, dtype=L.SLS_DTYPE_BF16, flags=0, scale=0.0)
    d.update(kw)
    return L.AttnDesc(**d)


def test_exports_every_declared_symbol(lib):
    syms = declared_symbols()
    assert len(syms) >= 10
    for s in syms:
        assert hasattr(lib, s), s
    assert set(syms) == set(L.SIGNATURES)
    assert lib.sls_version() == 10000


def err(lib):
    return lib.sls_last_error().decode()


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=96), L.SLS_EUNSUPPORTED),
    (dict(num_q_heads=18, num_kv_heads=2), L.SLS_EUNSUPPORTED),   # G = 9
    (dict(num_q_heads=7, num_kv_heads=2), L.SLS_EINVAL),
    (dict(page_size=3), L.SLS_EINVAL),
    (dict(page_size=512, capacity=1024), L.SLS_EINVAL),
    (dict(capacity=1000), L.SLS_EINVAL),                          # not a multiple of P
    (dict(dtype=7), L.SLS_EUNSUPPORTED),
    (dict(batch=0), L.SLS_EINVAL),
    (dict(scale=-1.0), L.SLS_EINVAL),
    (dict(flags=8), L.SLS_EINVAL),
    (dict(batch=1 << 30, num_q_heads=4, num_kv_heads=4), L.SLS_EOVERFLOW),    # rows > 2^31
    (dict(batch=1 << 20, num_kv_heads=2, capacity=1 << 30), L.SLS_EOVERFLOW),  # > 2^48 elements
])
def test_descriptor_validation(lib, kw, code):
    d = desc(**kw)
    st = lib.sls_pagemeta_build(ctypes.byref(d), BAD, BAD, BAD, BAD, None)
    assert st == code, err(lib)
    assert err(lib)


def test_null_arguments(lib):
    d = desc()
    assert lib.sls_pagemeta_build(None, BAD, BAD, BAD, BAD, None) == L.SLS_EINVAL
    assert lib.sls_pagemeta_build(ctypes.byref(d), None, BAD, BAD, BAD, None) == L.SLS_EINVAL
    assert "k_cache" in err(lib)
    assert lib.sls_sparse_decode_attend(ctypes.byref(d), BAD, BAD, BAD, BAD, 8, None, 8, BAD, 4,
                                        None, BAD, BAD, None) == L.SLS_EINVAL
    assert lib.sls_combine_splits(ctypes.byref(d), BAD, BAD, BAD, 4, None, None, None, None) == L.SLS_EINVAL


def test_select_pages_validation(lib):
    d = desc()
    ws = lib.sls_select_pages_workspace_size(ctypes.byref(d))
    assert ws == 2 * 2 * 64 * 4
    sel = lambda k, ns, nl, kmin=BAD, kmax=BAD, dd=d, wsb=1 << 40: lib.sls_select_pages(
        ctypes.byref(dd), BAD, kmin, kmax, BAD, k, ns, nl, BAD, BAD, wsb, None)
    assert sel(0, 0, 0) == L.SLS_EINVAL                  # k < 1
    assert sel(65, 0, 0) == L.SLS_EINVAL                 # k > Cap/P = 64
    assert sel(4, 1, 64) == L.SLS_EINVAL                 # forced pages do not fit
    assert "forced" in err(lib)
    assert sel(8, -1, 0) == L.SLS_EINVAL
    d1 = desc(page_size=1)
    assert sel(8, 4, 0, kmin=BAD, kmax=ctypes.c_void_p(0x2000), dd=d1) == L.SLS_EINVAL
    big = desc(page_size=1, capacity=1 << 22)            # 4M pages per row > supported
    assert sel(8, 0, 0, dd=big) == L.SLS_EUNSUPPORTED
    assert sel(8, 0, 0, wsb=ws - 1) == L.SLS_EWORKSPACE


def test_select_delta_validation_and_workspace(lib):
    d = desc(page_size=64, capacity=4096)
    ws = lib.sls_select_delta_workspace_size(ctypes.byref(d), 64)
    assert ws == ((2 * 2 * 64 + 255) // 256) * 256
    assert lib.sls_select_delta_workspace_size(ctypes.byref(d), 48) == 0
    call = lambda block=64, delta=5.0, stride=64, wsb=ws, wsp=BAD: lib.sls_select_delta(
        ctypes.byref(d), BAD, BAD, BAD, BAD, BAD, block, delta, BAD, BAD, stride, wsp, wsb, None)
    assert call(block=48) == L.SLS_EINVAL
    assert call(delta=-1.0) == L.SLS_EINVAL
    assert call(delta=float("inf")) == L.SLS_EINVAL
    assert call(stride=63) == L.SLS_EINVAL
    assert call(wsb=ws - 1) == L.SLS_EWORKSPACE
    assert call(wsp=None) == L.SLS_EWORKSPACE


def test_attend_validation(lib):
    d = desc()
    att = lambda stride=8, count=None, kf=8, S=4: lib.sls_sparse_decode_attend(
        ctypes.byref(d), BAD, BAD, BAD, BAD, stride, count, kf, BAD, S, BAD, BAD, BAD, None)
    assert att(S=0) == L.SLS_EINVAL
    assert att(S=1025) == L.SLS_EINVAL
    assert att(stride=0) == L.SLS_EINVAL
    assert att(kf=9) == L.SLS_EINVAL
    assert att(kf=-1) == L.SLS_EINVAL


def test_attend_combine_validation(lib):
    d = desc()
    ws = lib.sls_attend_combine_workspace_size(ctypes.byref(d), 4)
    # tickets (2*2 rows) + o_part (2*8*4*128 floats) + m and l (2*8*4 floats each), 256-aligned
    assert ws == 256 + 2 * 8 * 4 * 128 * 4 + 2 * 256
    assert lib.sls_attend_combine_workspace_size(ctypes.byref(d), -1) == 0
    assert lib.sls_attend_combine_workspace_size(ctypes.byref(d), 0) > 0   # library schedule
    call = lambda S=4, wsb=ws, out=BAD: lib.sls_sparse_decode_attend_combine(
        ctypes.byref(d), BAD, BAD, BAD, BAD, 8, None, 8, BAD, S, None, out, None, BAD, wsb, None)
    assert call(S=-1) == L.SLS_EINVAL
    assert call(S=1025) == L.SLS_EINVAL
    assert call(out=None) == L.SLS_EINVAL
    assert call(wsb=ws - 1) == L.SLS_EWORKSPACE
    assert lib.sls_attend_default_splits(None, 8) == 1


def test_quest_step_validation(lib):
    d = desc()
    ws = lib.sls_quest_decode_step_workspace_size(ctypes.byref(d), 8, 0)
    assert ws > 0
    call = lambda k=8, ms=0.0, wsb=ws, dd=d: lib.sls_quest_decode_step(
        ctypes.byref(dd), BAD, BAD, BAD, BAD, BAD, BAD, k, 0, 0, None, None, BAD, None, 0, ms, BAD, wsb, None)
    assert call(k=0) == L.SLS_EINVAL
    assert call(ms=-1.0) == L.SLS_EINVAL
    assert call(ms=float("inf")) == L.SLS_EINVAL
    assert call(wsb=ws - 1) == L.SLS_EWORKSPACE
    # the gate needs the one-launch kernel, which the CUDA-core flag turns off
    d2 = desc(flags=L.SLS_FLAG_CUDA_CORES)
    ws2 = lib.sls_quest_decode_step_workspace_size(ctypes.byref(d2), 8, 0)
    assert call(ms=8.0, wsb=ws2, dd=d2) == L.SLS_EUNSUPPORTED
    assert lib.sls_quest_decode_step_splits(ctypes.byref(d2), 8) == 0


def test_python_layer_raises_on_status(lib):
    d = desc(head_dim=96)
    with pytest.raises(L.SlsError) as e:
        L.call("sls_pagemeta_build", ctypes.byref(d), BAD, BAD, BAD, BAD, None)
    assert e.value.code == L.SLS_EUNSUPPORTED


def test_decode_append_validation(lib):
    d = desc()
    call = lambda kmin=BAD, kmax=BAD, ctx=BAD, dd=d: lib.sls_decode_append(
        ctypes.byref(dd), BAD, BAD, BAD, BAD, kmin, kmax, ctx, None, None)
    assert call(ctx=None) == L.SLS_EINVAL
    assert call(kmax=None) == L.SLS_EINVAL          # both summaries or neither
    assert "both or neither" in err(lib)
    assert call(dd=desc(page_size=1)) == L.SLS_EINVAL  # page size 1: the cache is its own metadata


def test_thumb_residual_validation(lib):
    d = desc(page_size=64)
    build = lambda block=64, res=BAD: lib.sls_thumb_residual_build(ctypes.byref(d), BAD, BAD, block, BAD, BAD, res,
                                                                   None)
    update = lambda block=64, res=BAD: lib.sls_thumb_residual_update(ctypes.byref(d), BAD, BAD, block, BAD, BAD, res,
                                                                     None)
    for f in (build, update):
        assert f(res=None) == L.SLS_EINVAL
        assert f(block=48) == L.SLS_EINVAL   # not a power of two
        assert f(block=8) == L.SLS_EINVAL    # below 16


def test_refined_attend_validation(lib):
    d = desc(page_size=64)
    ws = lib.sls_refined_decode_attend_workspace_size(ctypes.byref(d))
    assert ws > 0
    call = lambda dd=d, codes=BAD, res=BAD, stride=8, wsb=ws, out=BAD: lib.sls_refined_decode_attend_combine(
        ctypes.byref(dd), BAD, BAD, BAD, codes, BAD, res, BAD, stride, BAD, BAD, None, out, None, BAD, wsb, None)
    assert call(out=None) == L.SLS_EINVAL
    assert call(res=None) == L.SLS_EINVAL               # codes, scales and res: all or none
    assert call(stride=0) == L.SLS_EINVAL
    assert call(res=ctypes.c_void_p(0x1008)) == L.SLS_EINVAL  # 16-byte alignment
    assert call(codes=ctypes.c_void_p(0x1004)) == L.SLS_EINVAL
    assert call(wsb=ws - 1) == L.SLS_EWORKSPACE
    assert call(dd=desc(page_size=64, dtype=L.SLS_DTYPE_F32)) == L.SLS_EUNSUPPORTED
    assert call(dd=desc(page_size=64, num_q_heads=32, num_kv_heads=2)) == L.SLS_EUNSUPPORTED  # G = 16
    assert call(dd=desc(page_size=1)) == L.SLS_EUNSUPPORTED


def test_stats_counters_without_a_launch(lib):
    """Calls that fail validation launch nothing and count nothing; the
    counters read back and reset without a GPU."""
    st = L.Stats()
    assert lib.sls_get_stats(None, 0) == L.SLS_EINVAL
    d = desc()
    lib.sls_pagemeta_build(ctypes.byref(d), None, BAD, BAD, BAD, None)   # fails validation
    rc = lib.sls_get_stats(ctypes.byref(st), 1)
    assert rc in (L.SLS_OK, L.SLS_ECUDA)          # no device here: the row counters cannot be read
    assert st.metadata == 0 and st.quest_step_one_launch == 0


def test_misaligned_tensors_are_rejected(lib):
    """Tensors read in 16-byte vectors must be 16-byte aligned; a misaligned
    pointer is an argument error, reported before anything launches."""
    d = desc()
    M = ctypes.c_void_p(0x1002)   # a bf16 element past an aligned address
    ws = lib.sls_quest_decode_step_workspace_size(ctypes.byref(d), 8, 0)
    cases = {
        "k_cache": lambda: lib.sls_pagemeta_build(ctypes.byref(d), M, BAD, BAD, BAD, None),
        "kmax": lambda: lib.sls_pagemeta_update(ctypes.byref(d), BAD, BAD, BAD, M, None),
        "q": lambda: lib.sls_select_pages(ctypes.byref(d), M, BAD, BAD, BAD, 8, 0, 0, BAD, BAD, 1 << 40, None),
        "v_cache": lambda: lib.sls_sparse_decode_attend(ctypes.byref(d), BAD, BAD, M, BAD, 8, None, 8, BAD, 4,
                                                        BAD, BAD, BAD, None),
        "o_part": lambda: lib.sls_combine_splits(ctypes.byref(d), M, BAD, BAD, 4, None, BAD, None, None),
        "kmin": lambda: lib.sls_quest_decode_step(ctypes.byref(d), BAD, BAD, BAD, M, BAD, BAD, 8, 0, 0, None,
                                                  None, BAD, None, 0, 0.0, BAD, ws, None),
        "k_new": lambda: lib.sls_decode_append(ctypes.byref(d), M, BAD, BAD, BAD, None, None, BAD, None, None),
        "scales": lambda: lib.sls_thumb_build(ctypes.byref(desc(page_size=64)), BAD, BAD, 64, BAD, M, None),
    }
    for name, call in cases.items():
        assert call() == L.SLS_EINVAL, name
        assert name in err(lib) and "aligned" in err(lib), (name, err(lib))
