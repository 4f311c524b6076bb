"""ctypes binding of libsls.so (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

LIB_PATH = _build.LIB

SLS_OK, SLS_EINVAL, SLS_EUNSUPPORTED, SLS_EOVERFLOW, SLS_EWORKSPACE, SLS_ECUDA = 0, -1, -2, -3, -4, -5
SLS_ETIMEOUT, SLS_EDEVICE = -6, -7
SLS_DTYPE_F32, SLS_DTYPE_BF16 = 0, 1
SLS_FLAG_CUDA_CORES = 1
SLS_FLAG_NO_TMA = 2
SLS_FLAG_TEST_WAIT_TIMEOUT = 4  # test hook of the bounded waits (include/sls.h)


class AttnDesc(ctypes.Structure):
    """ctypes mirror of sls_attn_desc."""
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("capacity", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("scale", ctypes.c_float)]


class Stats(ctypes.Structure):
    """sls_stats: which paths the library took (include/sls.h)."""
    _fields_ = [(n, ctypes.c_uint64) for n in (
        "quest_step_one_launch", "quest_step_two_launch", "step_rows_dense", "step_rows_all_keys",
        "select_pages", "select_delta_tensor_cores", "select_delta_cuda_cores", "attend_tma", "attend_mma",
        "attend_cuda_cores", "attend_stream_k", "attend_refined", "combine", "metadata", "recall",
        "select_rows_all_keys", "attend_stream_k_tma", "attend_refined_tma")]


_P = ctypes.c_void_p
_I = ctypes.c_int32
_D = ctypes.POINTER(AttnDesc)
SIGNATURES = {
    "sls_pagemeta_build": (_I, [_D, _P, _P, _P, _P, _P]),
    "sls_pagemeta_update": (_I, [_D, _P, _P, _P, _P, _P]),
    "sls_decode_append": (_I, [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "sls_thumb_build": (_I, [_D, _P, _P, _I, _P, _P, _P]),
    "sls_thumb_update": (_I, [_D, _P, _P, _I, _P, _P, _P]),
    "sls_thumb_residual_build": (_I, [_D, _P, _P, _I, _P, _P, _P, _P]),
    "sls_thumb_residual_update": (_I, [_D, _P, _P, _I, _P, _P, _P, _P]),
    "sls_select_pages": (_I, [_D, _P, _P, _P, _P, _I, _I, _I, _P, _P, ctypes.c_size_t, _P]),
    "sls_select_pages_workspace_size": (ctypes.c_size_t, [_D]),
    "sls_select_pages_static": (_I, [_D, _P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "sls_select_delta_workspace_size": (ctypes.c_size_t, [_D, _I]),
    "sls_select_delta": (_I, [_D, _P, _P, _P, _P, _P, _I, ctypes.c_float, _P, _P, _I, _P,
                              ctypes.c_size_t, _P]),
    "sls_sparse_decode_attend": (_I, [_D, _P, _P, _P, _P, _I, _P, _I, _P, _I, _P, _P, _P, _P]),
    "sls_combine_splits": (_I, [_D, _P, _P, _P, _I, _P, _P, _P, _P]),
    "sls_attend_default_splits": (_I, [_D, _I]),
    "sls_attend_combine_workspace_size": (ctypes.c_size_t, [_D, _I]),
    "sls_sparse_decode_attend_combine": (_I, [_D, _P, _P, _P, _P, _I, _P, _I, _P, _I, _P, _P, _P, _P,
                                              ctypes.c_size_t, _P]),
    "sls_refined_decode_attend_workspace_size": (ctypes.c_size_t, [_D]),
    "sls_get_stats": (_I, [ctypes.POINTER(Stats), _I]),
    "sls_refined_decode_attend_combine": (_I, [_D, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P, _P,
                                               _P, ctypes.c_size_t, _P]),
    "sls_quest_decode_step_workspace_size": (ctypes.c_size_t, [_D, _I, _I]),
    "sls_quest_decode_step_splits": (_I, [_D, _I]),
    "sls_quest_decode_step": (_I, [_D, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _I, ctypes.c_float,
                                   _P, ctypes.c_size_t, _P]),
    "sls_selection_recall_workspace_size": (ctypes.c_size_t, [_D]),
    "sls_selection_recall": (_I, [_D, _P, _P, _P, _I, _P, _I, _P, _P, _P, ctypes.c_size_t, _P]),
    "sls_pipeline_check": (_I, []),
    "sls_last_error": (ctypes.c_char_p, []),
    "sls_version": (_I, []),
}

_lock = threading.Lock()
_lib = None


class SlsError(RuntimeError):
    """A non-zero sls_status, with the library's sls_last_error() message."""
    def __init__(self, fn, code, msg):
        super().__init__(f"{fn} failed with status {code}: {msg}")
        self.code = code


def load(build_if_missing: bool = False):
    """Load libsls.so.  Raises if it is missing (unless asked to build it)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            if not build_if_missing:
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -m sparse_long_context_gb300.build)")
            _build.build()
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def check(fn_name: str, status: int) -> None:
    """Raises SlsError when a C call returned a non-zero status."""
    if status != SLS_OK:
        msg = _lib.sls_last_error().decode() if _lib is not None else ""
        raise SlsError(fn_name, status, msg)


def call(name: str, *args) -> None:
    """Calls the named C entry point and raises SlsError on a non-zero status."""
    lib = load()
    check(name, getattr(lib, name)(*args))
