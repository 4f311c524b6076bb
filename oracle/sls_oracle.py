"""The fp64 CPU oracle: Python binding of the plain C++ oracle.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline leg import this module; the library never
does.  Every computation happens in ``sls_oracle.cpp`` (C++17, double
precision, plain loops over the pages' definitions; the sources and readings
are cited there, function by function).  This module only marshals numpy
arrays into pointers and sizes and the results back into arrays, with the
same function names and signatures as the numpy implementation in
``numpy_oracle.py`` (a second oracle, cross-checked against this one).

``Oracle(path)`` binds any build of the source (the mutation check binds
planted-mistake builds); the module-level functions are bound to the
default build, ``oracle/libslsoracle.so``, which is compiled from the source
on first import when it is missing or older than the source.
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional

import numpy as np

from . import build_oracle

NEG_INF = -math.inf
RES_DENOM = 508.0

_c_i64 = ctypes.c_longlong
_c_int = ctypes.c_int
_c_dbl = ctypes.c_double
_vp = ctypes.c_void_p


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float64)


def _i64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64).reshape(-1))


def _u8(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.uint8)


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(_vp)


def _mat(x) -> np.ndarray:
    """A 2-D float64 array (a [0, D] array stays 2-D)."""
    a = _f64(x)
    return a.reshape(1, -1) if a.ndim == 1 else a


class Oracle:
    """One build of the C++ oracle, with the oracle's functions as methods."""

    _SIGS = {
        "orc_bf16_to_f64": (None, [_vp, _c_i64, _vp]),
        "orc_f32_to_f64": (None, [_vp, _c_i64, _vp]),
        "orc_softmax_attention": (None, [_vp, _c_int, _c_int, _vp, _vp, _c_i64, _c_int, _c_dbl, _vp, _vp, _vp]),
        "orc_split_partials": (None, [_vp, _c_int, _c_int, _vp, _vp, _c_int, _c_dbl, _vp, _c_int, _vp, _vp, _vp]),
        "orc_combine_partials": (None, [_c_int, _c_int, _c_int, _vp, _vp, _vp, _vp, _vp, _vp]),
        "orc_num_pages": (_c_i64, [_c_i64, _c_i64]),
        "orc_page_minmax": (None, [_vp, _c_int, _c_i64, _c_int, _vp, _vp]),
        "orc_quest_bound": (None, [_vp, _c_int, _c_int, _vp, _vp, _c_i64, _vp]),
        "orc_group_score": (None, [_vp, _c_int, _c_i64, _vp]),
        "orc_forced_pages": (_c_i64, [_c_i64, _c_int, _c_int, _c_int, _vp]),
        "orc_select_topk": (_c_i64, [_vp, _c_i64, _c_i64, _vp, _c_i64, _vp]),
        "orc_kth_score": (_c_dbl, [_vp, _c_i64, _c_i64, _vp, _c_i64]),
        "orc_pages_to_tokens": (_c_i64, [_vp, _c_i64, _c_i64, _c_int, _vp]),
        "orc_quest_select_row": (_c_i64, [_vp, _c_int, _c_int, _vp, _c_i64, _c_int, _c_i64, _c_int, _c_int,
                                          _vp, _vp, _vp]),
        "orc_thumb_quantize": (None, [_vp, _c_int, _c_int, _vp, _vp]),
        "orc_thumb_dequant": (None, [_vp, _vp, _c_int, _c_int, _c_int, _vp]),
        "orc_pack_codes": (None, [_vp, _c_int, _c_int, _vp]),
        "orc_unpack_codes": (None, [_vp, _c_int, _c_int, _vp]),
        "orc_thumbnails_row": (None, [_vp, _c_int, _c_i64, _c_int, _vp, _vp]),
        "orc_delta_forced_blocks": (_c_i64, [_c_i64, _c_int, _vp]),
        "orc_pseudo_max": (None, [_vp, _c_int, _c_int, _vp, _c_i64, _c_int, _c_dbl, _vp]),
        "orc_delta_block_margin": (_c_i64, [_vp, _c_int, _c_int, _vp, _c_i64, _c_int, _c_dbl, _vp, _vp]),
        "orc_delta_select_row": (_c_i64, [_vp, _c_int, _c_int, _vp, _c_i64, _c_int, _c_dbl, _c_dbl, _vp, _vp,
                                          _vp, _vp]),
        "orc_residual_quantize": (None, [_vp, _vp, _vp, _c_int, _c_int, _vp]),
        "orc_refined_keys": (None, [_vp, _vp, _vp, _c_int, _c_int, _c_int, _vp]),
        "orc_residuals_row": (None, [_vp, _c_int, _c_i64, _c_int, _vp, _vp, _vp]),
        "orc_refined_attention_row": (None, [_vp, _c_int, _c_int, _vp, _vp, _vp, _c_i64, _c_i64, _c_int, _c_dbl,
                                             _vp, _vp, _vp]),
        "orc_attention_mass_recall": (None, [_vp, _c_int, _c_int, _vp, _vp, _c_i64, _c_i64, _c_int, _c_dbl, _vp]),
        "orc_sparse_attention_row": (None, [_vp, _c_int, _c_int, _vp, _vp, _vp, _c_i64, _c_i64, _c_int, _c_dbl,
                                            _vp, _vp, _vp]),
        "orc_quest_step": (_c_int, [_vp, _vp, _vp, _c_int, _vp, _c_int, _c_int, _c_int, _c_int, _c_i64, _c_int,
                                         _c_int, _c_int, _c_int, _c_dbl, _vp, _vp, _c_int, _c_int, _c_dbl,
                                         _vp, _vp, _vp, _vp]),
        "orc_delta_step": (_c_int, [_vp, _vp, _vp, _c_int, _vp, _c_int, _c_int, _c_int, _c_int, _c_i64, _c_int,
                                         _c_dbl, _c_dbl, _vp, _c_int, _vp, _c_int, _c_int, _c_dbl, _vp, _vp,
                                         _vp, _vp, _vp]),
    }

    NEG_INF = NEG_INF
    RES_DENOM = RES_DENOM

    def __init__(self, path: Optional[str] = None):
        self.path = path or build_oracle.build()
        self.lib = ctypes.CDLL(self.path)
        for name, (res, args) in self._SIGS.items():
            fn = getattr(self.lib, name)
            fn.restype = res
            fn.argtypes = args

    # ------------------------------------------------------------ decoding

    def to_f64(self, x, dtype: str) -> np.ndarray:
        """Exact float64 value of an fp32 array or of bf16 bit patterns (uint16)."""
        if dtype == "bf16":
            a = np.ascontiguousarray(x, dtype=np.uint16)
            out = np.empty(a.shape, np.float64)
            self.lib.orc_bf16_to_f64(_p(a), a.size, _p(out))
            return out
        a = np.ascontiguousarray(x, dtype=np.float32)
        out = np.empty(a.shape, np.float64)
        self.lib.orc_f32_to_f64(_p(a), a.size, _p(out))
        return out

    # ----------------------------------------------------------- attention

    def softmax_attention(self, q, K, V, scale: float, sink=None):
        """(o [G, Dv], lse [G]) of G query rows over the rows of K and V."""
        q = _mat(q)
        G, Dq = q.shape
        K = _f64(K).reshape(-1, Dq)
        V = _f64(V)
        Dv = V.shape[1] if V.ndim == 2 else Dq
        sk = None if sink is None else _f64(sink).reshape(-1)
        o, lse = np.empty((G, Dv)), np.empty(G)
        self.lib.orc_softmax_attention(_p(q), G, Dq, _p(K), _p(V), K.shape[0], Dv, float(scale), _p(sk),
                                       _p(o), _p(lse))
        return o, lse

    def split_partials(self, q, K, V, scale, bounds):
        """[(m [G], l [G], acc [G, Dv])] for each key slice [a, b) in bounds."""
        q, K, V = _mat(q), _f64(K), _f64(V)
        G, Dq = q.shape
        Dv = V.shape[1]
        b = _i64([x for ab in bounds for x in ab])
        S = len(bounds)
        m, l, acc = np.empty((S, G)), np.empty((S, G)), np.empty((S, G, Dv))
        self.lib.orc_split_partials(_p(q), G, Dq, _p(K), _p(V), Dv, float(scale), _p(b), S, _p(m), _p(l), _p(acc))
        return [(m[s], l[s], acc[s]) for s in range(S)]

    def combine_partials(self, parts, sink=None):
        """(o [G, D], lse [G]) merged from split partials."""
        m = _f64(np.stack([p[0] for p in parts]))
        l = _f64(np.stack([p[1] for p in parts]))
        acc = _f64(np.stack([p[2] for p in parts]))
        S, G, D = acc.shape
        sk = None if sink is None else _f64(sink).reshape(-1)
        o, lse = np.empty((G, D)), np.empty(G)
        self.lib.orc_combine_partials(S, G, D, _p(m), _p(l), _p(acc), _p(sk), _p(o), _p(lse))
        return o, lse

    # --------------------------------------------------------------- Quest

    def num_pages(self, n: int, page_size: int) -> int:
        return int(self.lib.orc_num_pages(int(n), int(page_size)))

    def page_minmax(self, K, n: int, page_size: int):
        """(kmin, kmax) [NP, D] over the valid keys of each page."""
        K = _mat(K)
        D = K.shape[1]
        NP = self.num_pages(n, page_size)
        kmin, kmax = np.empty((NP, D)), np.empty((NP, D))
        self.lib.orc_page_minmax(_p(K), D, int(n), int(page_size), _p(kmin), _p(kmax))
        return kmin, kmax

    def quest_bound(self, q, kmin, kmax, chunk: int = 4096):
        """U [G, NP] = sum_c max(q kmin, q kmax)."""
        q, kmin, kmax = _mat(q), _mat(kmin), _mat(kmax)
        G, D = q.shape
        NP = kmin.shape[0]
        U = np.empty((G, NP))
        self.lib.orc_quest_bound(_p(q), G, D, _p(kmin), _p(kmax), NP, _p(U))
        return U

    def group_score(self, U) -> np.ndarray:
        U = _mat(U)
        s = np.empty(U.shape[1])
        self.lib.orc_group_score(_p(U), U.shape[0], U.shape[1], _p(s))
        return s

    def forced_pages(self, n: int, page_size: int, n_sink_pages: int, n_local_tokens: int) -> np.ndarray:
        out = np.empty(self.num_pages(n, page_size) + 1, np.int64)
        c = self.lib.orc_forced_pages(int(n), int(page_size), int(n_sink_pages), int(n_local_tokens), _p(out))
        return out[:c].copy()

    def select_topk(self, score, k: int, forced) -> np.ndarray:
        score, forced = _f64(score).reshape(-1), _i64(forced)
        NP = score.shape[0]
        out = np.empty(max(int(k), NP) + 1, np.int64)
        c = self.lib.orc_select_topk(_p(score), NP, int(k), _p(forced), forced.size, _p(out))
        if c < 0:
            raise ValueError("budget smaller than the forced pages")
        return out[:c].copy()

    def kth_score(self, score, k: int, forced) -> float:
        score, forced = _f64(score).reshape(-1), _i64(forced)
        return float(self.lib.orc_kth_score(_p(score), score.shape[0], int(k), _p(forced), forced.size))

    def pages_to_tokens(self, pages, n: int, page_size: int) -> np.ndarray:
        pages = _i64(pages)
        out = np.empty(pages.size * int(page_size) + 1, np.int64)
        c = self.lib.orc_pages_to_tokens(_p(pages), pages.size, int(n), int(page_size), _p(out))
        return out[:c].copy()

    def quest_select_row(self, q, K, n, page_size, k, n_sink_pages, n_local_tokens):
        """(pages, group score per page, k-th admitted score) of one row."""
        q, K = _mat(q), _mat(K)
        G, D = q.shape
        NP = self.num_pages(n, page_size)
        pages = np.empty(max(int(k), NP) + 1, np.int64)
        score = np.empty(NP)
        kth = _c_dbl(0.0)
        c = self.lib.orc_quest_select_row(_p(q), G, D, _p(K), int(n), int(page_size), int(k), int(n_sink_pages),
                                          int(n_local_tokens), _p(pages), _p(score), ctypes.byref(kth))
        if c < 0:
            raise ValueError("budget smaller than the forced pages")
        return pages[:c].copy(), score, float(kth.value)

    # ----------------------------------------------------------------- FFD

    def thumb_quantize(self, Kb):
        """(codes [T, D] uint8, s [D]) of one block."""
        Kb = _mat(Kb)
        T, D = Kb.shape
        codes, s = np.empty((T, D), np.uint8), np.empty(D)
        self.lib.orc_thumb_quantize(_p(Kb), T, D, _p(codes), _p(s))
        return codes, s

    def thumb_dequant(self, codes, s) -> np.ndarray:
        codes = _u8(codes)
        T, D = codes.shape
        s = _f64(s)
        rows = 1 if s.size == D else T
        s = np.ascontiguousarray(s.reshape(rows, D))
        out = np.empty((T, D))
        self.lib.orc_thumb_dequant(_p(codes), _p(s), T, D, rows, _p(out))
        return out

    def pack_codes(self, codes) -> np.ndarray:
        codes = _u8(codes)
        T, D = codes.shape
        out = np.empty((T, D // 4), np.uint8)
        self.lib.orc_pack_codes(_p(codes), T, D, _p(out))
        return out

    def unpack_codes(self, packed) -> np.ndarray:
        packed = _u8(packed)
        T, W = packed.shape
        out = np.empty((T, 4 * W), np.uint8)
        self.lib.orc_unpack_codes(_p(packed), T, W, _p(out))
        return out

    def thumbnails_row(self, K, n: int, block: int):
        K = _mat(K)
        D = K.shape[1]
        nfull = int(n) // int(block)
        codes, scales = np.zeros((nfull * block, D), np.uint8), np.zeros((nfull, D))
        self.lib.orc_thumbnails_row(_p(K), D, int(n), int(block), _p(codes), _p(scales))
        return codes, scales

    def delta_forced_blocks(self, n: int, block: int) -> np.ndarray:
        out = np.empty(2, np.int64)
        c = self.lib.orc_delta_forced_blocks(int(n), int(block), _p(out))
        return out[:c].copy()

    def pseudo_max(self, q, K, n: int, block: int, scale: float) -> np.ndarray:
        q, K = _mat(q), _mat(K)
        G, D = q.shape
        out = np.empty(G)
        self.lib.orc_pseudo_max(_p(q), G, D, _p(K), int(n), int(block), float(scale), _p(out))
        return out

    def delta_block_margin(self, q, K, n, block, scale):
        """(scanned blocks, margins) of the complete non-forced blocks."""
        q, K = _mat(q), _mat(K)
        G, D = q.shape
        cap = int(n) // int(block) + 1
        blocks, margins = np.empty(cap, np.int64), np.empty(cap)
        c = self.lib.orc_delta_block_margin(_p(q), G, D, _p(K), int(n), int(block), float(scale), _p(blocks),
                                            _p(margins))
        return blocks[:c].copy(), margins[:c].copy()

    def delta_select_row(self, q, K, n, block, delta, scale):
        """(kept blocks ascending, (scanned blocks, margins))."""
        q, K = _mat(q), _mat(K)
        G, D = q.shape
        cap = -(-int(n) // int(block)) + 2
        sel, blocks, margins = np.empty(cap, np.int64), np.empty(cap, np.int64), np.empty(cap)
        ns = _c_i64(0)
        c = self.lib.orc_delta_select_row(_p(q), G, D, _p(K), int(n), int(block), float(delta), float(scale),
                                          _p(sel), _p(blocks), _p(margins), ctypes.byref(ns))
        k = int(ns.value)
        return sel[:c].copy(), (blocks[:k].copy(), margins[:k].copy())

    def residual_quantize(self, Kb, codes, s) -> np.ndarray:
        Kb, codes, s = _mat(Kb), _u8(codes), _f64(s).reshape(-1)
        T, D = Kb.shape
        r = np.empty((T, D), np.int8)
        self.lib.orc_residual_quantize(_p(Kb), _p(codes), _p(s), T, D, _p(r))
        return r

    def refined_keys(self, codes, s, r) -> np.ndarray:
        codes = _u8(codes)
        T, D = codes.shape
        s = _f64(s)
        rows = 1 if s.size == D else T
        s = np.ascontiguousarray(s.reshape(rows, D))
        r = np.ascontiguousarray(r, dtype=np.int8)
        out = np.empty((T, D))
        self.lib.orc_refined_keys(_p(codes), _p(s), _p(r), T, D, rows, _p(out))
        return out

    def residuals_row(self, K, n: int, block: int):
        K = _mat(K)
        D = K.shape[1]
        nfull = int(n) // int(block)
        codes, scales = np.zeros((nfull * block, D), np.uint8), np.zeros((nfull, D))
        res = np.zeros((nfull * block, D), np.int8)
        self.lib.orc_residuals_row(_p(K), D, int(n), int(block), _p(codes), _p(scales), _p(res))
        return codes, scales, res

    def refined_attention_row(self, q, K, V, blocks, n, block, scale, sink=None):
        q, K, V, blocks = _mat(q), _mat(K), _mat(V), _i64(blocks)
        G, D = q.shape
        sk = None if sink is None else _f64(sink).reshape(-1)
        o, lse = np.empty((G, D)), np.empty(G)
        self.lib.orc_refined_attention_row(_p(q), G, D, _p(K), _p(V), _p(blocks), blocks.size, int(n), int(block),
                                           float(scale), _p(sk), _p(o), _p(lse))
        return o, lse

    # --------------------------------------------------- selection quality

    def attention_mass_recall(self, q, K, pages, n: int, page_size: int, scale: float) -> np.ndarray:
        q, K, pages = _mat(q), _mat(K), _i64(pages)
        G, D = q.shape
        out = np.empty(G)
        self.lib.orc_attention_mass_recall(_p(q), G, D, _p(K), _p(pages), pages.size, int(n), int(page_size),
                                           float(scale), _p(out))
        return out

    # ------------------------------------------------------- one decode row

    def sparse_attention_row(self, q, K, V, pages, n, page_size, scale, sink=None):
        q, K, V, pages = _mat(q), _mat(K), _mat(V), _i64(pages)
        G, D = q.shape
        sk = None if sink is None else _f64(sink).reshape(-1)
        o, lse = np.empty((G, D)), np.empty(G)
        self.lib.orc_sparse_attention_row(_p(q), G, D, _p(K), _p(V), _p(pages), pages.size, int(n), int(page_size),
                                          float(scale), _p(sk), _p(o), _p(lse))
        return o, lse

    # ------------------------------------------------ whole steps (timed)

    @staticmethod
    def _step_inputs(q, K, V, ctx_len, rows):
        f32 = np.asarray(K).dtype == np.float32
        dt = np.float32 if f32 else np.uint16
        return (np.ascontiguousarray(q, dt), np.ascontiguousarray(K, dt), np.ascontiguousarray(V, dt), int(f32),
                np.ascontiguousarray(ctx_len, np.int32), np.ascontiguousarray(rows, np.int32))

    def quest_step(self, q, K, V, ctx_len, num_q_heads, page_size, k, n_sink_pages, n_local_tokens,
                   scale, sink, rows, threads: int = 1, min_busy: float = 0.0):
        """The Quest step over the listed rows (ids b * Hkv + h) of a
        workload (bf16 bit patterns or fp32), on `threads` std::threads;
        returns (pages [nrows, k], o [nrows, G, D], lse [nrows, G], busy
        seconds, bytes, repetitions)."""
        q, K, V, f32, ctx, rows = self._step_inputs(q, K, V, ctx_len, rows)
        B, Hkv, Cap, D = K.shape
        G = num_q_heads // Hkv
        sk = None if sink is None else np.ascontiguousarray(sink, np.float32)
        nr = rows.size
        pages = np.empty((nr, int(k)), np.int32)
        o, lse, st = np.empty((nr, G, D)), np.empty((nr, G)), np.empty(3)
        rc = self.lib.orc_quest_step(_p(q), _p(K), _p(V), f32, _p(ctx), B, int(num_q_heads), Hkv, D, Cap,
                                     int(page_size), int(k), int(n_sink_pages), int(n_local_tokens),
                                     float(scale), _p(sk), _p(rows), nr, int(threads), float(min_busy),
                                     _p(pages), _p(o), _p(lse), _p(st))
        if rc != 0:
            raise ValueError("budget smaller than the forced pages")
        return pages, o, lse, float(st[0]), float(st[1]), int(st[2])

    def delta_step(self, q, K, V, ctx_len, num_q_heads, block, delta, scale, sink, rows, refined=False,
                   threads: int = 1, min_busy: float = 0.0):
        """The top-delta step over the listed rows of a bf16 workload; returns
        (count [nrows], blocks [nrows, Cap/block], o, lse, busy seconds,
        bytes, repetitions)."""
        q, K, V, f32, ctx, rows = self._step_inputs(q, K, V, ctx_len, rows)
        if f32:
            raise ValueError("the top-delta step takes bf16 inputs")
        B, Hkv, Cap, D = K.shape
        G = num_q_heads // Hkv
        sk = None if sink is None else np.ascontiguousarray(sink, np.float32)
        nr = rows.size
        count, blocks = np.empty(nr, np.int32), np.empty((nr, Cap // int(block)), np.int32)
        o, lse, st = np.empty((nr, G, D)), np.empty((nr, G)), np.empty(3)
        self.lib.orc_delta_step(_p(q), _p(K), _p(V), f32, _p(ctx), B, int(num_q_heads), Hkv, D, Cap, int(block),
                                float(delta), float(scale), _p(sk), int(bool(refined)), _p(rows), nr,
                                int(threads), float(min_busy), _p(count), _p(blocks), _p(o), _p(lse), _p(st))
        return count, blocks, o, lse, float(st[0]), float(st[1]), int(st[2])


_DEFAULT = Oracle()

_FUNCS = ("to_f64", "softmax_attention", "split_partials", "combine_partials", "num_pages", "page_minmax",
          "quest_bound", "group_score", "forced_pages", "select_topk", "kth_score", "pages_to_tokens",
          "quest_select_row", "thumb_quantize", "thumb_dequant", "pack_codes", "unpack_codes", "thumbnails_row",
          "delta_forced_blocks", "pseudo_max", "delta_block_margin", "delta_select_row", "residual_quantize",
          "refined_keys", "residuals_row", "refined_attention_row", "attention_mass_recall",
          "sparse_attention_row", "quest_step", "delta_step")
for _name in _FUNCS:
    globals()[_name] = getattr(_DEFAULT, _name)
del _name
