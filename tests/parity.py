"""Helpers of the GPU parity tests: move a generated workload to the device,
run the CUDA path through the C ABI, and compare it with the fp64 oracle.

Tolerances (the workload list's stated ones): bf16 inputs max-abs <= 2e-2
and rel-L2 <= 1e-2; fp32 inputs rel-L2 <= 1e-5.  Page and block sets must
be identical except boundary ties: a page may differ only when its oracle
score is within 1e-5 (relative) of the k-th admitted score; a block only
when its margin is within 1e-5 * max(1, |pseudo-max|) of -delta.  Ties are
counted and returned.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

from oracle import sls_oracle as O
from sparse_long_context_gb300 import harness as H
from sparse_long_context_gb300 import ops
from sparse_long_context_gb300 import workloads as W

TIE_REL = 1e-5
BF16_MAX_ABS, BF16_REL_L2 = 2e-2, 1e-2
F32_REL_L2 = 1e-5


to_device = H.to_device
DeviceWorkload = H.DeviceWorkload
upload = H.upload
run_step = H.run_step


def attend_on(dw: DeviceWorkload, pages_per_row, num_splits=4):
    """GPU attend + combine over the given page lists (one per row)."""
    s = dw.spec
    width = max(1, max(len(p) for p in pages_per_row))
    idx = np.full((s.rows, width), -1, dtype=np.int32)
    for r, p in enumerate(pages_per_row):
        idx[r, :len(p)] = p
    idx_d = torch.from_numpy(idx).cuda()
    parts = ops.sparse_decode_attend(dw.desc, dw.q, dw.K, dw.V, idx_d, dw.ctx, num_splits)
    out, lse = ops.combine_splits(dw.desc, parts, dw.sink)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


@dataclasses.dataclass
class OracleRow:
    pages: np.ndarray
    score: np.ndarray      # quest: group score per page; delta: margins of scanned blocks
    kth: float             # quest: k-th admitted score
    blocks: np.ndarray     # delta: scanned blocks
    pseudo_max: np.ndarray
    o: np.ndarray
    lse: np.ndarray


def oracle_row(spec: W.Spec, host: W.Tensors, b: int, h: int) -> OracleRow:
    G = spec.group
    q = O.to_f64(host.q[b, h * G:(h + 1) * G], spec.dtype)
    K = O.to_f64(host.K[b, h], spec.dtype)
    V = O.to_f64(host.V[b, h], spec.dtype)
    n = int(host.ctx_len[b])
    sink = None if host.sink is None else host.sink[h * G:(h + 1) * G].astype(np.float64)
    if spec.selector == "quest":
        pages, score, kth = O.quest_select_row(q, K, n, spec.page_size, spec.k_pages,
                                               spec.n_sink_pages, spec.n_local_tokens)
        blocks, pm = np.zeros(0, np.int64), np.zeros(0)
    else:
        pages, (blocks, score) = O.delta_select_row(q, K, n, spec.block, spec.delta, spec.scale)
        pm = O.pseudo_max(q, K, n, spec.block, spec.scale) if n > 0 else np.zeros(G)
        kth = math.nan
    o, lse = O.sparse_attention_row(q, K, V, pages, n, spec.page_size, spec.scale, sink)
    return OracleRow(pages, score, kth, blocks, pm, o, lse)


def check_quest_list(gpu_row: np.ndarray, orc: OracleRow, n: int, P: int, k: int) -> int:
    """Assert the GPU page list matches the oracle's up to boundary ties;
    returns the number of tied pages that differ."""
    NP = -(-n // P)
    if NP <= k:
        expect = np.concatenate([np.arange(NP), np.full(k - NP, -1)])
        assert np.array_equal(gpu_row, expect), (gpu_row[:16], NP)
        return 0
    assert np.all(gpu_row >= 0) and np.all(gpu_row < NP), "page index out of range"
    assert np.all(np.diff(gpu_row) > 0), "list not strictly ascending"
    g, o = set(gpu_row.tolist()), set(orc.pages.tolist())
    diff = g ^ o
    for p in diff:
        assert abs(orc.score[p] - orc.kth) <= TIE_REL * abs(orc.kth), \
            f"page {p} differs: score {orc.score[p]!r} vs k-th {orc.kth!r}"
    return len(diff) // 2


def check_delta_list(count: int, gpu_row: np.ndarray, orc: OracleRow, delta: float) -> int:
    lst = gpu_row[:count]
    assert np.all(np.diff(lst) > 0), "list not strictly ascending"
    g, o = set(lst.tolist()), set(orc.pages.tolist())
    diff = g ^ o
    margin = dict(zip(orc.blocks.tolist(), orc.score.tolist()))
    tol = TIE_REL * max(1.0, float(np.abs(orc.pseudo_max).max()) if orc.pseudo_max.size else 1.0)
    for j in diff:
        assert j in margin, f"block {j} is forced or out of range but differs"
        assert abs(margin[j] + delta) <= tol, f"block {j} differs: margin {margin[j]!r}"
    return len(diff)


def out_errors(gpu: np.ndarray, ref: np.ndarray):
    d = gpu - ref
    rn = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(d)) / rn if rn > 0 else float(np.linalg.norm(d))
    return float(np.abs(d).max()) if d.size else 0.0, rel


def assert_close(spec: W.Spec, gpu: np.ndarray, ref: np.ndarray, what=""):
    mx, rel = out_errors(gpu, ref)
    if spec.dtype == "bf16":
        assert mx <= BF16_MAX_ABS and rel <= BF16_REL_L2, f"{what}: max-abs {mx:.3g} rel-L2 {rel:.3g}"
    else:
        assert rel <= F32_REL_L2, f"{what}: rel-L2 {rel:.3g}"
    return mx, rel


RES_TIE_REL = 1e-6  # float32 rounding of the kernel's residual quotient (a few ulps of 2^-24)


def check_residuals(gpu_res: np.ndarray, K: np.ndarray, n: int, block: int) -> int:
    """Compare a row's GPU 8-bit residuals [>= nfull*block, D] with the
    oracle's, which decides r = round((k - k^) * 508 / s) exactly.  The
    kernel decides it in float32, so an element may differ by one only where
    the exact quotient lies within float32 rounding of a half-integer; such
    elements are counted and returned.  Codes and scales must agree exactly
    (checked by the caller)."""
    codes, scales, ores = O.residuals_row(K, n, block)
    nfull = n // block
    got = gpu_res[:nfull * block].astype(np.int32)
    want = ores.astype(np.int32)
    bad = np.argwhere(got != want)
    for t, c in bad:
        assert abs(int(got[t, c]) - int(want[t, c])) == 1, (t, c, got[t, c], want[t, c])
        s = scales[t // block, c]
        kh = (float(codes[t, c]) - 1.5) * (s / 2.0)
        x = (K[t, c] - kh) * O.RES_DENOM / s
        frac = x - np.floor(x)
        assert abs(frac - 0.5) <= RES_TIE_REL * max(1.0, abs(x)), (t, c, x)
    return len(bad)
