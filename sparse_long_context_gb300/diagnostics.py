"""Selection-quality diagnostics on the synthetic workloads.

For one decode step of a workload this reports, per query head:

* attention-mass recall of the selected pages ("Don't read the haystack",
  Part three: how much of the true attention mass the selection holds),
  from ``sls_selection_recall``;
* the relative L2 error of the sparse output against dense attention over
  the whole context (the split-K attend kernel with no page list);
* for the top-delta workload, top-delta against Quest top-k at the same
  budget (the mean number of blocks top-delta keeps per row): recall of both,
  and the device time of each selector run as its own kernels ("Faster Than
  Flash", the selection-rule overhead at identical keep ratios), L2 flushed
  before every timed launch;
* needle recall: the share of each row's planted needle pages (blocks) that
  its list holds (the synthetic queries are built to look for the needles,
  so this checks the generator as much as the selection).

Usage: ``python -m sparse_long_context_gb300.diagnostics --workload qwen1p5b --batch 4``
prints one JSON object.  Everything runs on the GPU through the C ABI; the
statistics at the end are host arithmetic on the results.
"""
from __future__ import annotations

import argparse
import json

import numpy as np
import torch

from . import harness as H
from . import ops
from . import workloads as W


def _stats(x: np.ndarray) -> dict:
    x = np.asarray(x, np.float64).ravel()
    return {"min": float(x.min()), "p10": float(np.percentile(x, 10)), "median": float(np.median(x)),
            "mean": float(x.mean())}


def needle_recall(lists: np.ndarray, counts, needles, unit: int, num_kv_heads: int) -> np.ndarray:
    """Per row r = b * Hkv + h: the fraction of the pages (blocks) of ``unit``
    tokens holding row r's needle tokens that appear in the row's list
    (``lists[r, :counts[r]]``, or the whole row when counts is None).  Rows
    without needles are left out."""
    out = []
    for r in range(lists.shape[0]):
        b, h = divmod(r, num_kv_heads)
        nd = needles[b][h] if b < len(needles) else None
        if nd is None or np.asarray(nd).size == 0:
            continue
        pages = np.unique(np.asarray(nd, dtype=np.int64) // unit)
        sel = lists[r] if counts is None else lists[r, :int(counts[r])]
        out.append(float(np.isin(pages, sel).mean()))
    return np.asarray(out, np.float64)


def quest_quality(dw: H.DeviceWorkload) -> dict:
    """Recall of the Quest selection and the sparse output's error vs dense."""
    s = dw.spec
    step = H.make_step(dw)
    out, _ = step(dw.q, dw.K, dw.V, dw.kmin, dw.kmax, dw.ctx, dw.sink)
    out = out.float().clone()
    rec = ops.selection_recall(dw.desc, dw.q, dw.K, step.page_idx, dw.ctx)
    S = ops.default_splits(dw.desc, s.capacity // s.page_size)
    dense, _ = ops.sparse_decode_attend_combine(dw.desc, dw.q, dw.K, dw.V, None, dw.ctx, S, sink=dw.sink)
    dense = dense.float()
    rel = torch.linalg.vector_norm(out - dense, dim=-1) / torch.linalg.vector_norm(dense, dim=-1).clamp_min(1e-30)
    ops.pipeline_check()
    nr = needle_recall(step.page_idx.cpu().numpy(), None, dw.host.needles, s.page_size, s.num_kv_heads)
    return {"selector": "quest", "budget_pages": s.k_pages, "recall": _stats(rec.cpu().numpy()),
            "rel_l2_vs_dense": _stats(rel.cpu().numpy()), "needle_recall": _stats(nr) if nr.size else None}


def _timed(fn, reps: int = 30) -> float:
    """Mean device time (us) of fn() over reps launches, each preceded by a
    write of a buffer larger than L2 (outside the timed events)."""
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    times = []
    for i in range(reps + 3):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    return float(np.mean([1e3 * a.elapsed_time(b) for a, b in times[3:]]))


def delta_vs_topk(dw: H.DeviceWorkload, time_selectors: bool = True) -> dict:
    """Top-delta's kept blocks against Quest top-k at the same mean budget."""
    s = dw.spec
    step = H.make_step(dw)
    step(dw.q, dw.K, dw.V, dw.codes, dw.scales, dw.ctx, dw.sink)
    cnt = step.count
    rec_d = ops.selection_recall(dw.desc, dw.q, dw.K, step.block_idx, dw.ctx, count=cnt)
    k = max(1, int(round(float(cnt.float().mean()))))
    kmin, kmax = ops.pagemeta_build(dw.desc, dw.K, dw.ctx)
    page_idx = ops.select_pages(dw.desc, dw.q, kmin, kmax, dw.ctx, k, 1, s.block)
    rec_q = ops.selection_recall(dw.desc, dw.q, dw.K, page_idx, dw.ctx)
    ops.pipeline_check()
    times = None
    if time_selectors:
        ws = ops.select_pages_workspace(dw.desc)
        times = {"select_delta_us": _timed(lambda: step.select(dw.q, dw.K, dw.codes, dw.scales, dw.ctx)),
                 "select_pages_us": _timed(lambda: ops.select_pages(dw.desc, dw.q, kmin, kmax, dw.ctx, k, 1, s.block,
                                                                    out=page_idx, workspace=ws)),
                 "how": "each selector alone (top-delta: scan + compaction; Quest: bound + top-k over "
                        f"{s.block}-token page min/max at the matched budget), L2 flushed before each launch"}
        ops.pipeline_check()
    nr = needle_recall(step.block_idx.cpu().numpy(), cnt.cpu().numpy(), dw.host.needles, s.block, s.num_kv_heads)
    nblk = np.array([-(-int(n) // s.block) for n in s.ctx_len for _ in range(s.num_kv_heads)])
    return {"selector": "top-delta", "delta": s.delta,
            "kept_fraction": float(cnt.cpu().numpy().sum() / nblk.sum()),
            "recall_top_delta": _stats(rec_d.cpu().numpy()),
            "matched_budget_blocks": k, "recall_quest_topk": _stats(rec_q.cpu().numpy()),
            "selector_time": times,
            "needle_recall_top_delta": _stats(nr) if nr.size else None}


def run(name: str, batch=None, ctx=None) -> dict:
    kw = {}
    if batch:
        kw["batch"] = batch
    if ctx:
        kw["ctx_len"] = ctx
    s = W.spec(name, **kw)
    dw = H.upload(s, W.generate(s))
    res = {"workload": name, "batch": s.batch, "ctx_len": int(s.ctx_len[0])}
    res.update(quest_quality(dw) if s.selector == "quest" else delta_vs_topk(dw))
    return res


def main():
    ap = argparse.ArgumentParser(description="selection-quality diagnostics")
    ap.add_argument("--workload", default="qwen1p5b", choices=W.CONFIG_NAMES)
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--ctx", type=int, default=None)
    a = ap.parse_args()
    print(json.dumps(run(a.workload, a.batch, a.ctx)))


if __name__ == "__main__":
    main()
