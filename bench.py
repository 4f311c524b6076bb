#!/usr/bin/env python3
"""Benchmark of one sparse decode step (select + attend + combine) on GB300.

Default workload: the Qwen2.5-1.5B-like layer, bf16, batch 32, 12 query /
2 KV heads, head_dim 128, 64k context, 16-token pages, 2048-token budget
(128 pages incl. the sink page and the last 64 tokens).  Synthetic seeded
inputs (no real KV cache exists here).

value = algorithmic bytes of the step (page min/max metadata of every page
+ K and V of the selected tokens) / device time per step, in GB/s.

The timed region replays CUDA graphs of up to 32 consecutive steps each (a
decode engine captures a whole iteration over the model's layers in one
graph; consecutive step kernels overlap launch and tail through
programmatic dependent launch).
NSETS copies of the KV cache and metadata rotate, step i using set
i % NSETS, so that consecutive steps never find their bytes in L2
(NSETS * step bytes >= 4 * L2).  `replay_us` times graphs of one step.  `python bench.py --impl
reference` times the fp64 CPU oracle on the same workload instead.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_long_context_gb300 import workloads as W  # noqa: E402

METRIC = "decode-step µs and achieved HBM GB/s (% of GB300 peak) for select+attend"

# DRAM bytes per launch of the one-launch step kernel, from the committed ncu
# capture (profiles/quest_step_qwen1p5b_64k_b8_full.md: batch 8 at 64k, read +
# written; traffic grows with the rows, so x4 for batch 32).  Reported only
# for that workload and only while the kernel's sources hash to the ones
# captured; otherwise null.
STEP_TRAFFIC_B32 = 4 * (50.470656e6 + 0.101632e6)
STEP_SOURCES = ("quest_step.cu", "attend_tma.cuh", "tma.cuh", "mma.cuh", "attend_common.cuh", "common.cuh",
                "status.cuh")
STEP_SOURCES_SHA256 = "a55d7811c3f7b3e114d0b70d4b5f02d64f96135c2122dd7d5d16c9577bbe5bfd"


# DRAM bytes per launch of the top-delta step's bf16-key attend
# (attend_stream_tma_kernel) on the ffd workload, from the committed capture
# (profiles/topdelta_ffd_256k.md, read + written; the kept set is the seeded
# workload's), under the same source-hash rule.
FFD_ATTEND_TRAFFIC = 490.973696e6 + 3.187712e6
FFD_ATTEND_SOURCES = ('attend_refined.cu', 'attend_tma.cuh', 'tma.cuh', 'mma.cuh', 'attend_common.cuh', 'common.cuh', 'status.cuh')
FFD_ATTEND_SOURCES_SHA256 = "9717fadbd32d4e7cecc3dc4e33e65abd9b13a93053d2b4e02423068159baf6e6"


def sources_sha256(files) -> str:
    import hashlib
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "sparse_long_context_gb300", "csrc")
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def ffd_attend_traffic(s: W.Spec):
    """Per-launch DRAM bytes of the ffd attend for the captured workload, else None."""
    if (s.name, s.batch, s.ctx_len[0]) != ("ffd", 2, 262144):
        return None
    return round(FFD_ATTEND_TRAFFIC) if sources_sha256(FFD_ATTEND_SOURCES) == FFD_ATTEND_SOURCES_SHA256 else None


def step_traffic(s: W.Spec):
    """Per-launch DRAM bytes of the step kernel for the captured workload, else None."""
    if (s.name, s.batch, s.ctx_len[0]) != ("qwen1p5b", 32, 65536):
        return None
    return round(STEP_TRAFFIC_B32) if sources_sha256(STEP_SOURCES) == STEP_SOURCES_SHA256 else None


# ------------------------------------------------------------------ helpers

def algorithmic_bytes(s: W.Spec, kept_blocks_total: int = 0) -> dict:
    """Bytes the step must read: selector metadata + selected K and V."""
    esz = 2 if s.dtype == "bf16" else 4
    rows = s.rows
    if s.selector == "quest":
        meta = 0
        sel_tokens = 0
        for b in range(s.batch):
            n = s.ctx_len[b]
            npg = -(-n // s.page_size)
            per_page = (1 if s.page_size == 1 else 2) * s.head_dim * esz
            meta += s.num_kv_heads * npg * per_page
            sel_tokens += s.num_kv_heads * min(npg, s.k_pages) * s.page_size
        kv = sel_tokens * 2 * s.head_dim * esz
    else:
        meta = 0
        for b in range(s.batch):
            n = s.ctx_len[b]
            nfull = n // s.block
            meta += s.num_kv_heads * (nfull * s.block * s.head_dim // 4 + nfull * s.head_dim * esz)
            meta += s.num_kv_heads * min(n, 2 * s.block) * s.head_dim * esz  # pseudo-max keys
        kv = kept_blocks_total * s.block * 2 * s.head_dim * esz
    return {"select": int(meta), "attend": int(kv), "total": int(meta + kv), "rows": rows}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        self.gpu = gpu_index
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def window(self, t0, t1):
        self.t0, self.t1 = t0, t1

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
                except ValueError:
                    continue
        os.unlink(self.path)
        inwin = [r for r in rows if self.t0 is not None and self.t0 - 1 <= r[0] <= self.t1 + 1]
        use = inwin or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use),
                "window": "timed" if inwin else "run"}


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def aggregate(elapsed_s: float, units: float, world: int):
    """Max time and summed units over ranks (identity on one process)."""
    if world == 1:
        return elapsed_s, units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ---------------------------------------------------------------- CPU oracle

def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.TimeoutExpired):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def cpu_oracle(s: W.Spec, host, rows, threads: int, min_busy: float = 0.0, refined: bool = False):
    """The C++ fp64 oracle's decode step over the listed (b, h) rows of the
    host workload on `threads` std::threads, each row repeated until it has
    run `min_busy` seconds (its page summaries or thumbnails are prepared
    before the timed part).  Returns (GB/s, threads, wall s, bytes,
    repetitions); wall = the rows' summed busy time / threads."""
    from oracle import sls_oracle as O
    ids = [b * s.num_kv_heads + h for b, h in rows]
    if s.selector == "quest":
        *_, busy, nbytes, reps = O.quest_step(host.q, host.K, host.V, host.ctx_len, s.num_q_heads, s.page_size,
                                              s.k_pages, s.n_sink_pages, s.n_local_tokens, s.scale, host.sink, ids,
                                              threads=threads, min_busy=min_busy)
    else:
        *_, busy, nbytes, reps = O.delta_step(host.q, host.K, host.V, host.ctx_len, s.num_q_heads, s.block,
                                              s.delta, s.scale, host.sink, ids, refined=refined, threads=threads,
                                              min_busy=min_busy)
    wall = busy / max(threads, 1)
    return nbytes / wall / 1e9, threads, wall, nbytes, reps


def parity_rows(s: W.Spec, count: int = 4):
    """Rows of the benchmarked step that the CPU-baseline leg checks: the
    first, the last and seeded others."""
    rng = np.random.default_rng(s.seed)
    rows = {0, s.rows - 1} | {int(r) for r in rng.integers(0, s.rows, size=count)}
    return sorted(rows)[:count + 2]


def parity_check(s: W.Spec, host, sel, out, count=None):
    """Sampled rows of the benchmarked step against the oracle (part of the
    CPU-baseline leg).  Raises if a row disagrees; returns the rows, the
    boundary ties counted and the largest output errors."""
    from tests import parity as PT
    res = {"rows": parity_rows(s), "ties": 0, "max_abs": 0.0, "rel_l2": 0.0}
    for r in res["rows"]:
        b, h = divmod(r, s.num_kv_heads)
        orc = PT.oracle_row(s, host, b, h)
        if s.selector == "quest":
            t = PT.check_quest_list(sel[r], orc, int(host.ctx_len[b]), s.page_size, s.k_pages)
        else:
            t = PT.check_delta_list(int(count[r]), sel[r], orc, s.delta)
        res["ties"] += t
        if t == 0:
            mx, rel = PT.assert_close(s, out[b, h * s.group:(h + 1) * s.group], orc.o, f"row {r}")
            res["max_abs"] = max(res["max_abs"], mx)
            res["rel_l2"] = max(res["rel_l2"], rel)
    return res


# ----------------------------------------------------------------- reference

def run_reference(args, s: W.Spec):
    """The C++ fp64 oracle as the reference arm, on one host core."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    # each step: one (b, kv head) row of the workload on one core, its page
    # summaries (or thumbnails) prepared outside the timed part; rows whose
    # whole context would take too long are cut to their first `pl` pages so
    # that warmup + steps finish within about two minutes
    total = args.steps + args.warmup
    per_step = 90.0 / max(total, 1)
    full_pages = -(-s.ctx_len[0] // s.page_size)
    est_per_page = 2e-6 if s.selector == "quest" else 40e-6  # seconds per page or block (prep + step)
    pl = int(min(full_pages, max(s.k_pages + 8, per_step / est_per_page)))
    n_cut = min(s.ctx_len[0], pl * s.page_size)
    host = W.generate(s, rows=[(i % s.batch, (i // s.batch) % s.num_kv_heads) for i in range(min(total, s.rows))])
    host.ctx_len = np.minimum(host.ctx_len, n_cut).astype(np.int32)
    times, nbytes = [], []
    for i in range(total):
        r = i % min(total, s.rows)
        b, h = r % s.batch, (r // s.batch) % s.num_kv_heads
        _, _, wall, nb, _ = cpu_oracle(s, host, [(b, h)], threads=1)
        if i >= args.warmup:
            times.append(wall)
            nbytes.append(nb)
    t = sum(times)
    value = sum(nbytes) / t / 1e9
    sample = (f"one (b, kv head) row per step, first {pl} of {full_pages} pages, fp64 C++ oracle, "
              f"1 thread on {cpu_model()} ({os.cpu_count()} cores)")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * t / max(len(times), 1), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": _workload_name(s), "batch": s.batch, "ctx_len": s.ctx_len[0],
                   "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _workload_name(s: W.Spec) -> str:
    base = f"{s.name}: B={s.batch} Hq={s.num_q_heads} Hkv={s.num_kv_heads} D={s.head_dim} ctx={s.ctx_len[0]}"
    if s.selector == "quest":
        return f"{base} P={s.page_size} budget={s.k_pages * s.page_size} tokens{' sink' if s.has_sink else ''} {s.dtype}"
    return f"{base} block={s.block} delta={s.delta} {s.dtype}"


# ---------------------------------------------------------------------- ours

NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e nominal bandwidth, for context beside the measured peak


def make_sets(dw, nsets: int):
    """`nsets` distinct copies of the cache and the selector metadata (the
    first is the workload's own).  A one-token page is its own summary, so
    with page_size 1 each set passes its key cache as kmin and kmax."""
    s = dw.spec
    sets = [(dw.K, dw.V, dw.kmin, dw.kmax)]
    for _ in range(nsets - 1):
        K, V = dw.K.clone(), dw.V.clone()
        if s.page_size == 1:
            kmin = kmax = K
        else:
            kmin, kmax = dw.kmin.clone(), dw.kmax.clone()
        sets.append((K, V, kmin, kmax))
    return sets


def steps_per_graph(steps: int) -> int:
    """Consecutive steps captured in one timed graph: the largest divisor of
    `steps` up to 32 (a decode engine replays one graph per iteration over a
    model's layers, each layer one step)."""
    return next(r for r in range(min(32, steps), 0, -1) if steps % r == 0)


def timed_windows(stream, graphs, steps: int, spg: int, world: int, min_total_s: float = 0.2,
                  max_windows: int = 200):
    """Time windows of exactly `steps` steps each (graph i replays steps
    spg*i .. spg*i + spg - 1, buffer sets rotating across graphs), each
    bracketed by a synchronise (and a barrier on several ranks) and CUDA
    events on the launching stream, repeated until `min_total_s` seconds of
    device time have been timed (at least 3 windows).  Returns the windows'
    seconds, each the max over ranks."""
    import torch
    import torch.distributed as dist
    out, gi = [], 0
    while len(out) < 3 or (sum(out) < min_total_s and len(out) < max_windows):
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps // spg):
                graphs[gi % len(graphs)].replay()
                gi += 1
            e1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t, _ = aggregate(e0.elapsed_time(e1) / 1e3, 0.0, world)
        out.append(t)
    return out


def window_stats(windows, steps: int) -> dict:
    us = sorted(1e6 * w / steps for w in windows)
    n = len(us)
    return {"windows": n, "steps_per_window": steps, "us_per_step_p10": round(us[n // 10], 3),
            "us_per_step_p50": round(statistics.median(us), 3), "us_per_step_p90": round(us[(n * 9) // 10], 3),
            "timed_s": round(sum(windows), 4)}


def roofline_block(kernel: str, achieved: float, peak: float, peak_kind: str, traffic, best_seen=None) -> dict:
    """The line's roofline object for the dominant kernel, with the
    fraction also against the best bandwidth this run saw and the nominal
    HBM bandwidth."""
    best = max(peak, best_seen or 0.0)
    return {"bound": "hbm", "kernel": kernel, "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "peak_kind": f"{peak_kind} (burst copy)",
            "frac_of_best_seen": round(achieved / best, 4), "best_seen_gbs": round(best, 1),
            "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4), "nominal_gbs": NOMINAL_HBM_GBS}


def capture_graphs(stream, sets, steps_obj, run, nsets: int, spg: int):
    """Single-step graphs (one per buffer set) and the timed loop's graphs
    of `spg` consecutive steps each (global step i uses set i % nsets,
    continuing across graphs).  run(step_obj, set) issues one step."""
    import torch
    with torch.cuda.stream(stream):
        for st, bufs in zip(steps_obj, sets):
            run(st, bufs)  # warm the kernels before capture
        torch.cuda.synchronize()
        single = []
        for st, bufs in zip(steps_obj, sets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                run(st, bufs)
            single.append(g)
        multi = []
        for gi in range(nsets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for j in range(spg):
                    u = (gi * spg + j) % nsets
                    run(steps_obj[u], sets[u])
            multi.append(g)
    torch.cuda.synchronize()
    return single, multi


def replay_spread(stream, graphs, steps: int) -> dict:
    """p10/p50/p90 of single graph replays, each bracketed by its own
    events (a separate pass: the timed windows have no events inside)."""
    import torch
    nrep = max(200, min(steps, 1000))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nrep)]
    with torch.cuda.stream(stream):
        for i, (a, b_) in enumerate(evs):
            if i % 100 == 0:
                torch.cuda._sleep(int(2e7))  # keeps the queue ahead of the device
            a.record(stream)
            graphs[i % len(graphs)].replay()
            b_.record(stream)
    torch.cuda.synchronize()
    per = sorted(1e3 * a.elapsed_time(b_) for a, b_ in evs)
    return {"p10": round(per[nrep // 10], 2), "p50": round(per[nrep // 2], 2), "p90": round(per[nrep * 9 // 10], 2),
            "replays": nrep}


def stage_times(stream, stages, reps: int) -> dict:
    """Mean device time of each named stage issued eagerly between events
    on the launching stream (queued behind a sleep so the host stays ahead)."""
    import torch
    ev = {k: [] for k, _ in stages[0]}
    with torch.cuda.stream(stream):
        for i in range(reps):
            if i % 25 == 0:
                torch.cuda._sleep(int(4e7))
            for name, fn in stages[i % len(stages)]:
                a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b_.record(stream)
                ev[name].append((a, b_))
    torch.cuda.synchronize()
    return {k: 1e3 * statistics.mean(a.elapsed_time(b_) for a, b_ in v) for k, v in ev.items()}


def run_ours(args, s: W.Spec):
    """The Quest step (qwen1p5b, qwen7b, gptoss, tiny) through the public API."""
    import torch
    import torch.distributed as dist
    from sparse_long_context_gb300 import _lib
    from sparse_long_context_gb300 import harness as H
    from sparse_long_context_gb300 import ops

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _lib.load()

    host = W.generate(s, batch_offset=rank * s.batch)
    dw = H.upload(s, host)
    nbytes = algorithmic_bytes(s)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    nsets = max(2, math.ceil(4 * l2 / nbytes["total"]))

    # one untimed step whose sampled rows the CPU-baseline leg checks
    first_sel, _, first_out, _ = H.run_step(dw, args.splits)

    sets = make_sets(dw, nsets)
    steps_obj = [ops.QuestDecode(dw.desc, s.k_pages, s.n_sink_pages, s.n_local_tokens, args.splits) for _ in sets]
    one = steps_obj[0].one_launch and ops.quest_step_splits(dw.desc, s.k_pages) > 0
    S = steps_obj[0].S
    stream = torch.cuda.Stream()
    spg = steps_per_graph(args.steps)

    def run(st, bufs):
        K, V, kmin, kmax = bufs
        return st(dw.q, K, V, kmin, kmax, dw.ctx, dw.sink)

    graphs, mgraphs = capture_graphs(stream, sets, steps_obj, run, nsets, spg)
    # kernels the library picked while the graphs were captured (the replays
    # make no host calls); the device-side row counters restart here
    paths_capture = {k: v for k, v in ops.get_stats(reset=True).items() if v}

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        for i in range(-(-args.warmup // spg)):
            mgraphs[i % nsets].replay()
    torch.cuda.synchronize()
    w0 = time.time()
    windows = timed_windows(stream, mgraphs, args.steps, spg, world)
    w1 = time.time()
    clocks.window(w0, w1)
    ops.pipeline_check()
    timed_rows = ops.get_stats(reset=True)  # rows the one-launch step handled off its fast path
    t_max = statistics.median(windows)
    total_bytes = nbytes["total"] * args.steps * world
    rep_us = replay_spread(stream, graphs, args.steps)

    # dense decode on the same workload (the sparsity gate forced open: every
    # row attends its whole context through the same kernel)
    dense = None
    if not args.no_dense and one:
        dsteps = [ops.QuestDecode(dw.desc, s.k_pages, s.n_sink_pages, s.n_local_tokens, args.splits,
                                  min_sparsity=1e9) for _ in sets]
        dgraphs, _ = capture_graphs(stream, sets, dsteps, run, nsets, 1)
        nd = max(20, min(args.steps, 200))
        with torch.cuda.stream(stream):
            for i in range(3):
                dgraphs[i % nsets].replay()
            torch.cuda.synchronize()
            d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            d0.record(stream)
            for i in range(nd):
                dgraphs[i % nsets].replay()
            d1.record(stream)
        torch.cuda.synchronize()
        dense_s = d0.elapsed_time(d1) / 1e3 / nd
        esz = 2 if s.dtype == "bf16" else 4
        dense_bytes = sum(s.num_kv_heads * n * 2 * s.head_dim * esz for n in s.ctx_len)
        dense = {"us_per_step": round(dense_s * 1e6, 2), "GB/s": round(dense_bytes / dense_s / 1e9, 1),
                 "frac_of_peak": None, "bytes_per_step": int(dense_bytes), "steps": nd}
        del dgraphs, dsteps

    # per-stage device time, eager launches between events
    def stages_for(i):
        st = steps_obj[i % nsets]
        K, V, kmin, kmax = sets[i % nsets]
        out = [("select", lambda: st.select(dw.q, kmin, kmax, dw.ctx)),
               ("attend", lambda: st.attend(dw.q, K, V, dw.ctx, dw.sink))]
        if one:
            out.insert(0, ("step", lambda: run(st, sets[i % nsets])))
        return out
    kern_us = stage_times(stream, [stages_for(i) for i in range(nsets)], max(50, min(args.steps, 400)))
    clk = clocks.stop()

    # end to end through the public API with host buffers: per step, the H2D
    # copy of q from pinned memory, the step and the D2H copy of the output,
    # issued eagerly, and as a decode loop runs them (one graph per buffer
    # set), each step followed by a host synchronise
    q_host = dw.q.cpu().pin_memory()
    out_host = torch.empty(steps_obj[0].out.shape, dtype=steps_obj[0].out.dtype).pin_memory()
    q_dev = torch.empty_like(dw.q)
    esteps = max(10, min(args.steps, 300))

    def e2e_step(u):
        K, V, kmin, kmax = sets[u]
        q_dev.copy_(q_host, non_blocking=True)
        o, _ = steps_obj[u](q_dev, K, V, kmin, kmax, dw.ctx, dw.sink)
        out_host.copy_(o, non_blocking=True)

    for i in range(3):
        e2e_step(i % nsets)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for i in range(esteps):
        e2e_step(i % nsets)
        torch.cuda.current_stream().synchronize()
    e2e_eager_max, _ = aggregate(time.perf_counter() - t0, 0.0, world)
    egraphs = []
    with torch.cuda.stream(stream):
        for u in range(nsets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                e2e_step(u)
            egraphs.append(g)
        for i in range(3):
            egraphs[i % nsets].replay()
        stream.synchronize()
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for i in range(esteps):
            egraphs[i % nsets].replay()
            stream.synchronize()
        e2e_t = time.perf_counter() - t0
    e2e_max, _ = aggregate(e2e_t, 0.0, world)
    e2e_bytes = nbytes["total"] * esteps * world
    del egraphs

    # multi-step decode from CUDA graphs: each replay appends one token per
    # sequence (cache row + page min/max) and runs the step on the longer
    # context; one loop per buffer set, each with its ctx_len rewound by `per`
    # tokens, replayed in rotation
    loop_rec = None
    if not args.no_loop and one:
        per, warm_tok = 64, 4
        loops = []
        with torch.cuda.stream(stream):
            for K, V, kmin, kmax in sets:
                ctx = (dw.ctx - per).clamp_min(0).to(torch.int32)
                lp = H.DecodeLoop(dataclasses.replace(dw, K=K, V=V, kmin=kmin, kmax=kmax, ctx=ctx), args.splits)
                lp.k_new.normal_()
                lp.v_new.normal_()
                lp.capture(stream)
                loops.append(lp)
            for _ in range(warm_tok):
                for lp in loops:
                    lp.graph.replay()
            torch.cuda.synchronize()
            l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            l0.record(stream)
            for _ in range(per - warm_tok):
                for lp in loops:
                    lp.graph.replay()
            l1.record(stream)
        ops.pipeline_check()
        nloop = (per - warm_tok) * len(loops)
        loop_s = l0.elapsed_time(l1) / 1e3 / nloop
        loop_rec = {"us_per_step": round(loop_s * 1e6, 2), "tokens_per_s": round(s.batch / loop_s, 1),
                    "steps": nloop, "launches_per_step": 2,
                    "what": "graph replay of decode_append (k/v row + page min/max, ctx_len += 1) "
                            "then the one-launch step",
                    "ctx_after": [int(c) for c in loops[0].dw.ctx.cpu()][:4]}
        del loops

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peak, peak_kind = load_peaks()
    if dense:
        dense["frac_of_peak"] = round(dense["GB/s"] / peak, 4)
    value = total_bytes / t_max / 1e9
    ms_step = 1e3 * t_max / args.steps
    wst = window_stats(windows, args.steps)
    # dominant kernel: the one-launch step (all bytes of the step), else the
    # larger of the two stages by algorithmic bytes
    if one:
        dom_name = "quest_step_kernel (score + top-k + attend + combine)"
        achieved = nbytes["total"] / (t_max / args.steps) / 1e9   # its average launch over the timed windows
        single = nbytes["total"] / (rep_us["p50"] * 1e-6) / 1e9
    else:
        dom = "select" if nbytes["select"] >= nbytes["attend"] else "attend"
        dom_name = ("select: quest_score_kernel + top-k kernel (two launches)" if dom == "select"
                    else "attend: split-K attend with the combine fused")
        achieved = nbytes[dom] / (kern_us[dom] * 1e-6) / 1e9
        single = None
    launches = 1 if one else 3
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "us_per_step": round(1e3 * ms_step, 2), "tokens_per_s": round(s.batch * world / (ms_step / 1e3), 1),
        "frac_of_peak": round(value / peak, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": s.dtype, "data": "synthetic (seeded numpy, see workloads.py)",
        "config": {"workload": _workload_name(s), "batch": s.batch, "ctx_len": s.ctx_len[0],
                   "seq_len": s.ctx_len[0], "page_size": s.page_size, "budget_tokens": s.k_pages * s.page_size,
                   "num_splits": ops.quest_step_splits(dw.desc, s.k_pages) if one else S,
                   "launches_per_step": launches, "buffer_sets": nsets, "steps_per_graph": spg,
                   "l2": f"inputs rotate over {nsets} buffer sets ({nsets * nbytes['total'] / 1e6:.0f} MB >= 4x L2 "
                         f"{l2 / 1e6:.0f} MB)",
                   "parallelism": f"weak: {world} GPU(s), {s.batch} sequences each"},
        "bytes_per_step": nbytes["total"], "bytes_select": nbytes["select"], "bytes_attend": nbytes["attend"],
        "timing": dict(wst, how="value and ms_per_step: the median window; each window times exactly `steps` "
                                "steps, repeated until >= 0.2 s of device time"),
        "kernel_us": {k: round(v, 2) for k, v in kern_us.items()},
        "replay_us": rep_us,
        "roofline": roofline_block(dom_name, achieved, peak, peak_kind, step_traffic(s) if one else None,
                                   dense["GB/s"] if dense else None),
        "step_roofline": {"achieved": round(value, 1), "peak": peak, "frac": round(value / peak, 4),
                          "single_step_graph_frac": None if single is None else round(single / peak, 4)},
        "dense": dense,
        "decode_loop": loop_rec,
        "speedup_vs_dense": round(dense["us_per_step"] / (1e3 * ms_step), 2) if dense else None,
        "gpu_launches": launches * args.steps,  # per timed window of `steps` steps
        "gpu_launches_all_windows": launches * args.steps * wst["windows"],
        "paths": {"at_capture": paths_capture,
                  "timed_rows_dense": timed_rows["step_rows_dense"],
                  "timed_rows_all_keys": timed_rows["step_rows_all_keys"]},
        "clocks": clk,
        "e2e": {"value": round(e2e_bytes / e2e_max / 1e9, 2), "unit": "GB/s",
                "us_per_step": round(1e6 * e2e_max / esteps, 2),
                "how": "per step: graph replay of H2D q (pinned) + step + D2H out, then a host synchronise",
                "us_per_step_eager_calls": round(1e6 * e2e_eager_max / esteps, 2),
                "h2d_bytes_per_step": int(q_host.numel() * q_host.element_size()),
                "d2h_bytes_per_step": int(out_host.numel() * out_host.element_size())},
    }
    if world == 1 and not args.no_cpu_baseline:
        line["parity"] = parity_check(s, host, first_sel, first_out)
        rows = [(b, h) for b in range(s.batch) for h in range(s.num_kv_heads)]
        ncore = os.cpu_count() or 1
        take = rows[:max(ncore, 1) * 4]
        # about 16 core-seconds: each row repeats until it has run 0.25 s
        gbs, cores, wall, nb, reps = cpu_oracle(s, host, take, threads=ncore, min_busy=0.25)
        line["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "cpu": cpu_model(),
                                "sample": f"{len(take)} of {s.rows} rows of one step (full rows), fp64 C++ oracle "
                                          f"on {cores} std::threads, {reps} row evaluations, {nb / 1e6:.0f} MB "
                                          f"in {wall:.1f} s ({wall * cores:.0f} core-s)"}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def delta_bytes(s: W.Spec, ctx, count, block_idx) -> dict:
    """Algorithmic bytes of one top-delta step: the scan (codes, scales, the
    pseudo-max keys) plus the kept blocks' keys and values, and the same
    with the refined attend, which reads codes + residuals + the block's
    scales instead of the bf16 key of every complete block."""
    D, esz, blk = s.head_dim, 2, s.block
    scan = algorithmic_bytes(s)["select"]
    kv_exact = kv_refined = 0
    for r in range(s.rows):
        n = int(ctx[r // s.num_kv_heads])
        nfull = n // blk
        for j in block_idx[r, :int(count[r])].tolist():
            ntok = max(0, min(blk, n - j * blk))
            kv_exact += ntok * 2 * D * esz
            if j < nfull:
                kv_refined += ntok * (D // 4 + D + D * esz) + D * esz
            else:
                kv_refined += ntok * 2 * D * esz
    return {"scan": int(scan), "attend_exact": int(kv_exact), "attend_refined": int(kv_refined)}


def run_delta(args, s: W.Spec):
    """The top-delta step on the FFD workload: select_delta, then attention
    over the kept blocks with the exact (bf16) keys, which is the workload's
    step; the refined (2-bit + 8-bit residual) attend is timed beside it."""
    import torch
    from sparse_long_context_gb300 import _lib
    from sparse_long_context_gb300 import harness as H
    from sparse_long_context_gb300 import ops

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    _lib.load()
    host = W.generate(s)
    dw = H.upload(s, host)
    codes, scales, res = ops.thumb_residual_build(dw.desc, dw.K, dw.ctx, s.block)
    first_sel, first_cnt, first_out, _ = H.run_step(dw, args.splits)
    probe = ops.DeltaDecode(dw.desc, s.block, s.delta, args.splits)
    probe.select(dw.q, dw.K, codes, scales, dw.ctx)
    nb = delta_bytes(s, host.ctx_len, probe.count.cpu().numpy(), probe.block_idx.cpu().numpy())
    tot_exact, tot_ref = nb["scan"] + nb["attend_exact"], nb["scan"] + nb["attend_refined"]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    nsets = max(2, math.ceil(4 * l2 / tot_ref))
    sets = [(dw.K, dw.V, codes, scales, res)] + [
        (dw.K.clone(), dw.V.clone(), codes.clone(), scales.clone(), res.clone()) for _ in range(nsets - 1)]
    exact = [ops.DeltaDecode(dw.desc, s.block, s.delta, args.splits) for _ in sets]
    refined = [ops.DeltaDecode(dw.desc, s.block, s.delta, args.splits, refined=True) for _ in sets]
    stream = torch.cuda.Stream()
    spg = steps_per_graph(args.steps)

    def run(st, bufs):
        K, V, c, sc, r = bufs
        return st(dw.q, K, V, c, sc, dw.ctx, dw.sink, res=r)

    g_exact, m_exact = capture_graphs(stream, sets, exact, run, nsets, spg)
    g_ref, m_ref = capture_graphs(stream, sets, refined, run, nsets, spg)
    paths_capture = {k: v for k, v in ops.get_stats(reset=True).items() if v}
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    res_t = {}
    w0 = time.time()
    for name, mg in (("exact", m_exact), ("refined", m_ref)):
        with torch.cuda.stream(stream):
            for i in range(-(-args.warmup // spg)):
                mg[i % nsets].replay()
        torch.cuda.synchronize()
        res_t[name] = timed_windows(stream, mg, args.steps, spg, 1)
    w1 = time.time()
    clocks.window(w0, w1)
    ops.pipeline_check()
    rep_us = replay_spread(stream, g_exact, args.steps)

    def stages_for(i):
        e, r = exact[i % nsets], refined[i % nsets]
        K, V, c, sc, rr = sets[i % nsets]
        return [("select", lambda: e.select(dw.q, K, c, sc, dw.ctx)),
                ("attend_exact", lambda: e.attend(dw.q, K, V, dw.ctx, dw.sink)),
                ("attend_refined", lambda: r.attend_refined(dw.q, K, V, c, sc, rr, dw.ctx, dw.sink))]
    for i in range(nsets):  # every set's lists, for the eager stages below
        exact[i].select(dw.q, sets[i][0], sets[i][2], sets[i][3], dw.ctx)
        refined[i].select(dw.q, sets[i][0], sets[i][2], sets[i][3], dw.ctx)
    kus = stage_times(stream, [stages_for(i) for i in range(nsets)], 60)
    ops.pipeline_check()
    clk = clocks.stop()

    # end to end: H2D q (pinned) + the step + D2H out, one graph per set,
    # each step followed by a host synchronise
    q_host = dw.q.cpu().pin_memory()
    out_host = torch.empty(exact[0].out.shape, dtype=exact[0].out.dtype).pin_memory()
    q_dev = torch.empty_like(dw.q)
    esteps = max(10, min(args.steps, 200))
    egraphs = []
    with torch.cuda.stream(stream):
        for u in range(nsets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                q_dev.copy_(q_host, non_blocking=True)
                K, V, c, sc, r = sets[u]
                o, _ = exact[u](q_dev, K, V, c, sc, dw.ctx, dw.sink)
                out_host.copy_(o, non_blocking=True)
            egraphs.append(g)
        for i in range(3):
            egraphs[i % nsets].replay()
        stream.synchronize()
        t0 = time.perf_counter()
        for i in range(esteps):
            egraphs[i % nsets].replay()
            stream.synchronize()
        e2e_t = time.perf_counter() - t0
    del egraphs

    peak, peak_kind = load_peaks()
    t_ex = statistics.median(res_t["exact"]) / args.steps
    t_rf = statistics.median(res_t["refined"]) / args.steps
    value = tot_exact / t_ex / 1e9
    kept = int(probe.count.sum().item())
    nblk = sum(-(-n // s.block) for n in s.ctx_len) * s.num_kv_heads
    dom = "attend_exact" if nb["attend_exact"] >= nb["scan"] else "select"
    achieved = nb[dom if dom != "select" else "scan"] / (kus[dom] * 1e-6) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_ex * 1e3, 5), "us_per_step": round(t_ex * 1e6, 2),
        "tokens_per_s": round(s.batch / t_ex, 1), "frac_of_peak": round(value / peak, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": s.dtype,
        "data": "synthetic (seeded numpy, see workloads.py)",
        "config": {"workload": _workload_name(s), "batch": s.batch, "ctx_len": s.ctx_len[0],
                   "kept_blocks": kept, "kept_fraction": round(kept / nblk, 4), "steps_per_graph": spg,
                   "launches_per_step": 3, "buffer_sets": nsets,
                   "l2": f"inputs rotate over {nsets} buffer sets ({nsets * tot_ref / 1e6:.0f} MB >= 4x L2 "
                         f"{l2 / 1e6:.0f} MB)"},
        "bytes_per_step": tot_exact, "bytes": nb,
        "timing": dict(window_stats(res_t["exact"], args.steps),
                       how="value and ms_per_step: the median window of the step with the exact attend"),
        "refined_step": {"us_per_step": round(t_rf * 1e6, 2), "bytes_per_step": tot_ref,
                         "GB/s": round(tot_ref / t_rf / 1e9, 1), "frac_of_peak": round(tot_ref / t_rf / 1e9 / peak, 4),
                         "timing": window_stats(res_t["refined"], args.steps)},
        "kernel_us": {k: round(v, 2) for k, v in kus.items()},
        "stage_GBs": {"select": round(nb["scan"] / (kus["select"] * 1e-6) / 1e9, 1),
                      "attend_exact": round(nb["attend_exact"] / (kus["attend_exact"] * 1e-6) / 1e9, 1),
                      "attend_refined": round(nb["attend_refined"] / (kus["attend_refined"] * 1e-6) / 1e9, 1)},
        "replay_us": rep_us,
        "roofline": roofline_block("attend_stream_tma_kernel (stream-K attend, bf16 keys, tensor-map fed, "
                                   "combine fused)" if dom == "attend_exact"
                                   else "delta_scan_mma_kernel + delta_compact_kernel",
                                   achieved, peak, peak_kind, ffd_attend_traffic(s) if dom == "attend_exact" else None),
        "step_roofline": {"achieved": round(value, 1), "peak": peak, "frac": round(value / peak, 4)},
        "gpu_launches": 3 * args.steps,  # scan, compaction, attend; per timed window of `steps` steps
        "paths": {"at_capture": paths_capture},
        "clocks": clk,
        "e2e": {"value": round(tot_exact * esteps / e2e_t / 1e9, 2), "unit": "GB/s",
                "us_per_step": round(1e6 * e2e_t / esteps, 2),
                "how": "per step: graph replay of H2D q (pinned) + step + D2H out, then a host synchronise",
                "h2d_bytes_per_step": int(q_host.numel() * q_host.element_size()),
                "d2h_bytes_per_step": int(out_host.numel() * out_host.element_size())},
    }
    # top-delta against Quest top-k at the same mean budget: recall and each
    # selector's own device time ("Faster Than Flash", selection-rule overhead)
    from sparse_long_context_gb300 import diagnostics as DG
    line["selection_comparison"] = DG.delta_vs_topk(dw)
    if not args.no_cpu_baseline:
        line["parity"] = parity_check(s, host, first_sel, first_out, first_cnt)
        rows = [(b, h) for b in range(s.batch) for h in range(s.num_kv_heads)]
        ncore = os.cpu_count() or 1
        gbs, cores, wall, nbo, reps = cpu_oracle(s, host, rows, threads=ncore, min_busy=0.25)
        line["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "cpu": cpu_model(),
                                "sample": f"all {len(rows)} rows of one step (exact attend), fp64 C++ oracle on "
                                          f"{cores} std::threads, {reps} row evaluations, {nbo / 1e6:.0f} MB in "
                                          f"{wall:.1f} s ({wall * cores:.0f} core-s)"}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="qwen1p5b", choices=W.CONFIG_NAMES,
                    help="qwen1p5b (default), qwen7b, gptoss, tiny: the Quest step; ffd: the top-delta step")
    ap.add_argument("--ctx", type=int, default=None, help="context length (default: the workload's)")
    ap.add_argument("--batch", type=int, default=None, help="sequences per GPU (default: the workload's)")
    ap.add_argument("--no-dense", action="store_true", help="skip the dense-decode comparison")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-loop", action="store_true", help="skip the multi-step decode-loop measurement")
    ap.add_argument("--splits", type=int, default=None,
                    help="attend splits per (sequence, KV head) (default: the library's choice)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    kw = {}
    if args.ctx:
        kw["ctx_len"] = args.ctx
    if args.batch:
        kw["batch"] = args.batch
    s = W.spec(args.workload, **kw)
    if args.impl == "reference":
        run_reference(args, s)
    elif s.selector != "quest":
        run_delta(args, s)
    else:
        run_ours(args, s)


if __name__ == "__main__":
    main()
