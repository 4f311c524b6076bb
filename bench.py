#!/usr/bin/env python3
"""Benchmark of one sparse decode step (select + attend + combine) on GB300.

Default workload: the Qwen2.5-1.5B-like layer, bf16, batch 32, 12 query /
2 KV heads, head_dim 128, 64k context, 16-token pages, 2048-token budget
(128 pages incl. the sink page and the last 64 tokens).  Synthetic seeded
inputs (no real KV cache exists here).

value = algorithmic bytes of the step (page min/max metadata of every page
+ K and V of the selected tokens) / device time per step, in GB/s.

The timed region replays CUDA graphs of up to 8 consecutive steps each (a
decode engine captures a whole iteration in one graph; consecutive step
kernels overlap launch and tail through programmatic dependent launch).
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
STEP_TRAFFIC_B32 = 4 * (50.475264e6 + 0.102912e6)
STEP_SOURCES = ("quest_step.cu", "attend_tma.cuh", "tma.cuh", "mma.cuh", "attend_common.cuh", "common.cuh")
STEP_SOURCES_SHA256 = "47e78991e4c5f32f831eb2f0adca24a306946651ca07f62fdb6ea567eb81491a"


def step_traffic(s: W.Spec):
    """Per-launch DRAM bytes of the step kernel for the captured workload, else None."""
    import hashlib
    if (s.name, s.batch, s.ctx_len[0]) != ("qwen1p5b", 32, 65536):
        return None
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "sparse_long_context_gb300", "csrc")
    h = hashlib.sha256()
    for f in STEP_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return round(STEP_TRAFFIC_B32) if h.hexdigest() == STEP_SOURCES_SHA256 else None


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


def parity_check(s: W.Spec, host, sel, out):
    """Sampled rows of the benchmarked step against the oracle (part of the
    CPU-baseline leg).  Raises if a row disagrees."""
    from tests import parity as PT
    res = {"rows": [0, s.rows - 1], "ties": 0, "max_abs": 0.0, "rel_l2": 0.0}
    for r in res["rows"]:
        b, h = divmod(r, s.num_kv_heads)
        orc = PT.oracle_row(s, host, b, h)
        t = PT.check_quest_list(sel[r], orc, int(host.ctx_len[b]), s.page_size, s.k_pages)
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
    return (f"{s.name}: B={s.batch} Hq={s.num_q_heads} Hkv={s.num_kv_heads} D={s.head_dim} "
            f"ctx={s.ctx_len[0]} P={s.page_size} budget={s.k_pages * s.page_size} tokens {s.dtype}")


# ---------------------------------------------------------------------- ours

def run_ours(args, s: W.Spec):
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
    first_sel, _, first_out, _ = H.run_step(dw)

    # buffer sets: distinct copies of cache + metadata
    sets = [(dw.K, dw.V, dw.kmin, dw.kmax)]
    for _ in range(nsets - 1):
        sets.append(tuple(t.clone() for t in sets[0]))
    steps_obj = [ops.QuestDecode(dw.desc, s.k_pages, s.n_sink_pages, s.n_local_tokens, args.splits)
                 for _ in sets]
    S = steps_obj[0].S
    stream = torch.cuda.Stream()
    graphs = []
    with torch.cuda.stream(stream):
        for st, (K, V, kmin, kmax) in zip(steps_obj, sets):
            st(dw.q, K, V, kmin, kmax, dw.ctx)  # warm the kernels before capture
        torch.cuda.synchronize()
        for st, (K, V, kmin, kmax) in zip(steps_obj, sets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                st(dw.q, K, V, kmin, kmax, dw.ctx)
            graphs.append(g)
        # the timed loop's graphs: `spg` consecutive steps each (global step i
        # uses buffer set i % nsets, continuing across graphs), as a decode
        # engine captures a whole iteration; consecutive kernels overlap
        # their launch with the previous one's tail (programmatic launch)
        spg = next(r for r in (8, 4, 2, 1) if args.steps % r == 0)
        mgraphs = []
        for gi in range(nsets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for j in range(spg):
                    u = (gi * spg + j) % nsets
                    K, V, kmin, kmax = sets[u]
                    steps_obj[u](dw.q, K, V, kmin, kmax, dw.ctx)
            mgraphs.append(g)
    torch.cuda.synchronize()
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
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(args.steps // spg):
            mgraphs[i % nsets].replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    w1 = time.time()
    clocks.window(w0, w1)
    elapsed = e0.elapsed_time(e1) / 1e3
    timed_rows = ops.get_stats(reset=True)  # rows the one-launch step handled off its fast path
    t_max, total_bytes = aggregate(elapsed, float(nbytes["total"] * args.steps), world)

    # per-replay spread: events around single replays (a separate pass, so the
    # timed loop above has no events inside it)
    nrep = max(200, min(args.steps, 1000))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nrep)]
    with torch.cuda.stream(stream):
        for i, (a, b_) in enumerate(evs):
            if i % 100 == 0:
                torch.cuda._sleep(int(2e7))  # keeps the queue ahead of the device
            a.record(stream)
            graphs[i % nsets].replay()
            b_.record(stream)
    torch.cuda.synchronize()
    per_rep = sorted(1e3 * a.elapsed_time(b_) for a, b_ in evs)
    rep_us = {"p10": round(per_rep[nrep // 10], 2), "p50": round(per_rep[nrep // 2], 2),
              "p90": round(per_rep[nrep * 9 // 10], 2), "replays": nrep}

    # dense decode on the same workload (the sparsity gate forced open: every
    # row attends its whole context through the same kernel), for the
    # speedup of the sparse step and dense GB/s against the peak
    dense = None
    if not args.no_dense and steps_obj[0].one_launch and ops.quest_step_splits(dw.desc, s.k_pages) > 0:
        dsteps = [ops.QuestDecode(dw.desc, s.k_pages, s.n_sink_pages, s.n_local_tokens, args.splits,
                                  min_sparsity=1e9) for _ in sets]
        dgraphs = []
        with torch.cuda.stream(stream):
            for st, (K, V, kmin, kmax) in zip(dsteps, sets):
                st(dw.q, K, V, kmin, kmax, dw.ctx)
            torch.cuda.synchronize()
            for st, (K, V, kmin, kmax) in zip(dsteps, sets):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    st(dw.q, K, V, kmin, kmax, dw.ctx)
                dgraphs.append(g)
            for i in range(3):
                dgraphs[i % nsets].replay()
            torch.cuda.synchronize()
            nd = max(20, min(args.steps, 200))
            d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            d0.record(stream)
            for i in range(nd):
                dgraphs[i % nsets].replay()
            d1.record(stream)
        torch.cuda.synchronize()
        dense_s = d0.elapsed_time(d1) / 1e3 / nd
        dense_bytes = sum(s.num_kv_heads * n * 2 * s.head_dim * 2 for n in s.ctx_len)
        dense = {"us_per_step": round(dense_s * 1e6, 2), "GB/s": round(dense_bytes / dense_s / 1e9, 1),
                 "frac_of_peak": None, "bytes_per_step": int(dense_bytes), "steps": nd}
        del dgraphs, dsteps

    # per-kernel device time: eager launches bracketed by events on the
    # launching stream, queued behind a sleep so the host stays ahead
    ksteps = max(50, min(args.steps, 400))
    one = steps_obj[0].one_launch and ops.quest_step_splits(dw.desc, s.k_pages) > 0
    ev = {k: ([], []) for k in (("step",) if one else ()) + ("select", "attend")}
    with torch.cuda.stream(stream):
        for i in range(ksteps):
            if i % 25 == 0:
                torch.cuda._sleep(int(4e7))  # keeps the queue ahead of the device
            st = steps_obj[i % nsets]
            K, V, kmin, kmax = sets[i % nsets]
            stages = [("select", lambda: st.select(dw.q, kmin, kmax, dw.ctx)),
                      ("attend", lambda: st.attend(dw.q, K, V, dw.ctx))]
            if one:
                stages.insert(0, ("step", lambda: st(dw.q, K, V, kmin, kmax, dw.ctx)))
            for name, fn in stages:
                a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b_.record(stream)
                ev[name][0].append(a)
                ev[name][1].append(b_)
    torch.cuda.synchronize()
    kern_us = {k: 1e3 * statistics.mean(a.elapsed_time(b_) for a, b_ in zip(*v)) for k, v in ev.items()}
    clk = clocks.stop()

    # end to end through the public API with host buffers
    q_host = dw.q.cpu().pin_memory()
    out_host = torch.empty(steps_obj[0].out.shape, dtype=steps_obj[0].out.dtype).pin_memory()
    q_dev = torch.empty_like(dw.q)
    esteps = max(10, min(args.steps, 300))
    for i in range(3):
        K, V, kmin, kmax = sets[i % nsets]
        steps_obj[i % nsets](q_dev, K, V, kmin, kmax, dw.ctx)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for i in range(esteps):
        K, V, kmin, kmax = sets[i % nsets]
        q_dev.copy_(q_host, non_blocking=True)
        o, _ = steps_obj[i % nsets](q_dev, K, V, kmin, kmax, dw.ctx)
        out_host.copy_(o, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    e2e_t = time.perf_counter() - t0
    e2e_eager_max, _ = aggregate(e2e_t, float(nbytes["total"] * esteps), world)
    # the same steps as a decode loop runs them: one graph per buffer set
    # holding the copy of q from pinned host memory, the step and the copy of
    # the output back, replayed and synchronised every step
    egraphs = []
    with torch.cuda.stream(stream):
        for u, (K, V, kmin, kmax) in enumerate(sets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                q_dev.copy_(q_host, non_blocking=True)
                o, _ = steps_obj[u](q_dev, K, V, kmin, kmax, dw.ctx)
                out_host.copy_(o, non_blocking=True)
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
    e2e_max, e2e_bytes = aggregate(e2e_t, float(nbytes["total"] * esteps), world)
    del egraphs

    # multi-step decode from CUDA graphs: each replay appends one token per
    # sequence (cache row + page min/max) and runs the step on the longer
    # context.  One loop per buffer set, each with its own ctx_len rewound by
    # `per` tokens, replayed in rotation so consecutive replays do not share
    # L2.
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
        ctx_end = [int(c) for c in loops[0].dw.ctx.cpu()]
        loop_rec = {"us_per_step": round(loop_s * 1e6, 2), "tokens_per_s": round(s.batch / loop_s, 1),
                    "steps": nloop, "launches_per_step": 2,
                    "what": "graph replay of decode_append (k/v row + page min/max, ctx_len += 1) "
                            "then the one-launch step",
                    "ctx_after": ctx_end[:4]}
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
    # dominant kernel: the one-launch step (all bytes of the step), else the
    # larger of the two stages by algorithmic bytes
    if one:
        dom, dom_bytes, dom_name = "step", nbytes["total"], "quest_step_kernel (score + top-k + attend + combine)"
    else:
        dom = "select" if nbytes["select"] >= nbytes["attend"] else "attend"
        dom_bytes = nbytes[dom]
        dom_name = ("select: quest_score_kernel + topk_kernel" if dom == "select"
                    else "attend: attend_tma_kernel with the cluster combine")
    if one:
        # the step is this one kernel: its average launch over the timed region
        achieved = dom_bytes / (t_max / args.steps) / 1e9
    else:
        achieved = dom_bytes / (kern_us[dom] * 1e-6) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "us_per_step": round(1e3 * ms_step, 2), "tokens_per_s": round(s.batch * world / (ms_step / 1e3), 1),
        "frac_of_peak": round(value / peak, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded numpy, see workloads.py)",
        "config": {"workload": _workload_name(s), "batch": s.batch, "ctx_len": s.ctx_len[0],
                   "seq_len": s.ctx_len[0], "page_size": s.page_size, "budget_tokens": s.k_pages * s.page_size,
                   "num_splits": ops.quest_step_splits(dw.desc, s.k_pages) if one else S,
                   "launches_per_step": 1 if one else 3, "buffer_sets": nsets, "steps_per_graph": spg,
                   "l2": f"inputs rotate over {nsets} buffer sets ({nsets * nbytes['total'] / 1e6:.0f} MB >= 4x L2 {l2 / 1e6:.0f} MB)",
                   "parallelism": f"weak: {world} GPU(s), {s.batch} sequences each"},
        "bytes_per_step": nbytes["total"], "bytes_select": nbytes["select"], "bytes_attend": nbytes["attend"],
        "kernel_us": {k: round(v, 2) for k, v in kern_us.items()},
        "replay_us": rep_us,
        "roofline": {"bound": "hbm", "kernel": dom_name,
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": step_traffic(s) if one else None,
                     "peak_kind": f"{peak_kind} (burst copy)"},
        "step_roofline": {"achieved": round(value, 1), "peak": peak, "frac": round(value / peak, 4)},
        "dense": dense,
        "decode_loop": loop_rec,
        "speedup_vs_dense": round(dense["us_per_step"] / (1e6 * t_max / args.steps), 2) if dense else None,
        "gpu_launches": (1 if one else 3) * args.steps,  # one step kernel, or score, top-k, attend
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
    """The top-delta step on the FFD workload, with the exact-key attend and
    with the refined (2-bit + 8-bit residual) attend."""
    import torch
    from sparse_long_context_gb300 import _lib
    from sparse_long_context_gb300 import harness as H
    from sparse_long_context_gb300 import ops

    torch.cuda.set_device(0)
    _lib.load()
    host = W.generate(s)
    dw = H.upload(s, host)
    codes, scales, res = ops.thumb_residual_build(dw.desc, dw.K, dw.ctx, s.block)
    exact = ops.DeltaDecode(dw.desc, s.block, s.delta, args.splits)
    refined = ops.DeltaDecode(dw.desc, s.block, s.delta, args.splits, refined=True)
    stream = torch.cuda.Stream()
    spg = next(r for r in (8, 4, 2, 1) if args.steps % r == 0)
    graphs = {}
    with torch.cuda.stream(stream):
        exact(dw.q, dw.K, dw.V, codes, scales, dw.ctx, dw.sink)
        refined(dw.q, dw.K, dw.V, codes, scales, dw.ctx, dw.sink, res=res)
        torch.cuda.synchronize()
        for name, st in (("exact", exact), ("refined", refined)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(spg):
                    st(dw.q, dw.K, dw.V, codes, scales, dw.ctx, dw.sink, res=res)
            graphs[name] = g
    ops.pipeline_check()
    nb = delta_bytes(s, host.ctx_len, refined.count.cpu().numpy(), refined.block_idx.cpu().numpy())
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    us = {}
    with torch.cuda.stream(stream):
        for name, g in graphs.items():
            for _ in range(-(-args.warmup // spg)):
                g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps // spg):
                g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            us[name] = 1e3 * e0.elapsed_time(e1) / args.steps
        # per-stage device time, eager launches between events
        ev = {k: [] for k in ("select", "attend_exact", "attend_refined")}
        for i in range(50):
            if i % 10 == 0:
                torch.cuda._sleep(int(2e7))
            for name, fn in (("select", lambda: refined.select(dw.q, dw.K, codes, scales, dw.ctx)),
                             ("attend_exact", lambda: exact.attend(dw.q, dw.K, dw.V, dw.ctx, dw.sink)),
                             ("attend_refined", lambda: refined.attend_refined(dw.q, dw.K, dw.V, codes, scales,
                                                                               res, dw.ctx, dw.sink))):
                a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b_.record(stream)
                ev[name].append((a, b_))
    torch.cuda.synchronize()
    ops.pipeline_check()
    clk = clocks.stop()
    kus = {k: 1e3 * statistics.mean(a.elapsed_time(b_) for a, b_ in v) for k, v in ev.items()}
    peak, peak_kind = load_peaks()
    tot_ref = nb["scan"] + nb["attend_refined"]
    value = tot_ref / (us["refined"] * 1e-6) / 1e9
    achieved = nb["attend_refined"] / (kus["attend_refined"] * 1e-6) / 1e9
    kept = int(refined.count.sum().item())
    nblk = sum(-(-n // s.block) for n in s.ctx_len) * s.num_kv_heads
    line = {
        "metric": "top-delta decode step us and achieved HBM GB/s, refined attend", "value": round(value, 2),
        "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(us["refined"] / 1e3, 5), "us_per_step": round(us["refined"], 2),
        "us_per_step_exact_attend": round(us["exact"], 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded numpy, see workloads.py)",
        "config": {"workload": f"{s.name}: B={s.batch} Hq={s.num_q_heads} Hkv={s.num_kv_heads} D={s.head_dim} "
                               f"ctx={s.ctx_len[0]} block={s.block} delta={s.delta} bf16",
                   "kept_blocks": kept, "kept_fraction": round(kept / nblk, 4), "steps_per_graph": spg,
                   "l2": f"one buffer set of {(tot_ref) / 1e6:.0f} MB per step (> L2)"},
        "bytes_per_step": tot_ref, "bytes": nb,
        "kernel_us": {k: round(v, 2) for k, v in kus.items()},
        "roofline": {"bound": "hbm", "kernel": "attend_refined_kernel (combine fused)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": None, "peak_kind": f"{peak_kind} (burst copy)"},
        "gpu_launches": 3 * args.steps,  # delta scan, compaction, refined attend
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="qwen1p5b", choices=("qwen1p5b", "qwen7b", "ffd"),
                    help="ffd: the top-delta step with exact and refined attends (a study line)")
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
