"""Moves a generated workload onto the GPU and builds the selector metadata
with the library's own kernels (used by the benchmark, the smoke check and
the tests)."""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from . import ops
from . import workloads as W


def to_device(arr: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """Host array (bf16 bit patterns as uint16, or fp32) -> CUDA tensor."""
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).to(device)


@dataclasses.dataclass
class DeviceWorkload:
    """A workload's tensors on the device with its descriptor and selector
    metadata (page min/max for Quest, thumbnails for top-delta)."""
    spec: W.Spec
    host: W.Tensors
    K: torch.Tensor
    V: torch.Tensor
    q: torch.Tensor
    ctx: torch.Tensor
    sink: object
    desc: object
    kmin: object = None
    kmax: object = None
    codes: object = None
    scales: object = None


def upload(spec: W.Spec, host: W.Tensors, cuda_cores: bool = False, device="cuda",
           no_tma: bool = False) -> DeviceWorkload:
    """Copies a generated workload to the device and builds its selector
    metadata through the library."""
    K = to_device(host.K, spec.dtype, device)
    V = to_device(host.V, spec.dtype, device)
    q = to_device(host.q, spec.dtype, device)
    ctx = torch.from_numpy(host.ctx_len).to(device)
    sink = torch.from_numpy(host.sink).to(device) if host.sink is not None else None
    desc = ops.make_desc(spec.batch, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                         spec.page_size, spec.capacity, K.dtype, cuda_cores=cuda_cores, no_tma=no_tma)
    dw = DeviceWorkload(spec, host, K, V, q, ctx, sink, desc)
    if spec.selector == "quest":
        if spec.page_size == 1:
            dw.kmin = dw.kmax = K
        else:
            dw.kmin, dw.kmax = ops.pagemeta_build(desc, K, ctx)
    else:
        dw.codes, dw.scales = ops.thumb_build(desc, K, ctx, spec.block)
    return dw


def make_step(dw: DeviceWorkload, num_splits=None, fused: bool = True, one_launch: bool = True):
    """The decode step object (QuestDecode or DeltaDecode) for a workload."""
    s = dw.spec
    if s.selector == "quest":
        return ops.QuestDecode(dw.desc, s.k_pages, s.n_sink_pages, s.n_local_tokens, num_splits,
                               fused=fused, one_launch=one_launch)
    return ops.DeltaDecode(dw.desc, s.block, s.delta, num_splits, fused=fused)


def run_step(dw: DeviceWorkload, num_splits=None, fused: bool = True, one_launch: bool = True):
    """Select + attend + combine on the device.  Returns host arrays:
    (selection rows, counts or None, out [B,Hq,D] float64, lse [B,Hq])."""
    s = dw.spec
    step = make_step(dw, num_splits, fused, one_launch)
    if s.selector == "quest":
        out, lse = step(dw.q, dw.K, dw.V, dw.kmin, dw.kmax, dw.ctx, dw.sink)
        sel, cnt = step.page_idx, None
    else:
        out, lse = step(dw.q, dw.K, dw.V, dw.codes, dw.scales, dw.ctx, dw.sink)
        sel, cnt = step.block_idx, step.count
    ops.pipeline_check()  # synchronises; raises if a pipelined kernel gave up waiting
    return (sel.cpu().numpy(), None if cnt is None else cnt.cpu().numpy(),
            out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64))


class DecodeLoop:
    """A multi-step decode loop resident on the device.  One step appends the
    new token's key and value at ctx_len (keeping the selector's summaries
    current: page min/max, or the thumbnail of a block the token completes),
    advances ctx_len, then runs select + attend + combine on the longer
    context.  capture() records one step in a CUDA graph; each replay decodes
    one more token with no host work.  The caller writes the step's q,
    k_new and v_new into the fixed buffers before a replay.  refined=True
    (top-delta only) keeps the 8-bit residuals current as well and attends
    with the refined keys; `res` is then the residual tensor matching
    dw.codes and dw.scales."""

    def __init__(self, dw: DeviceWorkload, num_splits=None, min_sparsity: float = 0.0, refined: bool = False,
                 res=None):
        s = dw.spec
        self.dw = dw
        self.refined = refined
        self.res = res
        if refined and (s.selector == "quest" or res is None):
            raise ValueError("the refined loop is a top-delta loop and needs the residuals")
        if s.selector == "quest":
            self.step = ops.QuestDecode(dw.desc, s.k_pages, s.n_sink_pages, s.n_local_tokens, num_splits,
                                        min_sparsity=min_sparsity)
        else:
            self.step = ops.DeltaDecode(dw.desc, s.block, s.delta, num_splits, refined=refined)
        dt = dw.K.dtype
        self.k_new = torch.zeros((s.batch, s.num_kv_heads, s.head_dim), dtype=dt, device=dw.K.device)
        self.v_new = torch.zeros_like(self.k_new)
        self.pos = torch.empty(s.batch, dtype=torch.int32, device=dw.K.device)
        self.graph = None

    def run_once(self):
        dw, s = self.dw, self.dw.spec
        if s.selector == "quest":
            meta = (dw.kmin, dw.kmax) if s.page_size > 1 else (None, None)
            ops.decode_append(dw.desc, self.k_new, self.v_new, dw.K, dw.V, dw.ctx, *meta, pos_out=self.pos)
            return self.step(dw.q, dw.K, dw.V, dw.kmin, dw.kmax, dw.ctx, dw.sink)
        ops.decode_append(dw.desc, self.k_new, self.v_new, dw.K, dw.V, dw.ctx, pos_out=self.pos)
        if self.refined:
            ops.thumb_residual_update(dw.desc, dw.K, self.pos, s.block, dw.codes, dw.scales, self.res)
            return self.step(dw.q, dw.K, dw.V, dw.codes, dw.scales, dw.ctx, dw.sink, res=self.res)
        ops.thumb_update(dw.desc, dw.K, self.pos, s.block, dw.codes, dw.scales)
        return self.step(dw.q, dw.K, dw.V, dw.codes, dw.scales, dw.ctx, dw.sink)

    def capture(self, stream=None):
        """Records one step (nothing runs until replay())."""
        stream = stream or torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=stream):
            self.out, self.lse = self.run_once()
        torch.cuda.current_stream().wait_stream(stream)
        return self.graph

    def replay(self):
        self.graph.replay()
        return self.out, self.lse
