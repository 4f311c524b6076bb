"""Python binding over the C ABI: turns torch CUDA tensors into the raw
pointers, sizes and stream the C calls take.  Every step of the path runs in
libsls.so kernels; this module only marshals arguments and, where asked,
allocates output tensors with torch (the C library itself allocates
nothing).
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _lib as L

_DTYPES = {torch.float32: L.SLS_DTYPE_F32, torch.bfloat16: L.SLS_DTYPE_BF16}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _need(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def make_desc(batch, num_q_heads, num_kv_heads, head_dim, page_size, capacity, dtype,
              scale: float = 0.0, cuda_cores: bool = False, no_tma: bool = False,
              test_wait_timeout: bool = False) -> L.AttnDesc:
    """Descriptor of one layer's decode shapes (the C ABI's sls_attn_desc); dtype is a torch dtype
    or an SLS_DTYPE_* code, scale 0 means 1/sqrt(head_dim).  test_wait_timeout sets the
    bounded-wait test hook (SLS_FLAG_TEST_WAIT_TIMEOUT; tests only)."""
    code = _DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    flags = ((L.SLS_FLAG_CUDA_CORES if cuda_cores else 0) | (L.SLS_FLAG_NO_TMA if no_tma else 0)
             | (L.SLS_FLAG_TEST_WAIT_TIMEOUT if test_wait_timeout else 0))
    return L.AttnDesc(batch, num_q_heads, num_kv_heads, head_dim, page_size, capacity, code,
                      flags, float(scale))


def get_stats(reset: bool = False) -> dict:
    """Counters of the paths the library took (synchronises the device)."""
    st = L.Stats()
    L.call("sls_get_stats", ctypes.byref(st), int(bool(reset)))
    return {name: int(getattr(st, name)) for name, _ in L.Stats._fields_}


def pipeline_check() -> None:
    """Synchronises the device and reads the device status words; raises
    SlsError with code SLS_ETIMEOUT if a pipelined kernel gave up waiting for
    its copies, or SLS_EDEVICE if a kernel met (and skipped) page-list entries
    that are neither a page of the pool nor -1, since the last check."""
    L.call("sls_pipeline_check")


def desc_for(k_cache: torch.Tensor, num_q_heads: int, page_size: int, scale: float = 0.0,
             cuda_cores: bool = False) -> L.AttnDesc:
    """Descriptor read off a [B, Hkv, Cap, D] key cache."""
    B, Hkv, Cap, D = k_cache.shape
    return make_desc(B, num_q_heads, Hkv, D, page_size, Cap, k_cache.dtype, scale, cuda_cores)


def default_splits(desc: L.AttnDesc, max_entries: int) -> int:
    """The library's split count: one wave of attend CTAs, >= 64 tokens each."""
    return int(L.load().sls_attend_default_splits(ctypes.byref(desc), int(max_entries)))


# ----------------------------------------------------------------- metadata

def pagemeta_build(desc: L.AttnDesc, k_cache, ctx_len, kmin=None, kmax=None):
    """Per-page min and max of the valid keys (sls_pagemeta_build); allocates
    kmin/kmax [B, Hkv, Cap/P, D] when not given.  Returns (kmin, kmax)."""
    _need(k_cache, "k_cache")
    _need(ctx_len, "ctx_len", torch.int32)
    B, Hkv, Cap, D = k_cache.shape
    shape = (B, Hkv, Cap // desc.page_size, D)
    kmin = torch.empty(shape, dtype=k_cache.dtype, device=k_cache.device) if kmin is None else kmin
    kmax = torch.empty(shape, dtype=k_cache.dtype, device=k_cache.device) if kmax is None else kmax
    _need(kmin, "kmin", k_cache.dtype, shape)
    _need(kmax, "kmax", k_cache.dtype, shape)
    L.call("sls_pagemeta_build", ctypes.byref(desc), _ptr(k_cache), _ptr(ctx_len), _ptr(kmin),
           _ptr(kmax), _stream())
    return kmin, kmax


def pagemeta_update(desc: L.AttnDesc, k_cache, pos, kmin, kmax):
    """Folds the key at pos[b] of every sequence into its page's min/max
    (sls_pagemeta_update)."""
    _need(pos, "pos", torch.int32)
    L.call("sls_pagemeta_update", ctypes.byref(desc), _ptr(k_cache), _ptr(pos), _ptr(kmin),
           _ptr(kmax), _stream())


def thumb_build(desc: L.AttnDesc, k_cache, ctx_len, block: int, codes=None, scales=None):
    """2-bit thumbnails of every complete block (sls_thumb_build); allocates
    codes [B, Hkv, Cap, D/4] u8 and scales [B, Hkv, Cap/block, D] when not given.
    Returns (codes, scales)."""
    _need(k_cache, "k_cache")
    _need(ctx_len, "ctx_len", torch.int32)
    B, Hkv, Cap, D = k_cache.shape
    if codes is None:
        codes = torch.zeros((B, Hkv, Cap, D // 4), dtype=torch.uint8, device=k_cache.device)
    if scales is None:
        scales = torch.zeros((B, Hkv, Cap // block, D), dtype=k_cache.dtype, device=k_cache.device)
    _need(codes, "codes", torch.uint8, (B, Hkv, Cap, D // 4))
    _need(scales, "scales", k_cache.dtype, (B, Hkv, Cap // block, D))
    L.call("sls_thumb_build", ctypes.byref(desc), _ptr(k_cache), _ptr(ctx_len), int(block),
           _ptr(codes), _ptr(scales), _stream())
    return codes, scales


def thumb_update(desc: L.AttnDesc, k_cache, pos, block: int, codes, scales):
    """Quantises the block that the key at pos[b] completes (sls_thumb_update)."""
    _need(pos, "pos", torch.int32)
    L.call("sls_thumb_update", ctypes.byref(desc), _ptr(k_cache), _ptr(pos), int(block),
           _ptr(codes), _ptr(scales), _stream())


def thumb_residual_build(desc: L.AttnDesc, k_cache, ctx_len, block: int, codes=None, scales=None, res=None):
    """Thumbnails plus 8-bit residuals of every complete block."""
    B, H, Cap, D = desc.batch, desc.num_kv_heads, desc.capacity, desc.head_dim
    dev = k_cache.device
    codes = torch.zeros((B, H, Cap, D // 4), dtype=torch.uint8, device=dev) if codes is None else codes
    scales = torch.zeros((B, H, Cap // block, D), dtype=k_cache.dtype, device=dev) if scales is None else scales
    res = torch.zeros((B, H, Cap, D), dtype=torch.int8, device=dev) if res is None else res
    L.call("sls_thumb_residual_build", ctypes.byref(desc), _ptr(k_cache), _ptr(ctx_len), int(block), _ptr(codes),
           _ptr(scales), _ptr(res), _stream())
    return codes, scales, res


def thumb_residual_update(desc: L.AttnDesc, k_cache, pos, block: int, codes, scales, res):
    """Thumbnail and 8-bit residuals of the block that the key at pos[b]
    completes (sls_thumb_residual_update)."""
    _need(pos, "pos", torch.int32)
    L.call("sls_thumb_residual_update", ctypes.byref(desc), _ptr(k_cache), _ptr(pos), int(block), _ptr(codes),
           _ptr(scales), _ptr(res), _stream())


# ---------------------------------------------------------------- selection

def select_pages_workspace(desc: L.AttnDesc, device="cuda"):
    """Scratch buffer of select_pages (sls_select_pages_workspace_size bytes)."""
    n = L.load().sls_select_pages_workspace_size(ctypes.byref(desc))
    return torch.empty(max(int(n), 1), dtype=torch.uint8, device=device)


def select_pages(desc: L.AttnDesc, q, kmin, kmax, ctx_len, k: int, n_sink_pages: int = 0,
                 n_local_tokens: int = 0, out=None, workspace=None):
    """Quest selection (sls_select_pages): per (sequence, KV head) the k pages
    with the highest min/max bound, forced sink and local pages included,
    ascending, -1 padded.  Returns page_idx [B*Hkv, k] int32."""
    _need(q, "q")
    rows = desc.batch * desc.num_kv_heads
    out = torch.empty((rows, k), dtype=torch.int32, device=q.device) if out is None else out
    _need(out, "page_idx", torch.int32, (rows, k))
    workspace = select_pages_workspace(desc, q.device) if workspace is None else workspace
    L.call("sls_select_pages", ctypes.byref(desc), _ptr(q), _ptr(kmin), _ptr(kmax), _ptr(ctx_len),
           int(k), int(n_sink_pages), int(n_local_tokens), _ptr(out), _ptr(workspace),
           workspace.numel(), _stream())
    return out


def select_delta_workspace(desc: L.AttnDesc, block: int, device="cuda"):
    """Scratch buffer of select_delta (sls_select_delta_workspace_size bytes)."""
    n = L.load().sls_select_delta_workspace_size(ctypes.byref(desc), int(block))
    return torch.empty(max(int(n), 1), dtype=torch.uint8, device=device)


def select_delta(desc: L.AttnDesc, q, k_cache, codes, scales, ctx_len, block: int, delta: float,
                 count=None, block_idx=None, workspace=None):
    """Top-delta selection (sls_select_delta): the blocks whose thumbnail
    scores come within delta of the pseudo-max, plus the first and newest
    block.  Returns (count [B*Hkv], block_idx [B*Hkv, Cap/block])."""
    rows = desc.batch * desc.num_kv_heads
    nblk = desc.capacity // block
    count = torch.empty(rows, dtype=torch.int32, device=q.device) if count is None else count
    block_idx = torch.empty((rows, nblk), dtype=torch.int32, device=q.device) if block_idx is None else block_idx
    workspace = select_delta_workspace(desc, block, q.device) if workspace is None else workspace
    _need(block_idx, "block_idx", torch.int32)
    L.call("sls_select_delta", ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(codes), _ptr(scales),
           _ptr(ctx_len), int(block), float(delta), _ptr(count), _ptr(block_idx),
           int(block_idx.shape[1]), _ptr(workspace), workspace.numel(), _stream())
    return count, block_idx


# ---------------------------------------------------------------- attention

def partials(desc: L.AttnDesc, num_splits: int, device="cuda"):
    """Split partials (o [B, Hq, S, D], m and l [B, Hq, S], fp32) for
    sparse_decode_attend and combine_splits."""
    B, Hq, D = desc.batch, desc.num_q_heads, desc.head_dim
    return (torch.empty((B, Hq, num_splits, D), dtype=torch.float32, device=device),
            torch.empty((B, Hq, num_splits), dtype=torch.float32, device=device),
            torch.empty((B, Hq, num_splits), dtype=torch.float32, device=device))


def sparse_decode_attend(desc: L.AttnDesc, q, k_cache, v_cache, page_idx, ctx_len, num_splits: int,
                         count=None, k_fixed: Optional[int] = None, parts=None):
    """page_idx [rows, stride] int32 (or None for every page); count [rows]
    int32 or None (then k_fixed, default stride, entries per row)."""
    _need(q, "q")
    _need(k_cache, "k_cache")
    _need(v_cache, "v_cache")
    o, m, l = partials(desc, num_splits, q.device) if parts is None else parts
    stride = int(page_idx.shape[1]) if page_idx is not None else 0
    kf = stride if k_fixed is None else int(k_fixed)
    L.call("sls_sparse_decode_attend", ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache),
           _ptr(page_idx), stride, _ptr(count), kf, _ptr(ctx_len), int(num_splits), _ptr(o),
           _ptr(m), _ptr(l), _stream())
    return o, m, l


def attend_combine_workspace(desc: L.AttnDesc, num_splits: int, device="cuda"):
    """Zero-filled workspace of sparse_decode_attend_combine (reusable)."""
    n = L.load().sls_attend_combine_workspace_size(ctypes.byref(desc), int(num_splits))
    return torch.zeros(max(int(n), 1), dtype=torch.uint8, device=device)


def sparse_decode_attend_combine(desc: L.AttnDesc, q, k_cache, v_cache, page_idx, ctx_len,
                                 num_splits: int, count=None, k_fixed: Optional[int] = None,
                                 sink=None, out=None, lse=None, workspace=None, want_lse: bool = True):
    """Attend and combine in one launch; returns (out, lse)."""
    _need(q, "q")
    _need(k_cache, "k_cache")
    _need(v_cache, "v_cache")
    B, Hq, D = desc.batch, desc.num_q_heads, desc.head_dim
    dtype = torch.bfloat16 if desc.dtype == L.SLS_DTYPE_BF16 else torch.float32
    out = torch.empty((B, Hq, D), dtype=dtype, device=q.device) if out is None else out
    if want_lse and lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if sink is not None:
        _need(sink, "sink", torch.float32, (Hq,))
    workspace = attend_combine_workspace(desc, num_splits, q.device) if workspace is None else workspace
    stride = int(page_idx.shape[1]) if page_idx is not None else 0
    kf = stride if k_fixed is None else int(k_fixed)
    L.call("sls_sparse_decode_attend_combine", ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache),
           _ptr(page_idx), stride, _ptr(count), kf, _ptr(ctx_len), int(num_splits), _ptr(sink),
           _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), _stream())
    return out, lse


def refined_workspace(desc: L.AttnDesc, device="cuda"):
    """Zero-filled workspace of refined_decode_attend_combine (reusable)."""
    n = L.load().sls_refined_decode_attend_workspace_size(ctypes.byref(desc))
    return torch.zeros(max(int(n), 1), dtype=torch.uint8, device=device)


def refined_decode_attend_combine(desc: L.AttnDesc, q, k_cache, v_cache, codes, scales, res, block_idx, count,
                                  ctx_len, sink=None, out=None, lse=None, workspace=None, want_lse: bool = True):
    """Attention over the kept blocks of every row, the rows' lists cut into
    equal work items, combine fused; complete blocks are scored with the
    refined (2-bit + 8-bit) keys, or with the bf16 keys when codes, scales
    and res are None.  Returns (out, lse)."""
    for t, nm in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (block_idx, "block_idx"),
                  (count, "count")):
        _need(t, nm)
    B, Hq, D = desc.batch, desc.num_q_heads, desc.head_dim
    out = torch.empty((B, Hq, D), dtype=q.dtype, device=q.device) if out is None else out
    if want_lse and lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if sink is not None:
        _need(sink, "sink", torch.float32, (Hq,))
    workspace = refined_workspace(desc, q.device) if workspace is None else workspace
    L.call("sls_refined_decode_attend_combine", ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache),
           _ptr(codes), _ptr(scales), _ptr(res), _ptr(block_idx), int(block_idx.shape[-1]), _ptr(count),
           _ptr(ctx_len), _ptr(sink), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), _stream())
    return out, lse


def combine_splits(desc: L.AttnDesc, parts, sink=None, out=None, lse=None, want_lse: bool = True):
    """Log-sum-exp merge of the split partials with the optional sink
    (sls_combine_splits).  Returns (out [B, Hq, D], lse [B, Hq] or None)."""
    o, m, l = parts
    B, Hq, S, D = o.shape
    dtype = torch.bfloat16 if desc.dtype == L.SLS_DTYPE_BF16 else torch.float32
    out = torch.empty((B, Hq, D), dtype=dtype, device=o.device) if out is None else out
    if want_lse and lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=o.device)
    if sink is not None:
        _need(sink, "sink", torch.float32, (Hq,))
    L.call("sls_combine_splits", ctypes.byref(desc), _ptr(o), _ptr(m), _ptr(l), int(S), _ptr(sink),
           _ptr(out), _ptr(lse), _stream())
    return out, lse


def decode_append(desc: L.AttnDesc, k_new, v_new, k_cache, v_cache, ctx_len, kmin=None, kmax=None,
                  pos_out=None):
    """Writes one new token per sequence at ctx_len, keeps the page min/max
    current and advances ctx_len (all on the device)."""
    for t, nm in ((k_new, "k_new"), (v_new, "v_new"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, nm)
    L.call("sls_decode_append", ctypes.byref(desc), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
           _ptr(kmin), _ptr(kmax), _ptr(ctx_len), _ptr(pos_out), _stream())


def quest_step_workspace(desc: L.AttnDesc, k: int, num_splits: int = 0, device="cuda"):
    """Zero-filled workspace of quest_decode_step (reusable)."""
    n = L.load().sls_quest_decode_step_workspace_size(ctypes.byref(desc), int(k), int(num_splits))
    return torch.zeros(max(int(n), 1), dtype=torch.uint8, device=device)


def quest_step_splits(desc: L.AttnDesc, k: int) -> int:
    """Cluster size of the one-launch step for this shape (0: two launches)."""
    return int(L.load().sls_quest_decode_step_splits(ctypes.byref(desc), int(k)))


def quest_decode_step(desc: L.AttnDesc, q, k_cache, v_cache, kmin, kmax, ctx_len, k: int,
                      n_sink_pages: int = 0, n_local_tokens: int = 0, sink=None, page_idx=None,
                      out=None, lse=None, num_splits: int = 0, workspace=None, want_lse: bool = True,
                      min_sparsity: float = 0.0):
    """The whole Quest step (select + attend + combine), one launch where the
    shape allows; returns (out, lse).  page_idx, if given, receives the list."""
    for t, nm in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (kmin, "kmin"), (kmax, "kmax")):
        _need(t, nm)
    B, Hq, D = desc.batch, desc.num_q_heads, desc.head_dim
    dtype = torch.bfloat16 if desc.dtype == L.SLS_DTYPE_BF16 else torch.float32
    out = torch.empty((B, Hq, D), dtype=dtype, device=q.device) if out is None else out
    if want_lse and lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if sink is not None:
        _need(sink, "sink", torch.float32, (Hq,))
    if page_idx is not None:
        _need(page_idx, "page_idx", torch.int32, (desc.batch * desc.num_kv_heads, int(k)))
    workspace = quest_step_workspace(desc, k, num_splits, q.device) if workspace is None else workspace
    L.call("sls_quest_decode_step", ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kmin),
           _ptr(kmax), _ptr(ctx_len), int(k), int(n_sink_pages), int(n_local_tokens), _ptr(sink),
           _ptr(page_idx), _ptr(out), _ptr(lse), int(num_splits), float(min_sparsity), _ptr(workspace),
           workspace.numel(), _stream())
    return out, lse


def selection_recall(desc: L.AttnDesc, q, k_cache, page_idx, ctx_len, count=None,
                     k_fixed: Optional[int] = None, recall=None, workspace=None):
    """Attention-mass recall of each query head's page list: [B, Hq] float32."""
    _need(q, "q")
    _need(k_cache, "k_cache")
    recall = torch.empty((desc.batch, desc.num_q_heads), dtype=torch.float32, device=q.device) \
        if recall is None else recall
    n = L.load().sls_selection_recall_workspace_size(ctypes.byref(desc))
    workspace = torch.empty(max(int(n), 1), dtype=torch.uint8, device=q.device) if workspace is None else workspace
    stride = int(page_idx.shape[1]) if page_idx is not None else 0
    kf = stride if k_fixed is None else int(k_fixed)
    L.call("sls_selection_recall", ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(page_idx), stride, _ptr(count),
           kf, _ptr(ctx_len), _ptr(recall), _ptr(workspace), workspace.numel(), _stream())
    return recall


# ------------------------------------------------------------ decode step

class QuestDecode:
    """One Quest decode step (select + attend + combine) over preallocated
    buffers, capturable in a CUDA graph.  one_launch: the whole step in one
    kernel where the shape allows (quest_decode_step); otherwise select, then
    attend with the combine fused (fused=True) or as its own launch."""

    def __init__(self, desc: L.AttnDesc, k_budget: int, n_sink_pages: int, n_local_tokens: int,
                 num_splits: Optional[int] = None, device="cuda", fused: bool = True,
                 one_launch: bool = True, min_sparsity: float = 0.0):
        self.desc = desc
        self.k = int(k_budget)
        self.n_sink, self.n_local = int(n_sink_pages), int(n_local_tokens)
        self.fused = fused
        self.one_launch = fused and one_launch
        self.min_sparsity = float(min_sparsity)
        rows = desc.batch * desc.num_kv_heads
        self.S = num_splits or default_splits(desc, self.k)
        self.step_splits = int(num_splits or 0)
        self.step_workspace = quest_step_workspace(desc, self.k, self.step_splits, device)
        self.page_idx = torch.empty((rows, self.k), dtype=torch.int32, device=device)
        self.workspace = select_pages_workspace(desc, device)
        self.parts = partials(desc, self.S, device)
        self.ac_workspace = attend_combine_workspace(desc, self.S, device)
        dtype = torch.bfloat16 if desc.dtype == L.SLS_DTYPE_BF16 else torch.float32
        self.out = torch.empty((desc.batch, desc.num_q_heads, desc.head_dim), dtype=dtype, device=device)
        self.lse = torch.empty((desc.batch, desc.num_q_heads), dtype=torch.float32, device=device)

    def select(self, q, kmin, kmax, ctx_len):
        return select_pages(self.desc, q, kmin, kmax, ctx_len, self.k, self.n_sink, self.n_local,
                            out=self.page_idx, workspace=self.workspace)

    def attend(self, q, k_cache, v_cache, ctx_len, sink=None):
        if self.fused:
            return sparse_decode_attend_combine(self.desc, q, k_cache, v_cache, self.page_idx, ctx_len,
                                                self.S, sink=sink, out=self.out, lse=self.lse,
                                                workspace=self.ac_workspace)
        sparse_decode_attend(self.desc, q, k_cache, v_cache, self.page_idx, ctx_len, self.S,
                             parts=self.parts)
        return combine_splits(self.desc, self.parts, sink, out=self.out, lse=self.lse)

    def __call__(self, q, k_cache, v_cache, kmin, kmax, ctx_len, sink=None):
        if self.one_launch:
            return quest_decode_step(self.desc, q, k_cache, v_cache, kmin, kmax, ctx_len, self.k, self.n_sink,
                                     self.n_local, sink=sink, page_idx=self.page_idx, out=self.out,
                                     lse=self.lse, num_splits=self.step_splits, workspace=self.step_workspace,
                                     min_sparsity=self.min_sparsity)
        self.select(q, kmin, kmax, ctx_len)
        return self.attend(q, k_cache, v_cache, ctx_len, sink)


class DeltaDecode:
    """One top-delta decode step (select_delta + attend + combine).

    balanced=True (the default where the shape allows: bf16, G <= 8, no path
    flag in the descriptor) attends
    with the work-item kernel, which spreads rows of very different list
    lengths evenly over the GPU; otherwise the split-K attend with num_splits
    per row.  With refined=True the attend scores complete blocks with the
    refined keys (2-bit thumbnail + 8-bit residual, "Faster Than Flash"
    eq. 4): the call then takes the residuals as well."""

    def __init__(self, desc: L.AttnDesc, block: int, delta: float, num_splits: Optional[int] = None,
                 device="cuda", fused: bool = True, refined: bool = False, balanced: Optional[bool] = None):
        if desc.page_size != block:
            raise ValueError("attend page_size must equal the thumbnail block")
        self.desc, self.block, self.delta = desc, int(block), float(delta)
        self.fused = fused
        self.refined = refined
        ok = (desc.dtype == L.SLS_DTYPE_BF16 and desc.num_q_heads // desc.num_kv_heads <= 8
              and desc.batch * desc.num_kv_heads <= 4096)  # the work-item kernel's row limit
        # the default for the fast path only: the descriptor's path flags select the split-K attends
        self.balanced = (fused and ok and desc.flags == 0) if balanced is None else balanced
        if refined and not ok:
            raise ValueError("the refined attend needs bf16 and G <= 8")
        self.bal_workspace = refined_workspace(desc, device) if (self.balanced or refined) else None
        rows = desc.batch * desc.num_kv_heads
        nblk = desc.capacity // block
        self.S = num_splits or default_splits(desc, nblk)
        self.count = torch.empty(rows, dtype=torch.int32, device=device)
        self.block_idx = torch.empty((rows, nblk), dtype=torch.int32, device=device)
        self.workspace = select_delta_workspace(desc, block, device)
        self.parts = partials(desc, self.S, device)
        self.ac_workspace = attend_combine_workspace(desc, self.S, device)
        dtype = torch.bfloat16 if desc.dtype == L.SLS_DTYPE_BF16 else torch.float32
        self.out = torch.empty((desc.batch, desc.num_q_heads, desc.head_dim), dtype=dtype, device=device)
        self.lse = torch.empty((desc.batch, desc.num_q_heads), dtype=torch.float32, device=device)

    def select(self, q, k_cache, codes, scales, ctx_len):
        return select_delta(self.desc, q, k_cache, codes, scales, ctx_len, self.block, self.delta,
                            count=self.count, block_idx=self.block_idx, workspace=self.workspace)

    def attend(self, q, k_cache, v_cache, ctx_len, sink=None):
        if self.balanced:
            return refined_decode_attend_combine(self.desc, q, k_cache, v_cache, None, None, None, self.block_idx,
                                                 self.count, ctx_len, sink=sink, out=self.out, lse=self.lse,
                                                 workspace=self.bal_workspace)
        if self.fused:
            return sparse_decode_attend_combine(self.desc, q, k_cache, v_cache, self.block_idx, ctx_len,
                                                self.S, count=self.count, sink=sink, out=self.out,
                                                lse=self.lse, workspace=self.ac_workspace)
        sparse_decode_attend(self.desc, q, k_cache, v_cache, self.block_idx, ctx_len, self.S,
                             count=self.count, parts=self.parts)
        return combine_splits(self.desc, self.parts, sink, out=self.out, lse=self.lse)

    def attend_refined(self, q, k_cache, v_cache, codes, scales, res, ctx_len, sink=None):
        return refined_decode_attend_combine(self.desc, q, k_cache, v_cache, codes, scales, res, self.block_idx,
                                             self.count, ctx_len, sink=sink, out=self.out, lse=self.lse,
                                             workspace=self.bal_workspace)

    def __call__(self, q, k_cache, v_cache, codes, scales, ctx_len, sink=None, res=None):
        self.select(q, k_cache, codes, scales, ctx_len)
        if self.refined:
            if res is None:
                raise ValueError("the refined step needs the residuals")
            return self.attend_refined(q, k_cache, v_cache, codes, scales, res, ctx_len, sink)
        return self.attend(q, k_cache, v_cache, ctx_len, sink)
