"""Seeded synthetic decode-attention workloads.

This module only draws inputs: keys, values, queries, sink logits and context
lengths with the shapes and structure of the five workloads below.  It holds
none of the method's arithmetic (no scores, no bounds, no selection, no
softmax), so both the CUDA path and the fp64 oracle consume the same bytes.

Every (batch, kv-head) row has its own generator, seeded from
``(seed, b, h)``, so a single row can be regenerated alone (the oracle checks
sampled rows of full-size workloads that way) and is identical to that row of
the full tensor.

Workloads (sizes from the workload list this library is measured on):

* ``tiny``   fp32, B=1, Hq=4, Hkv=1, D=64, N=1024, P=16, top-8 pages.
  K, V ~ N(0,1); three planted pages; every query head is the sum of the
  planted keys plus N(0, 0.5^2) noise.
* ``qwen7b`` bf16, B=8, Hq=28, Hkv=4, D=128, N=32768, P=16, budget 128 pages.
* ``qwen1p5b`` bf16, B=32, Hq=12, Hkv=2, D=128, N=65536 (4k-64k sweep),
  P=16, budget 128 pages.
* ``gptoss`` bf16, B=4, Hq=64, Hkv=8, D=64, N=131072, token-level (P=1)
  selection of 4096 tokens per row, first 4 tokens always kept, per-head
  sink logit ~ N(0,1).
* ``ffd``    bf16, B=2, Hq=32, Hkv=8, D=128, N=262144, 64-token thumbnail
  blocks, top-delta with delta=5.

The "outlier" generator (all but ``tiny``): K[b,h,t,c] = sigma[h,c] * z with
sigma ~ LogNormal(0, 0.5) per (kv head, channel) and z ~ N(0,1); V ~ N(0,1);
each row plants needle tokens, and every query head of the row is
``a * sum(needle keys)/sqrt(#needles) + b * sum(last 64 keys)/8 + N(0,1)``
with a=4, b=1.  Cache slots at positions >= ctx_len hold keys and values
scaled by ``TAIL_GAIN`` so that a kernel reading past the context is caught.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

BASE_SEED = 20261202
NEEDLE_GAIN = 4.0   # a
RECENCY_GAIN = 1.0  # b
RECENCY_TOKENS = 64
TAIL_GAIN = 8.0
# Gain of the planted leading key of the ffd workload (token 0), in units of
# the group's mean query norm; fixed so that about 18% of blocks are kept.
FFD_SINK_GAIN = 0.11

CONFIG_NAMES = ("tiny", "qwen7b", "qwen1p5b", "gptoss", "ffd")


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (u.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class Spec:
    """Shape and selection parameters of one workload."""
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    ctx_len: tuple            # per batch entry
    capacity: int             # cache slots per (b, kv head), multiple of page and block
    dtype: str                # "f32" | "bf16"
    selector: str             # "quest" | "delta"
    k_pages: int = 0          # quest budget in pages (includes forced pages)
    n_sink_pages: int = 0
    n_local_tokens: int = 0
    block: int = 64           # thumbnail block (delta selector)
    delta: float = 5.0
    has_sink: bool = False
    seed: int = BASE_SEED
    generator: str = "outlier"  # "planted" (tiny) | "outlier"
    n_needles: int = 4        # needle pages / spans / blocks per row
    needle_len: int = 16      # tokens per needle
    ffd_sink_gain: float = 0.0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def rows(self) -> int:
        return self.batch * self.num_kv_heads

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


def spec(name: str, *, batch: Optional[int] = None, ctx_len=None,
         capacity: Optional[int] = None) -> Spec:
    """Build the named workload, optionally with a different batch, context
    length(s) (an int or one per batch entry) or cache capacity."""
    idx = CONFIG_NAMES.index(name)
    seed = BASE_SEED + idx
    if name == "tiny":
        s = Spec(name, 1, 4, 1, 64, 16, (1024,), 1024, "f32", "quest",
                 k_pages=8, seed=seed, generator="planted", n_needles=3)
    elif name == "qwen7b":
        s = Spec(name, 8, 28, 4, 128, 16, (32768,) * 8, 32768, "bf16", "quest",
                 k_pages=128, n_sink_pages=1, n_local_tokens=64, seed=seed)
    elif name == "qwen1p5b":
        s = Spec(name, 32, 12, 2, 128, 16, (65536,) * 32, 65536, "bf16", "quest",
                 k_pages=128, n_sink_pages=1, n_local_tokens=64, seed=seed)
    elif name == "gptoss":
        s = Spec(name, 4, 64, 8, 64, 1, (131072,) * 4, 131072, "bf16", "quest",
                 k_pages=4096, n_sink_pages=4, n_local_tokens=0, has_sink=True,
                 seed=seed)
    elif name == "ffd":
        s = Spec(name, 2, 32, 8, 128, 64, (262144,) * 2, 262144, "bf16", "delta",
                 block=64, delta=5.0, seed=seed, needle_len=64,
                 ffd_sink_gain=FFD_SINK_GAIN)
    else:  # pragma: no cover
        raise ValueError(name)
    if batch is not None:
        s.batch = batch
        s.ctx_len = tuple(s.ctx_len[:1]) * batch
    if ctx_len is not None:
        if np.isscalar(ctx_len):
            s.ctx_len = (int(ctx_len),) * s.batch
        else:
            s.ctx_len = tuple(int(c) for c in ctx_len)
            s.batch = len(s.ctx_len)
    if capacity is None:
        unit = max(s.page_size, s.block if s.selector == "delta" else 1, 16)
        capacity = max(max(s.ctx_len), 1)
        capacity = -(-capacity // unit) * unit
    s.capacity = int(capacity)
    assert s.capacity >= max(s.ctx_len)
    return s


@dataclasses.dataclass
class Row:
    """One (batch, kv head) row: keys and values [Cap, D], the group's
    queries [G, D] (bf16 bit patterns or fp32) and the planted needles."""
    K: np.ndarray
    V: np.ndarray
    q: np.ndarray
    needles: np.ndarray   # token positions of the planted needles


def _sigma(s: Spec) -> np.ndarray:
    rng = np.random.default_rng([s.seed, 1_000_000])
    return rng.lognormal(0.0, 0.5, size=(s.num_kv_heads, s.head_dim)).astype(np.float32)


def sinks(s: Spec) -> Optional[np.ndarray]:
    """Per query head sink logits (fp32, raw logits), or None."""
    if not s.has_sink:
        return None
    rng = np.random.default_rng([s.seed, 2_000_000])
    return rng.standard_normal(s.num_q_heads).astype(np.float32)


def _pick_needles(rng, s: Spec, n: int) -> np.ndarray:
    """Start positions of the planted needles, uniform over the interior of
    the valid context (away from the first needle-length and the recency
    window).  Needles are aligned to needle_len."""
    L = s.needle_len
    lo = 1                                   # in units of needle_len
    hi = (n - RECENCY_TOKENS - L) // L       # last admissible start unit
    if hi < lo:
        return np.zeros(0, dtype=np.int64)
    count = min(s.n_needles, hi - lo + 1)
    units = rng.choice(np.arange(lo, hi + 1), size=count, replace=False)
    return np.sort(units) * L


def gen_row(s: Spec, b: int, h: int, sigma: Optional[np.ndarray] = None,
            seq: Optional[int] = None) -> Row:
    """Generate row (b, h) of the workload (seeded by sequence number ``seq``,
    default b)."""
    rng = np.random.default_rng([s.seed, b if seq is None else seq, h])
    n = s.ctx_len[b]
    cap, d, g = s.capacity, s.head_dim, s.group
    if s.generator == "planted":
        npages = -(-n // s.page_size)
        count = min(s.n_needles, npages)
        pages = np.sort(rng.choice(npages, size=count, replace=False))
        K = rng.standard_normal((cap, d), dtype=np.float32)
        V = rng.standard_normal((cap, d), dtype=np.float32)
        toks = np.concatenate([np.arange(p * s.page_size, min((p + 1) * s.page_size, n))
                               for p in pages]) if count else np.zeros(0, np.int64)
        base = K[toks].sum(axis=0)
        q = base[None, :] + 0.5 * rng.standard_normal((g, d), dtype=np.float32)
        needles = toks
    else:
        if sigma is None:
            sigma = _sigma(s)
        starts = _pick_needles(rng, s, n)
        K = rng.standard_normal((cap, d), dtype=np.float32) * sigma[h][None, :]
        V = rng.standard_normal((cap, d), dtype=np.float32)
        needles = (starts[:, None] + np.arange(s.needle_len)[None, :]).reshape(-1)
        qv = np.zeros(d, dtype=np.float32)
        if needles.size:
            qv += NEEDLE_GAIN * K[needles].sum(axis=0) / np.float32(math.sqrt(needles.size))
        lo = max(n - RECENCY_TOKENS, 0)
        if n > lo:
            qv += RECENCY_GAIN * K[lo:n].sum(axis=0) / np.float32(math.sqrt(RECENCY_TOKENS))
        q = qv[None, :] + rng.standard_normal((g, d), dtype=np.float32)
        if s.ffd_sink_gain > 0 and n > 0:
            qbar = q.mean(axis=0)
            norm = float(np.linalg.norm(qbar)) or 1.0
            mean_q = float(np.linalg.norm(q, axis=1).mean())
            K[0] = (s.ffd_sink_gain * mean_q) * qbar / norm
    if n < cap:
        K[n:] *= TAIL_GAIN
        V[n:] *= TAIL_GAIN
    if s.dtype == "bf16":
        return Row(round_to_bf16_bits(K), round_to_bf16_bits(V),
                   round_to_bf16_bits(q), needles)
    return Row(K, V, q.astype(np.float32), needles)


@dataclasses.dataclass
class Tensors:
    """Host arrays of a whole workload.  bf16 tensors are uint16 bit patterns."""
    K: np.ndarray        # [B, Hkv, Cap, D]
    V: np.ndarray        # [B, Hkv, Cap, D]
    q: np.ndarray        # [B, Hq, D]
    ctx_len: np.ndarray  # [B] int32
    sink: Optional[np.ndarray]  # [Hq] fp32 or None
    needles: list        # [B][Hkv] arrays of needle token positions


def generate(s: Spec, rows=None, batch_offset: int = 0) -> Tensors:
    """Generate the whole workload (``rows=None``) or only the listed
    (b, h) rows (others stay zero).  ``batch_offset`` shifts the sequence
    numbers the rows are seeded with (shard r of a multi-GPU run draws
    sequences r*B .. r*B+B-1)."""
    B, Hkv, Cap, D, G = s.batch, s.num_kv_heads, s.capacity, s.head_dim, s.group
    dt = np.uint16 if s.dtype == "bf16" else np.float32
    K = np.zeros((B, Hkv, Cap, D), dtype=dt)
    V = np.zeros((B, Hkv, Cap, D), dtype=dt)
    q = np.zeros((B, Hkv * G, D), dtype=dt)
    needles = [[None] * Hkv for _ in range(B)]
    sigma = _sigma(s) if s.generator == "outlier" else None
    todo = [(b, h) for b in range(B) for h in range(Hkv)] if rows is None else rows
    for b, h in todo:
        r = gen_row(s, b, h, sigma, seq=b + batch_offset)
        K[b, h], V[b, h] = r.K, r.V
        q[b, h * G:(h + 1) * G] = r.q
        needles[b][h] = r.needles
    return Tensors(K, V, q, np.asarray(s.ctx_len, dtype=np.int32), sinks(s), needles)
