"""The multi-GPU bench path shards sequences across ranks with no data-path
collective; the only exchange is the timing/units reduction.  Checked here
with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t, u = bench.aggregate(1.0 + rank, 10.0 * (rank + 1), world)
    r, w, lr = bench.dist_env()
    q.put((rank, t, u, r, w))
    dist.destroy_process_group()


def test_aggregate_max_time_sum_units_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, u, r, w in res:
        assert t == 2.0 and u == 30.0 and r == rank and w == 2


def test_shards_draw_distinct_sequences():
    from sparse_long_context_gb300 import workloads as W
    s = W.spec("qwen7b", batch=2, ctx_len=256)
    a = W.generate(s, batch_offset=0)
    b = W.generate(s, batch_offset=2)
    assert not (a.K == b.K).all()
    one = W.generate(W.spec("qwen7b", batch=4, ctx_len=256))
    assert (one.K[2:] == b.K).all()


def test_algorithmic_bytes_of_the_benchmark_workload():
    from sparse_long_context_gb300 import workloads as W
    nb = bench.algorithmic_bytes(W.spec("qwen1p5b"))
    assert nb["select"] == 32 * 2 * 4096 * 2 * 128 * 2          # 134.2 MB of page min/max
    assert nb["attend"] == 32 * 2 * 2048 * 2 * 128 * 2          # 67.1 MB of selected K+V
    assert abs(nb["total"] / 1e6 - 201.3) < 0.1


def test_delta_bytes_counts_refined_and_partial_blocks():
    """Top-delta step bytes: bf16 K + V of every kept token; with residuals a
    complete block reads codes (D/4) + residuals (D) + V (2D) per token and
    its scales (2D) once, the partial newest block stays on bf16 keys."""
    import numpy as np
    from sparse_long_context_gb300 import workloads as W
    s = W.spec("ffd", batch=1, ctx_len=[64 * 3 + 10], capacity=64 * 4)
    D = s.head_dim
    count = np.zeros(s.rows, dtype=np.int32)
    idx = np.full((s.rows, 4), -1, dtype=np.int32)
    count[0], idx[0, :3] = 3, [0, 2, 3]          # two complete blocks, the partial one (10 tokens)
    count[1], idx[1, :1] = 1, [1]
    nb = bench.delta_bytes(s, s.ctx_len, count, idx)
    assert nb["scan"] == bench.algorithmic_bytes(s)["select"]
    assert nb["attend_exact"] == (64 + 64 + 10 + 64) * 2 * D * 2
    refined_block = 64 * (D // 4 + D + 2 * D) + 2 * D
    assert nb["attend_refined"] == 3 * refined_block + 10 * 2 * D * 2
    assert bench.step_traffic(W.spec("qwen1p5b", batch=8)) is None   # only the captured workload
