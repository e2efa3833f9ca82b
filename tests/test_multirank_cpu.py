"""The N > 1 path of the benchmark on CPU: two gloo ranks.

The layer has no exchange step: blocks are independent, so ranks are replicas
that each process their own rows (weak scaling).  What the ranks share is the
harness: distinct per-rank inputs of the same shape, the barrier around the
timed region and the maximum of the per-rank times.
"""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    from sparse_moe_layer_row_gb300 import workloads as W
    w = W.BLOCK32
    ws_, rank_, local_ = bench.dist_env()
    assert (ws_, rank_, local_) == (ws, rank, rank)
    seed = bench.rank_workload(w, rank)
    x = W.make_x(w, "cpu", rows=4, seed=seed)
    bench.barrier(ws)
    t = bench.reduce_max(1.0 + rank, ws)
    out[rank] = (seed, float(x.float().sum()), t)
    dist.destroy_process_group()


def test_two_gloo_ranks_are_independent_replicas():
    ws = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, out)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    (s0, x0, t0), (s1, x1, t1) = out[0], out[1]
    assert s0 != s1 and x0 != x1          # distinct rows per rank
    assert t0 == t1 == 2.0                # max over ranks reaches every rank


def test_single_process_helpers():
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
    from sparse_moe_layer_row_gb300 import workloads as W
    assert bench.rank_workload(W.BLOCK32, 0) == W.BLOCK32.x_seed
