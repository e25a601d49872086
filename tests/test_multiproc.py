"""Replica host logic of bench.py at world size 2 (gloo on CPU): the rank
environment, the barrier, and the maximum-over-ranks timing reduction."""
import os
import socket

import pytest


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    import torch.distributed as dist
    import bench
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, local, w = bench.dist_env()
        bench.barrier()
        t = bench.reduce_max(10.0 + 5.0 * rank)  # per-rank timings differ; the job time is the slowest
        bench.barrier()
        q.put((r, local, w, t))
    finally:
        dist.destroy_process_group()


def test_replica_timing_is_max_over_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 0, 2, 15.0), (1, 1, 2, 15.0)]


def test_single_process_reduce_is_identity():
    import bench
    assert bench.reduce_max(3.5) == 3.5
    bench.barrier()
