"""The N > 1 host logic of bench.py on CPU: two gloo ranks, each a replica
with its own elapsed time and FLOP count; the job time is the slowest rank
and the work is the sum over ranks."""
from __future__ import annotations

import os
import socket

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, rank)
        ms, fl = bench.aggregate(10.0 + 5.0 * rank, 1e12 * (rank + 1))
        bench.barrier()
        out.put((rank, ms, fl))
    finally:
        dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
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
    for rank, ms, fl in got:
        assert ms == 15.0           # the slowest rank
        assert fl == 3e12           # every rank's FLOPs


def test_aggregate_single_process_is_identity():
    import bench
    assert bench.aggregate(7.5, 2e9) == (7.5, 2e9)
