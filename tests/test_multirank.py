"""The benchmark's multi-rank arithmetic on CPU ranks (gloo, world size 2).

Each rank runs its own batch (weak scaling; the layer has no data-path
exchange between ranks).  The job time is the slowest rank's time and the
job throughput counts every rank's tokens.  Ranks run as spawned processes
rendezvousing on 127.0.0.1.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank: int, world: int, port: int, results):
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r took (r + 1) * 10 ms for 1000 tokens
        ms, value = bench.job_throughput(10.0 * (rank + 1), 1000, dist)
        results[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_job_throughput_uses_slowest_rank_and_all_tokens():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        ms, value = results[r]
        assert ms == pytest.approx(20.0)                 # max over ranks
        assert value == pytest.approx(2 * 1000 / 0.020)  # all ranks' tokens / job time


def test_job_throughput_single_process():
    import bench
    ms, value = bench.job_throughput(4.0, 500)
    assert ms == 4.0 and value == pytest.approx(500 / 0.004)
