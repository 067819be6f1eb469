"""The multi-rank bookkeeping of bench.py (replicas, max over ranks, whole-job
rate) with two gloo ranks on the CPU."""
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


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 10.0 + 5.0 * rank                 # rank 1 is the slow one
    worst = bench.max_over_ranks(ms, world, torch.device("cpu"))
    rate = bench.whole_job_rate(128, world, worst)
    out[rank] = (worst, rate)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        for r in range(world):
            worst, rate = out[r]
            assert worst == 15.0
            assert rate == pytest.approx(128 * 2 / 0.015)


def test_single_rank_passthrough():
    import bench
    assert bench.max_over_ranks(3.5, 1, None) == 3.5
    assert bench.whole_job_rate(128, 1, 10.0) == pytest.approx(12800.0)
