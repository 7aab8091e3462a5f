"""The N > 1 path of bench.py (independent replicas, one per GPU) with two gloo ranks on the CPU:
the slowest rank's time sets the job time, the job rate counts every rank's units, and the
reference arm runs on rank 0 alone."""
import os
import socket
import sys
import types

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        mine = 1.0 + rank * 0.5  # rank 1 is the slowest
        slowest = bench.max_over_ranks(mine, torch.device("cpu"))
        rate = bench.job_throughput(1000.0, 10, world, slowest)
        ref = bench.run_reference(types.SimpleNamespace(steps=1, warmup=0), rank, world) if rank != 0 else None
        dist.barrier()
        out[rank] = (slowest, rate, ref)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert set(res) == {0, 1}
    for r in range(world):
        slowest, rate, _ = res[r]
        assert slowest == pytest.approx(1.5)
        assert rate == pytest.approx(1000.0 * 10 * 2 / 1.5)
    assert res[1][2] is None  # the reference arm does no work off rank 0
