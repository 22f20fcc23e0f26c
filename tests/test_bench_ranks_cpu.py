"""The multi-rank timing logic of bench.py on CPU: two gloo ranks, the slowest rank's step time
wins, and the job throughput counts every rank's work (weak scaling)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world_size, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world_size)
    import bench
    ms = bench.max_over_ranks(1.5 + rank, torch.device("cpu"))
    out[rank] = ms
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_job_throughput_is_weak_scaling():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_throughput(1, 6.44e9, 0.058)
    assert abs(one - 6.44e9 / 0.058e-3 / 1e12) < 1e-9
    assert abs(bench.job_throughput(4, 6.44e9, 0.058) - 4 * one) < 1e-9
