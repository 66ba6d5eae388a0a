"""The multi-rank bookkeeping of bench.py on CPU with the gloo backend.

Under torchrun every rank runs its own replica of the GEMM; the job time is
the slowest rank's and the job throughput counts every rank's work.  Two
gloo ranks with different (fake) elapsed times check the max-reduction and
the throughput formula.
"""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = [12.5, 20.0][rank]
        slowest = bench.reduce_max(elapsed, world)
        out[rank] = (slowest, bench.job_throughput(2.0 * 8192 ** 3, 10, world, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
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
    assert out[0][0] == out[1][0] == 20.0
    expect = 2.0 * 8192 ** 3 * 10 * 2 / 20e-3 / 1e12
    assert out[0][1] == pytest.approx(expect)


def test_single_rank_needs_no_process_group():
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.job_throughput(1e12, 4, 1, 1000.0) == pytest.approx(4.0)
