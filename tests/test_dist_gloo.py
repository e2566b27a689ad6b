"""The multi-rank leg of the benchmark on CPU: world size 2 over gloo.

Heads and batches are independent, so ranks run replicas with no data-path
exchange; the only collective is the timing aggregation (slowest rank's time,
sum of all ranks' FLOPs), checked here without a GPU.
"""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_total = [40.0, 55.0][rank]  # rank 1 is the slowest
        flops = [1.0e12, 1.0e12][rank]
        ms_per_step, value = bench.aggregate_ranks(ms_total, flops, steps=10, world=world)
        out[rank] = (ms_per_step, value)
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
        res = dict(out)
    for rank in (0, 1):
        ms_per_step, value = res[rank]
        assert ms_per_step == pytest.approx(5.5)
        assert value == pytest.approx(2.0e12 / 5.5e-3 / 1e12)


def test_single_rank_aggregation():
    import bench

    ms, v = bench.aggregate_ranks(20.0, 4.0e12, steps=4, world=1)
    assert ms == 5.0 and v == pytest.approx(4.0e12 / 5e-3 / 1e12)
