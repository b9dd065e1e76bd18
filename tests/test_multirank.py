"""The bench's multi-rank host logic on CPU: two gloo ranks (127.0.0.1).

Each GPU runs an independent replica of the step ("replicas only": the path has
no exchange step on one GPU); the only cross-rank work is the barrier, the
maximum of the ranks' step times and the whole-job throughput.  No GPU involved.
"""
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


def _worker(rank, world, port, out):
    import sys

    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        local_ms = [12.5, 14.25][rank]
        slowest = bench.max_over_ranks(local_ms, world)
        value = bench.job_value(world, 38.5e12, slowest)
        dist.barrier()
        # the reference arm does its work on rank 0 only; other ranks return at once
        args = type("A", (), {"workload": bench.DEFAULT_WORKLOAD, "steps": 1, "warmup": 3})()
        ref = bench.run_reference(args, rank, world, rank) if rank != 0 else "rank0"
        out[rank] = (slowest, value, ref)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    assert set(out.keys()) == {0, 1}
    for rank in (0, 1):
        slowest, value, _ = out[rank]
        assert slowest == 14.25
        assert value == pytest.approx(2 * 38.5e12 / 14.25e-3 / 1e12)
    assert out[1][2] is None


def test_single_rank_is_identity():
    import sys

    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_value(1, 1e12, 1.0) == pytest.approx(1000.0)
