"""The N > 1 path of bench.py on the CPU: replicas with no data-path
collective, whose timings meet in one max-over-ranks all-reduce (gloo,
world size 2, two spawned processes on 127.0.0.1)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], world, "cpu")
        out[rank] = (ms, bench.replica_throughput(ms, world, 16, 100))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_throughput():
    world, port = 2, _free_port()
    times = [12.5, 17.25]  # ms: rank 1 is the slower replica
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, port, times, out), nprocs=world, start_method="spawn", join=True)
    for r in range(world):
        ms, value = out[r]
        assert ms == 17.25
        # two replicas x 16 tokens x 100 steps over the slowest replica's 17.25 ms
        assert value == pytest.approx(2 * 16 * 100 / 17.25e-3)


def test_single_replica_needs_no_process_group():
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.replica_throughput(2.0, 1, 1, 1000) == pytest.approx(500_000.0)
