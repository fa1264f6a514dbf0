"""Multi-GPU is replicas only (the path has no exchange step).  The host-side
aggregation bench.py uses under torchrun (max of the per-rank times, whole-job
units per second) is checked here with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [120.0, 150.0][rank]
        slowest = bench.max_over_ranks(local_ms, dist, "cpu")
        out[rank] = bench.replica_throughput(world, 64, 1000, slowest)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_agree_on_the_slowest_rank():
    mgr = mp.get_context("spawn").Manager()   # no fork of this multi-threaded process
    out = mgr.dict()
    mp.spawn(_rank, args=(2, _free_port(), out), nprocs=2, join=True)
    want = 2 * 64 * 1000 / 0.150
    assert out[0] == pytest.approx(want) and out[1] == pytest.approx(want)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.replica_throughput(1, 64, 10, 1000.0) == pytest.approx(640.0)
