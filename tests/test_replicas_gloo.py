"""The benchmark's multi-rank path on CPU: two gloo ranks, each an independent
replica; the job's time is the slowest rank's and its throughput counts every
rank's batch."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    slow = bench.max_over_ranks(10.0 + rank)  # rank 1 is the slower replica
    out[rank] = (slow, bench.replica_throughput(2e12, world, slow))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert out[0][0] == out[1][0] == 11.0
    assert out[0][1] == pytest.approx(2e12 * 2 / 11e-3 / 1e12)


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.replica_throughput(1e12, 1, 1.0) == pytest.approx(1000.0)
