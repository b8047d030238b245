"""The N>1 bench path: independent replicas, one per rank, no data-path
collective; the job's step time is the slowest rank's and its throughput
counts every rank's tokens.  Run as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [3.0, 5.0][rank]                       # rank 1 is the slow replica
    ms_max = bench.reduce_max(ms, dist, "cpu")
    value = bench.job_value(32, world, ms_max)
    dist.barrier()
    out[rank] = (ms_max, value)
    dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_rank():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        ms_max, value = out[r]
        assert ms_max == 5.0
        assert value == pytest.approx(32 * 2 / 5e-3)


def test_single_process_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(2.5, None, "cpu") == 2.5
    assert bench.job_value(32, 1, 2.0) == pytest.approx(16000.0)
