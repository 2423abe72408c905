"""Multi-rank host logic of bench.py (replicas): the job time is the maximum
over ranks and the throughput counts every rank's units.  Two gloo ranks on
CPU."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    local_seconds = [0.002, 0.005][rank]
    value, t = bench.aggregate(448, local_seconds, world)
    out[rank] = (value, t)
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_is_max_over_ranks():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    for r in range(world):
        value, t = out[r]
        assert t == pytest.approx(0.005)
        assert value == pytest.approx(448 * 2 / 0.005)


def test_single_rank_aggregate():
    import bench

    value, t = bench.aggregate(448, 0.004, 1)
    assert t == 0.004 and value == pytest.approx(448 / 0.004)
