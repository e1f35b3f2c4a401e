"""Replica aggregation of bench.py across ranks (world size 2, gloo, CPU):
every rank's bytes over the slowest rank's time."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        nbytes = 1.0e9 * (rank + 1)
        t = 0.010 * (rank + 1)
        per_rank = bench.all_gather_floats([nbytes, t], world)
        value, t_max = bench.aggregate([r[0] for r in per_rank], [r[1] for r in per_rank])
        out[rank] = (per_rank, value, t_max)
    finally:
        dist.destroy_process_group()


def test_aggregate_single_rank():
    import bench
    v, t = bench.aggregate([2.0e9], [0.5])
    assert t == 0.5 and v == 4.0e9
    assert bench.aggregate([1.0], [0.0]) == (0.0, 0.0)


def test_all_gather_and_aggregate_two_ranks():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    for rank in range(world):
        per_rank, value, t_max = out[rank]
        assert per_rank == [[1.0e9, 0.010], [2.0e9, 0.020]]
        assert t_max == pytest.approx(0.020)
        assert value == pytest.approx(3.0e9 / 0.020)
