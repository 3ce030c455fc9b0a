"""The replica path of bench.py with two gloo ranks on the CPU: the timing
reduction takes the slowest rank's time and the sum of the ranks' work, and
every rank sees the same result."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        assert bench.dist_env() == (rank, world, rank)
        elapsed = 0.5 + rank          # rank 1 is the slow one
        units = 1000.0 * (rank + 1)
        t, u = bench.reduce_timing(elapsed, units)
        bench.barrier()
        out[rank] = (t, u)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_timing_reduction():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    assert dict(out) == {0: (1.5, 3000.0), 1: (1.5, 3000.0)}


def test_single_process_reduction_is_identity():
    import bench
    assert not dist.is_initialized()
    assert bench.reduce_timing(0.25, 42.0) == (0.25, 42.0)


def test_buffer_rotation_exceeds_l2():
    import bench
    l2 = 126 * 2**20
    for set_bytes in (2**20, 32 * 2**20, 128 * 2**20, 2**30):
        n = bench.buffer_sets_for(set_bytes, l2)
        assert n >= 1
        assert n * set_bytes >= min(2 * l2, 64 * set_bytes)
