"""Multi-process host logic of the bench on CPU (gloo, world size 2): the
slowest rank sets the time and every rank gets the same reduced values."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        mine = [1.0 + rank, 10.0 - rank, 0.5 * rank]
        out[rank] = bench.max_over_ranks(mine)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_processes():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    expect = [2.0, 10.0, 0.5]
    assert res[0] == expect and res[1] == expect


def test_max_over_ranks_single_process_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 1.0]) == [3.0, 1.0]
