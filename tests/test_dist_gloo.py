"""The benchmark's multi-rank logic on CPU (gloo, world size 2): every rank
runs its own replica, the ranks meet in a barrier and take the max of their
elapsed times. No data-path collective exists."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(world)
    out[rank] = bench.reduce_max(1.5 + rank, world)
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_reduce_max_and_barrier_world_2():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.25, 1) == 3.25
    bench.barrier(1)
