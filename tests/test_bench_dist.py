"""The benchmark's multi-rank plumbing on the CPU: two gloo ranks (the same
code path torchrun drives on GPUs, where each rank runs its own replica of
the workload and only a barrier and a max of the timed region cross ranks)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    dist, r, w, local = bench.dist_setup()
    assert dist is not None and r == rank and w == world and local == rank
    bench.dist_barrier(dist)
    t = bench.dist_max(dist, 10.0 * (rank + 1))  # rank-local "elapsed ms"
    out[rank] = t
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    assert dict(out) == {0: 20.0, 1: 20.0}


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    env = {k: os.environ.pop(k) for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK") if k in os.environ}
    try:
        dist, rank, world, local = bench.dist_setup()
        assert dist is None and rank == 0 and world == 1
        assert bench.dist_max(None, 3.5) == 3.5
    finally:
        os.environ.update(env)
