"""The multi-replica reduction of bench.py (the slowest rank's time, every rank's
bytes) in world-size-2 process groups over gloo, on CPU."""

import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, nbytes = bench.reduce_over_ranks(1.5 + rank, 1000 * (rank + 1), dist, "cpu")
        results[rank] = (ms, nbytes)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_reduce_over_two_gloo_ranks():
    world = 2
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), results), nprocs=world, join=True)
        got = dict(results)
    # every rank sees the same whole-job figure: max time, summed bytes
    assert got == {0: (2.5, 3000), 1: (2.5, 3000)}


def test_single_process_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(0.25, 123) == (0.25, 123)
