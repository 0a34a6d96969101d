"""The host side of `bench.py --gpus N` (N > 1) on CPU: world-size-2 `gloo`
process groups, rendezvous on 127.0.0.1.  The benchmark times every rank
between two barriers and reports the maximum over ranks; each rank runs its
own replica of the op (no collective on the data path)."""

import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # every rank contributes its own elapsed time; all see the maximum
        slowest = bench.max_over_ranks(0.25 * (rank + 1), world, torch.device("cpu"))
        bench.barrier(world)
        q.put((rank, slowest))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_barrier_and_max_over_ranks_with_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    try:
        results = sorted(q.get(timeout=90) for _ in range(world))
    finally:
        for p in procs:
            p.join(timeout=30)
    assert all(p.exitcode == 0 for p in procs)
    assert results == [(0, 0.5), (1, 0.5)]


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import torch

    import bench

    bench.barrier(1)
    assert bench.max_over_ranks(1.5, 1, torch.device("cpu")) == 1.5
