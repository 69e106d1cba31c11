"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): every rank
runs its own replica of the workload; the job time is the maximum over ranks
and the throughput counts the tokens of all ranks."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        # rank-dependent "step times": the slowest replica must win everywhere
        got = bench.max_over_ranks([1.0 + rank, 5.0 - 3 * rank, 2.5], "cpu")
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(world):
        assert res[r] == [2.0, 5.0, 2.5]


def test_max_over_ranks_single_process_is_identity():
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks([3, 1.5], "cpu") == [3.0, 1.5]
