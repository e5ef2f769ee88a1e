"""Multi-process host logic of bench.py on CPU: world_size 2 over gloo.

Heads are independent problems, so ranks share no data; the only
cross-rank steps are the timing reduction (slowest rank) and, for a
strong-scaling split, the partition of heads.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # timing reduction: rank r "took" (r + 1) * 1.5 ms per step
        ms = (rank + 1) * 1.5
        total, launch = bench.reduce_max([ms, ms / 2], world, device="cpu")
        value = bench.aggregate_tflops(2.0e12, total, world)
        # head sharding: gather every rank's slice of 37 heads
        start, stop = bench.shard_heads(37, rank, world)
        slices = [None] * world
        dist.all_gather_object(slices, (start, stop))
        out[rank] = (total, launch, value, slices)
    finally:
        dist.destroy_process_group()


def test_two_ranks_reduce_and_shard():
    world = 2
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(worker, args=(world, free_port(), out), nprocs=world, join=True)
    for rank in range(world):
        total, launch, value, slices = out[rank]
        assert total == 3.0 and launch == 1.5                  # the slowest rank's times
        assert abs(value - world * 2.0e12 / 3.0e-3 / 1e12) < 1e-9
        covered = sorted(h for a, b in slices for h in range(a, b))
        assert covered == list(range(37))                     # every head exactly once
        assert max(b - a for a, b in slices) - min(b - a for a, b in slices) <= 1


def test_single_rank_is_identity():
    assert bench.reduce_max([1.0, 2.0], 1) == [1.0, 2.0]
    assert bench.shard_heads(5, 0, 1) == (0, 5)
