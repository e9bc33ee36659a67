"""The multi-rank host logic of bench.py on CPU: two gloo ranks, no GPU.

With N GPUs every rank runs its own replica of the workload (heads and batches
are independent, so the data path exchanges nothing); only the timing is
combined: the reported time is the maximum over ranks.
"""
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
    import bench
    r, w = bench.dist_init("gloo")
    assert (r, w) == (rank, world)
    bench.barrier()
    mx = bench.max_over_ranks(10.0 + 5.0 * rank)
    out[rank] = (mx, bench.replica_seed(rank))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_distinct_replicas():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 15.0
    assert out[0][1] != out[1][1]


def test_single_rank_is_identity(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    assert bench.dist_env() == (0, 1, 0)
    assert bench.max_over_ranks(3.5) == 3.5
