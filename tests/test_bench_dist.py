"""The benchmark's multi-rank host logic on CPU: two gloo ranks, each timing
its own replica, agree on the slowest rank's time through max_over_ranks, and
the launch environment is read from RANK / WORLD_SIZE / LOCAL_RANK."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    dev = torch.device("cpu")
    bench.barrier(w, dev)
    slowest = bench.max_over_ranks(10.0 * (rank + 1), w, dev)  # rank 1 is the slow one
    out[rank] = slowest
    dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 20.0, 1: 20.0}


def test_single_rank_needs_no_process_group(monkeypatch):
    import bench

    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_setup() == (0, 1, 0)
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
