"""The bench's multi-rank logic on CPU: world size 2 over gloo.  Each rank times its own
replica; rank 0 reports the maximum over ranks and the aggregate throughput."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 10.0 + rank * 5.0                      # rank 1 is slower
    got = bench.max_over_ranks(ms, dist, device="cpu")
    value = bench.aggregate_tokens_per_s(world, 16384, got)
    q.put((rank, got, value))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value in res:
        assert got == pytest.approx(15.0)                       # every rank sees the slowest
        assert value == pytest.approx(2 * 16384 / 15e-3)        # all tokens over the slowest time


def test_single_rank_helpers_without_process_group():
    assert bench.max_over_ranks(7.5, None) == 7.5
    assert bench.aggregate_tokens_per_s(1, 16384, 2.0) == pytest.approx(16384 / 2e-3)
