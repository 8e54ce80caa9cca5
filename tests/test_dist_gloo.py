"""Multi-rank logic on CPU, world size 2 over gloo: the bench's (each rank times its own
replica; rank 0 reports the maximum over ranks and the aggregate throughput), and the
data-parallel split of the path itself (token rows sharded across ranks, no exchange in the
forward, one sum of the weight gradients in the backward), checked with the oracle."""
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


def _shard_worker(rank, world, port, q):
    """Each rank runs the oracle's block forward and fused backward on its own shard of token
    rows, then the ranks all-gather the row outputs and all-reduce (sum) the weight gradients:
    the data-parallel split of the path (rows independent in the forward; weight gradients sum
    over tokens), here with the oracle standing in for each rank's kernels."""
    import numpy as np

    import coda_synth as S
    import oracle as O
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    M, H, F = 64, 32, 48
    inp = S.block_inputs(M, H, F, seed=3, with_grad=True)
    x = {k: inp[k].to(torch.float64).numpy() for k in ("O", "R", "W_o", "W_gu", "W_d", "g", "dY")}
    rows = slice(rank * M // world, (rank + 1) * M // world)
    f = O.block_forward(x["O"][rows], x["R"][rows], x["W_o"], x["g"], x["W_gu"], x["W_d"], inp["eps"])
    b = O.block_backward_fused(f, x["O"][rows], x["W_o"], x["g"], x["W_gu"], x["W_d"], x["dY"][rows])
    Y = [torch.zeros_like(torch.from_numpy(f["Y"])) for _ in range(world)]
    dist.all_gather(Y, torch.from_numpy(np.ascontiguousarray(f["Y"])))
    grads = {}
    for k in ("dW_o", "dW_gu", "dW_d", "dg"):
        t = torch.from_numpy(np.ascontiguousarray(b[k]))
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        grads[k] = t.numpy()
    q.put((rank, torch.cat(Y).numpy(), grads))
    dist.barrier()
    dist.destroy_process_group()


def test_row_sharded_chain_equals_the_whole_batch_gloo():
    import numpy as np

    import coda_synth as S
    import oracle as O
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_shard_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=180) for _ in range(world)), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    M, H, F = 64, 32, 48
    inp = S.block_inputs(M, H, F, seed=3, with_grad=True)
    x = {k: inp[k].to(torch.float64).numpy() for k in ("O", "R", "W_o", "W_gu", "W_d", "g", "dY")}
    f = O.block_forward(x["O"], x["R"], x["W_o"], x["g"], x["W_gu"], x["W_d"], inp["eps"])
    b = O.block_backward_fused(f, x["O"], x["W_o"], x["g"], x["W_gu"], x["W_d"], x["dY"])
    for rank, Y, grads in res:
        np.testing.assert_allclose(Y, f["Y"], rtol=1e-12, atol=1e-12)          # rows need no exchange
        for k, v in grads.items():
            np.testing.assert_allclose(v, b[k], rtol=1e-10, atol=1e-12, err_msg=k)   # one sum over ranks
