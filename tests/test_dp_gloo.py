"""Data-parallel decomposition of the layer, on CPU with two gloo ranks.

The layer is row-independent: a rank that holds a shard of the tokens (rows
of X and dY) computes its own rows of Y and dX, and partial dA, dB; one sum
all-reduce of dA and dB gives the full-batch adapter gradients.  Each rank
runs the oracle on its shard; the all-reduced result must equal the oracle
on the whole batch.  This is also the timing plumbing bench.py uses under
torchrun (barrier, max over ranks).
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_q):
    import torch
    import torch.distributed as dist

    import oracle
    from qlora_fine_tuning_gb300 import synth

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        li = synth.make_linear(10, 24, 64, 4, 0.5, seg_n=(16, 8), seed=9)
        rows = np.array_split(np.arange(li.M), world)[rank]
        _, w16 = oracle.dequant(li.idx, li.absmax, li.codebook, li.N, li.K)
        X = oracle.bf16_to_f64(li.X)[rows]
        dY = oracle.bf16_to_f64(li.dY)[rows]
        part = oracle.linear_full(X, oracle.bf16_to_f64(w16), oracle.bf16_to_f64(li.A), oracle.bf16_to_f64(li.B),
                                  dY, li.r, li.s, seg_n=li.seg_n)
        dA = torch.from_numpy(part["dA"].copy())
        dB = torch.from_numpy(part["dB"].copy())
        dist.all_reduce(dA)
        dist.all_reduce(dB)
        t = torch.tensor([float(rank + 1)], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)  # the bench's max-over-ranks timing reduction
        dist.barrier()
        out_q.put((rank, rows.tolist(), part["Y"], part["dX"], dA.numpy(), dB.numpy(), float(t.item())))
    finally:
        dist.destroy_process_group()


def test_two_rank_shards_all_reduce_to_full_batch():
    import oracle
    from qlora_fine_tuning_gb300 import synth

    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0

    li = synth.make_linear(10, 24, 64, 4, 0.5, seg_n=(16, 8), seed=9)
    _, w16 = oracle.dequant(li.idx, li.absmax, li.codebook, li.N, li.K)
    full = oracle.linear_full(oracle.bf16_to_f64(li.X), oracle.bf16_to_f64(w16), oracle.bf16_to_f64(li.A),
                              oracle.bf16_to_f64(li.B), oracle.bf16_to_f64(li.dY), li.r, li.s, seg_n=li.seg_n)
    for rank, rows, Y, dX, dA, dB, tmax in res:
        assert np.array_equal(Y, full["Y"][rows])
        assert np.array_equal(dX, full["dX"][rows])
        assert np.allclose(dA, full["dA"], rtol=1e-12, atol=1e-14)
        assert np.allclose(dB, full["dB"], rtol=1e-12, atol=1e-14)
        assert tmax == float(world)
