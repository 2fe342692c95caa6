"""Data-parallel step on CPU with two gloo ranks.

The layer is row-independent: a rank that holds a shard of the tokens (rows
of X and dY) computes its own rows of Y and dX and partial dA, dB; one sum
all-reduce of dA and dB per linear gives the full-batch adapter gradients.
Each rank runs the same step function bench.py runs under torchrun
(qlora_fine_tuning_gb300.dp.data_parallel_step, its reducer started after
every backward), with the oracle standing in for the GPU forward and
backward; the reduced result must equal the oracle on the whole batch.  The
bench's max-over-ranks timing reduction is checked too.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

LAYERS = [(10, 24, 64, 4, 0.5, (16, 8)), (7, 32, 128, 8, 2.0, None), (12, 16, 64, 4, 1.0, None)]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _layer(i):
    from qlora_fine_tuning_gb300 import synth
    M, N, K, r, s, seg = LAYERS[i]
    return synth.make_linear(M, N, K, r, s, seg_n=seg, seed=9 + i)


def _operands(li):
    import oracle
    _, w16 = oracle.dequant(li.idx, li.absmax, li.codebook, li.N, li.K)
    return (oracle.bf16_to_f64(li.X), oracle.bf16_to_f64(w16), oracle.bf16_to_f64(li.A), oracle.bf16_to_f64(li.B),
            oracle.bf16_to_f64(li.dY))


def _rank_main(rank, world, port, out_q):
    import torch
    import torch.distributed as dist

    import oracle
    from qlora_fine_tuning_gb300.dp import AdapterGradReducer, data_parallel_step

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        state = []
        for i in range(len(LAYERS)):
            li = _layer(i)
            X, Wd, A, B, dY = _operands(li)
            rows = np.array_split(np.arange(li.M), world)[rank]
            state.append({"li": li, "X": X[rows], "Wd": Wd, "A": A, "B": B, "dY": dY[rows], "rows": rows})

        def forward(i):
            s = state[i]
            seg = None if len(s["li"].seg_n) == 1 else s["li"].seg_n
            s["XA"], s["Y"] = oracle.forward_rows(s["X"], s["Wd"], s["A"], s["B"], s["li"].r, s["li"].s, seg_n=seg)

        def backward(i):
            s = state[i]
            li = s["li"]
            seg = None if len(li.seg_n) == 1 else li.seg_n
            _, s["dX"] = oracle.backward_dx_rows(s["dY"], s["Wd"], s["A"], s["B"], li.r, li.s, seg_n=seg)
            s["dA"] = torch.from_numpy(oracle.backward_da(s["X"], s["dY"], s["B"], li.r, li.s, seg_n=seg))
            s["dB"] = torch.from_numpy(oracle.backward_db(s["X"], s["dY"], s["A"], li.r, li.s, seg_n=seg))

        reducer = AdapterGradReducer()
        assert reducer.world == world
        data_parallel_step(len(LAYERS), forward, backward, lambda i: [state[i]["dA"], state[i]["dB"]], reducer)
        t = torch.tensor([float(rank + 1)], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)  # the bench's max-over-ranks timing reduction
        dist.barrier()
        out_q.put((rank, [(s["rows"].tolist(), s["Y"], s["dX"], s["dA"].numpy(), s["dB"].numpy()) for s in state],
                   float(t.item())))
    finally:
        dist.destroy_process_group()


def test_two_rank_step_all_reduces_to_the_full_batch():
    import oracle

    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=180) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0

    fulls = []
    for i in range(len(LAYERS)):
        li = _layer(i)
        X, Wd, A, B, dY = _operands(li)
        fulls.append(oracle.linear_full(X, Wd, A, B, dY, li.r, li.s, seg_n=None if len(li.seg_n) == 1 else li.seg_n))
    for rank, layers, tmax in res:
        assert tmax == float(world)
        for i, (rows, Y, dX, dA, dB) in enumerate(layers):
            full = fulls[i]
            assert np.array_equal(Y, full["Y"][rows])
            assert np.array_equal(dX, full["dX"][rows])
            assert np.allclose(dA, full["dA"], rtol=1e-12, atol=1e-14)
            assert np.allclose(dB, full["dB"], rtol=1e-12, atol=1e-14)


def test_single_rank_reducer_is_a_no_op():
    import torch
    from qlora_fine_tuning_gb300.dp import AdapterGradReducer, data_parallel_step

    calls = []
    red = AdapterGradReducer()
    assert red.world == 1
    g = torch.ones(3)
    data_parallel_step(2, lambda i: calls.append(("f", i)), lambda i: calls.append(("b", i)), lambda i: [g], red)
    assert calls == [("f", 0), ("f", 1), ("b", 1), ("b", 0)]
    assert torch.equal(g, torch.ones(3))
