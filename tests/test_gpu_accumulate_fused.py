"""Gradient accumulation (qlora_linear_bwd_accumulate) and the fused gate/up
call (two adapters side by side over N = 2 x 14336), against the oracle."""
import numpy as np
import pytest

import oracle
from qlora_fine_tuning_gb300 import binding, synth

from harness import GpuLayer, TOL, compare, dev, dev_bf16, host_bits, oracle_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.lib()
    yield


def _bwd_acc(g, dY, X, XA):
    li = g.li
    binding.qlora_linear_bwd_accumulate(dY, X, XA, li.M, g.w, g.A, g.B, li.r, g.seg, li.s, g.dX, g.dA, g.dB,
                                        g.ws, g.ws_bytes)


# (M, N, K, r, seg): a small case whose splits form clusters, a multi-adapter
# case and a case with one split per tile
ACC = [(300, 512, 256, 16, None), (200, 320, 128, 16, (128, 128, 64)), (8192, 1024, 1024, 64, None)]


@pytest.mark.parametrize("M,N,K,r,seg", ACC)
def test_accumulate_adds_two_micro_batches(M, N, K, r, seg):
    import torch
    li1 = synth.make_linear(M, N, K, r, 0.5, seg_n=seg, seed=41)
    # the second micro-batch shares the layer (W, A, B) and brings its own X, dY
    li2 = synth.make_linear(M, N, K, r, 0.5, seg_n=seg, seed=41, stream=1)
    li2 = synth.LinearInputs(M=M, N=N, K=K, r=r, s=li1.s, seg_n=li1.seg_n, idx=li1.idx, absmax=li1.absmax,
                             codebook=li1.codebook, X=li2.X, A=li1.A, B=li1.B, dY=li2.dY)
    g = GpuLayer(li1)
    g.forward()
    g.backward()
    first = g.results()
    X2, dY2 = dev_bf16(li2.X), dev_bf16(li2.dY)
    XA2 = torch.empty_like(g.XA)
    binding.qlora_linear_fwd(X2, M, g.w, g.A, g.B, r, g.seg, li1.s, g.Y, XA2, g.ws, g.ws_bytes)
    _bwd_acc(g, dY2, X2, XA2)
    g.check()
    got = g.results()
    ref1, ref2 = oracle_full(li1), oracle_full(li2)
    compare({"dA": got["dA"], "dB": got["dB"], "dX": got["dX"]},
            {"dA": ref1["dA"] + ref2["dA"], "dB": ref1["dB"] + ref2["dB"], "dX": ref2["dX"]},
            keys=("dA", "dB", "dX"))
    assert not np.array_equal(got["dA"], first["dA"])


def test_accumulate_onto_zeros_equals_overwrite_and_empty_batch_is_a_no_op():
    li = synth.make_linear(256, 384, 256, 16, 1.0, seed=43)
    g = GpuLayer(li)
    g.forward()
    g.backward()
    ref = g.results()
    g.dA.zero_()
    g.dB.zero_()
    _bwd_acc(g, g.dY, g.X, g.XA)
    got = g.results()
    assert np.array_equal(got["dA"], ref["dA"]) and np.array_equal(got["dB"], ref["dB"])
    binding.qlora_linear_bwd_accumulate(g.dY, g.X, g.XA, 0, g.w, g.A, g.B, li.r, None, li.s, g.dX, g.dA, g.dB,
                                        g.ws, g.ws_bytes)
    again = g.results()
    assert np.array_equal(again["dA"], ref["dA"]) and np.array_equal(again["dB"], ref["dB"])


def test_row_shards_accumulate_to_the_full_batch():
    """Data-parallel stand-in on one GPU: the backward of the first half of the
    rows, then the second half accumulated into the same dA, dB, equals the
    full batch's gradients (to 2e-3: the halves pick other split counts, so G can
    round differently in bf16)."""
    import torch
    li = synth.make_linear(640, 512, 384, 16, 0.5, seed=53)
    full = GpuLayer(li)
    full.forward()
    full.backward()
    full.check()
    ref = full.results()
    h = 320
    parts = []
    for rows in (slice(0, h), slice(h, li.M)):
        parts.append(synth.LinearInputs(M=h, N=li.N, K=li.K, r=li.r, s=li.s, seg_n=li.seg_n, idx=li.idx,
                                        absmax=li.absmax, codebook=li.codebook, X=li.X[rows], A=li.A, B=li.B,
                                        dY=li.dY[rows]))
    g = GpuLayer(parts[0])
    g.forward()
    g.backward()
    g2 = GpuLayer(parts[1])
    g2.forward()
    binding.qlora_linear_bwd_accumulate(g2.dY, g2.X, g2.XA, h, g2.w, g2.A, g2.B, li.r, None, li.s, g2.dX, g.dA, g.dB,
                                        g2.ws, g2.ws_bytes)
    g2.check()
    got = g.results()
    compare({"dA": got["dA"], "dB": got["dB"]}, {"dA": ref["dA"], "dB": ref["dB"]}, keys=("dA", "dB"), tol=2e-3)
    # and against the oracle's full batch
    compare({"dA": got["dA"], "dB": got["dB"]}, oracle_full(li), keys=("dA", "dB"))


def test_accumulate_without_dx_leaves_dx_untouched():
    import torch
    li = synth.make_linear(192, 256, 128, 8, 2.0, seed=47)
    g = GpuLayer(li)
    g.forward()
    g.dX.fill_(3.0)
    g.dA.zero_()
    g.dB.zero_()
    binding.qlora_linear_bwd_accumulate(g.dY, g.X, g.XA, li.M, g.w, g.A, g.B, li.r, None, li.s, None, g.dA, g.dB,
                                        g.ws, g.ws_bytes)
    g.check()
    got = g.results()
    assert np.all(got["dX"] == 3.0)
    ref = oracle_full(li)
    compare(got, ref, keys=("dA", "dB"))


def test_fused_gate_up_forward_equals_two_separate_calls():
    """One two-adapter call over N = 2 x 14336 against the gate and up calls
    made separately: XA and Y are the same numbers, bit for bit (every tile
    sums the same products in the same order)."""
    import torch
    label, kw = synth.WORKLOADS["llama3-8b-mlp-fused-gateup-m8192-4096x2x14336-r64"][0]
    li = synth.make_linear(seed=0, stream=0, **kw)
    g = GpuLayer(li)
    g.forward()
    g.check()
    fused = g.results()
    N1, r, K = li.seg_n[0], li.r, li.K
    for part in range(2):
        rows = slice(part * N1, (part + 1) * N1)
        idx = np.ascontiguousarray(li.idx.reshape(li.N, K // 2)[rows])
        am = np.ascontiguousarray(li.absmax.reshape(li.N, K // 64)[rows]).reshape(-1)
        A = np.ascontiguousarray(li.A[:, part * r:(part + 1) * r])
        B = np.ascontiguousarray(li.B[:, rows])
        sub = synth.LinearInputs(M=li.M, N=N1, K=K, r=r, s=li.s, seg_n=(N1,), idx=idx, absmax=am,
                                 codebook=li.codebook, X=li.X, A=A, B=B, dY=li.dY[:, rows])
        gs = GpuLayer(sub)
        gs.forward()
        gs.check()
        one = gs.results()
        assert np.array_equal(one["Y"], fused["Y"][:, rows])
        assert np.array_equal(one["XA"], fused["XA"][:, part * r:(part + 1) * r])
        del gs
        torch.cuda.empty_cache()
