"""The double-buffered reload component (pages: "如何用 Unsloth 和 NVIDIA 让 LLM
训练更快", section 2 双缓冲检查点重载): three steps whose X and dY reach the
device only through the reload buffers, forward and backward of every layer
through the C ABI, each step's outputs against the oracle."""
import numpy as np
import pytest

from qlora_fine_tuning_gb300 import binding, synth
from qlora_fine_tuning_gb300.reload import LayerReload

from harness import GpuLayer, compare, oracle_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.lib()
    yield


LAYERS = [(300, 384, 256, 16, 0.5), (256, 512, 384, 8, 2.0), (200, 256, 512, 16, 1.0)]


def _pinned_bf16(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).pin_memory()


@pytest.mark.parametrize("buffers", [2, 1])
def test_three_steps_through_the_reload_match_the_oracle(buffers):
    import torch
    # two input sets (same layers, other X and dY) alternate over the steps, so
    # a buffer still holding the previous step's data would be caught
    sets = []
    for v in range(2):
        lis = []
        for i, (M, N, K, r, s) in enumerate(LAYERS):
            base = synth.make_linear(M, N, K, r, s, seed=60 + i)
            other = synth.make_linear(M, N, K, r, s, seed=60 + i, stream=1 + v)
            lis.append(synth.LinearInputs(M=M, N=N, K=K, r=r, s=s, seg_n=base.seg_n, idx=base.idx,
                                          absmax=base.absmax, codebook=base.codebook, X=other.X, A=base.A,
                                          B=base.B, dY=other.dY))
        sets.append(lis)
    gls = [GpuLayer(li) for li in sets[0]]  # device weights, adapters, outputs, workspaces
    hosts = [[[_pinned_bf16(li.X), _pinned_bf16(li.dY)] for li in lis] for lis in sets]
    rl = LayerReload([[(li.M, li.K), (li.M, li.N)] for li in sets[0]], torch.bfloat16, buffers=buffers)

    def compute(i, dev):
        X, dY = dev
        g, li = gls[i], gls[i].li
        binding.qlora_linear_fwd(X, li.M, g.w, g.A, g.B, li.r, None, li.s, g.Y, g.XA, g.ws, g.ws_bytes)
        binding.qlora_linear_bwd(dY, X, g.XA, li.M, g.w, g.A, g.B, li.r, None, li.s, g.dX, g.dA, g.dB, g.ws,
                                 g.ws_bytes)

    got_steps = []
    for step in range(3):
        v = step % 2
        for g in gls:
            g.Y.zero_()
            g.dX.zero_()
        rl.run(hosts[v], compute, order=[2, 1, 0])
        torch.cuda.synchronize()
        outs = []
        for i, g in enumerate(gls):
            g.check()
            res = g.results()
            compare(res, oracle_full(sets[v][i]), keys=("Y", "dX", "dA", "dB", "XA"))
            outs.append(res)
        got_steps.append(outs)
    # the same inputs give the same numbers, step after step
    for i in range(len(LAYERS)):
        for k in ("Y", "dX", "dA", "dB"):
            assert np.array_equal(got_steps[0][i][k], got_steps[2][i][k])
