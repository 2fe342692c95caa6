"""qlora_linear_xa_static: XA = X A for callers that cannot allocate device
memory (for example a plug-in whose host application owns every device
allocation) and so cannot pass the workspace the other entry points need.
Its scratch is the library's static device array.  This file is collected
last on purpose: if it fails, a run that stops at the first failure has
already run every other test."""
import numpy as np
import pytest

import oracle
from qlora_fine_tuning_gb300 import binding, synth

from harness import TOL, GpuLayer, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.lib()
    yield


def _reference_xa(li):
    """XA_save written by the existing forward entry point."""
    g = GpuLayer(li)
    g.forward()
    g.check()
    return oracle.bf16_to_f64(host_bits(g.XA)[: li.M]), g


def test_static_scratch_xa_matches_forward_on_two_calls_in_a_row():
    import torch
    # first call: three adapters side by side (R = 48), ragged M
    li1 = synth.make_linear(1000, 512, 1024, 16, 0.5, seg_n=(256, 128, 128), seed=31)
    ref1, g1 = _reference_xa(li1)
    # second call: a shape whose rows need several chunks of the static array
    li2 = synth.make_linear(8192, 256, 14336, 64, 0.25, seed=32)
    ref2, g2 = _reference_xa(li2)

    out1 = torch.empty((li1.M, li1.R), dtype=torch.bfloat16, device="cuda")
    out2 = torch.empty((li2.M, li2.R), dtype=torch.bfloat16, device="cuda")
    binding.qlora_linear_xa_static(g1.X, li1.M, li1.K, g1.A, li1.R, out1)
    binding.qlora_linear_xa_static(g2.X, li2.M, li2.K, g2.A, li2.R, out2)
    torch.cuda.synchronize()
    got1 = oracle.bf16_to_f64(host_bits(out1))
    got2 = oracle.bf16_to_f64(host_bits(out2))
    assert oracle.rel_fro(got1, ref1) <= TOL
    assert oracle.rel_fro(got2, ref2) <= TOL
    # the same kernels, split count and tile order: identical values
    assert np.array_equal(got1, ref1) and np.array_equal(got2, ref2)

    # calling again reuses the array, which still holds the last call's data
    binding.qlora_linear_xa_static(g1.X, li1.M, li1.K, g1.A, li1.R, out1)
    torch.cuda.synchronize()
    assert np.array_equal(oracle.bf16_to_f64(host_bits(out1)), ref1)


def test_static_scratch_rejects_sizes_beyond_its_array():
    with pytest.raises(binding.QloraError) as e:
        binding.qlora_linear_xa_static(0x10000, 128, 16384, 0x10000, 256, 0x10000)
    assert e.value.status == binding.WORKSPACE
