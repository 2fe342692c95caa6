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

from harness import TOL, GpuLayer, compare, host_bits, oracle_operands

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


def _oracle_xa(li):
    X, Wd, A, B, _ = oracle_operands(li)
    seg = None if len(li.seg_n) == 1 else li.seg_n
    xa, _ = oracle.forward_rows(X, Wd, A, B, li.r, li.s, rows=list(range(li.M)), seg_n=seg)
    return xa


def _static_xa(li, g):
    import torch
    out = torch.empty((li.M, li.R), dtype=torch.bfloat16, device="cuda")
    binding.qlora_linear_xa_static(g.X, li.M, li.K, g.A, li.R, out)
    torch.cuda.synchronize()
    return oracle.bf16_to_f64(host_bits(out))


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
    # and within the bound of the CPU oracle itself (tensor, every tile, every element)
    compare({"XA": got1}, {"XA": _oracle_xa(li1)}, keys=("XA",))

    # calling again reuses the array, which still holds the last call's data
    binding.qlora_linear_xa_static(g1.X, li1.M, li1.K, g1.A, li1.R, out1)
    torch.cuda.synchronize()
    assert np.array_equal(oracle.bf16_to_f64(host_bits(out1)), ref1)
    assert binding.qlora_linear_xa_static_status() == binding.OK


# R = n_seg * r: 8 and 24 leave rows of the 16-row operand tile to the TMA zero
# fill; 128 and 256 use other tile widths than the rank-64 cases above
@pytest.mark.parametrize("M,N,K,r,seg", [(300, 256, 512, 8, None), (257, 320, 320, 8, (128, 128, 64)),
                                         (384, 256, 1024, 128, None), (200, 384, 256, 128, (256, 128))])
def test_static_scratch_xa_narrow_and_wide_ranks(M, N, K, r, seg):
    li = synth.make_linear(M, N, K, r, 1.0, seg_n=seg, seed=M + r)
    ref, g = _reference_xa(li)
    got = _static_xa(li, g)
    assert np.array_equal(got, ref)
    compare({"XA": got}, {"XA": _oracle_xa(li)}, keys=("XA",))


def test_static_scratch_reports_a_wait_that_ran_out():
    """A stalled launch is reported by the status query (and only once); the
    next call on the same context is correct."""
    li = synth.make_linear(256, 256, 512, 16, 1.0, seed=35)
    ref, g = _reference_xa(li)
    binding.qlora_set_wait_limit_ns(50_000_000)
    try:
        binding.qlora_debug_stall_next_launch("gemm_xa_static")
        _static_xa(li, g)
        assert binding.qlora_linear_xa_static_status() == binding.TIMEOUT
        assert binding.qlora_linear_xa_static_status() == binding.OK
        assert np.array_equal(_static_xa(li, g), ref)
        assert binding.qlora_linear_xa_static_status() == binding.OK
    finally:
        binding.qlora_debug_stall_next_launch(None)
        binding.qlora_set_wait_limit_ns(2_000_000_000)


def test_static_scratch_rejects_sizes_beyond_its_array():
    with pytest.raises(binding.QloraError) as e:
        binding.qlora_linear_xa_static(0x10000, 128, 16384, 0x10000, 256, 0x10000)
    assert e.value.status == binding.WORKSPACE
