"""Failure detection without a GPU fault: a kernel whose pipeline stalls gives
up after the wait limit, sets the workspace error flag and frees its tensor
memory; the call reports QLORA_ERR_TIMEOUT and the context stays usable."""
import pytest

from qlora_fine_tuning_gb300 import binding, synth

from harness import GpuLayer, compare, oracle_full

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _short_waits():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.qlora_set_wait_limit_ns(50_000_000)  # 50 ms
    yield
    binding.qlora_debug_stall_next_launch(None)
    binding.qlora_set_wait_limit_ns(2_000_000_000)


@pytest.mark.parametrize("label", ["gemm_xa", "gemm_fwd", "gemm_g", "gemm_dx", "gemm_dadb"])
def test_stalled_pipeline_reports_timeout_and_next_call_is_correct(label):
    li = synth.make_linear(256, 512, 512, 16, 1.0, seed=77)
    g = GpuLayer(li)
    binding.qlora_debug_stall_next_launch(label)
    g.forward()
    g.backward()
    assert binding.qlora_check_device_error(g.ws) == binding.TIMEOUT
    # flag cleared, hook consumed: the same layer now runs normally
    g.forward()
    g.backward()
    assert binding.qlora_check_device_error(g.ws) == binding.OK
    compare(g.results(), oracle_full(li), keys=("Y", "dX", "dA", "dB", "XA"))


@pytest.mark.parametrize("wd_in_rankr", ["0", "1"])
def test_single_cta_fallback_path_matches_oracle(wd_in_rankr, monkeypatch):
    """The forward and dX GEMMs also run on the single-CTA kernel (used when
    adapter segment boundaries are not multiples of 256), with the forward's
    Wd from the separate dequantiser or from the XA launch."""
    monkeypatch.setenv("QLORA_DISABLE_PAIR", "1")
    monkeypatch.setenv("QLORA_DQ_IN_RANKR", wd_in_rankr)
    for M, N, K, r, seg in [(300, 512, 256, 64, None), (129, 264, 128, 32, None)]:
        li = synth.make_linear(M, N, K, r, 0.5, seg_n=seg, seed=M)
        g = GpuLayer(li)
        g.forward()
        g.backward()
        g.check()
        compare(g.results(), oracle_full(li), keys=("Y", "dX", "dA", "dB", "XA"))
