"""Three ways to produce the bf16 weight the base GEMMs read:

* "rankr" (QLORA_DQ_IN_RANKR=1; the default from 8192 tokens on): the rank-r
  GEMM launch before each base GEMM (XA in the forward, G in the backward)
  writes the row-major Wd from spare warps;
* "separate" (QLORA_DQ_IN_RANKR=0; the default below 8192 tokens): a
  dequantiser launch of its own;
* "fused" (QLORA_FUSED_DQ=1): the pair GEMM expands the 4-bit weight into its
  operand tiles, no Wd at all (a forward that cannot use the pair GEMM takes
  its Wd from the XA launch).

All three are the same fp32 product and bf16 rounding as dequant_4bit and
leave the MMA order unchanged, so Y, dX, dA, dB and XA must be bit-identical
across them; each must also meet the oracle bound."""
import numpy as np
import pytest

from qlora_fine_tuning_gb300 import binding, synth

from harness import GpuLayer, check_sampled, compare, oracle_full

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.lib()
    yield


MODES = {"rankr": {"QLORA_DQ_IN_RANKR": "1"}, "separate": {"QLORA_DQ_IN_RANKR": "0"},
         "fused": {"QLORA_FUSED_DQ": "1", "QLORA_DQ_IN_RANKR": "1"}}


def _run(li, mode, monkeypatch):
    for k in ("QLORA_FUSED_DQ", "QLORA_DQ_IN_RANKR"):
        monkeypatch.delenv(k, raising=False)
    for k, v in MODES[mode].items():
        monkeypatch.setenv(k, v)
    g = GpuLayer(li)
    binding.qlora_profiler_enable(True)
    binding.qlora_profiler_collect()
    g.forward()
    g.backward()
    g.check()
    ran = {name for name, _, _ in binding.qlora_profiler_collect()}
    binding.qlora_profiler_enable(False)
    # only the "separate" mode launches the row-major dequantiser
    assert ("dequant4" in ran) == (mode == "separate"), ran
    return g.results()


@pytest.mark.parametrize("M,N,K,r,s,seg", [
    (256, 1024, 1024, 8, 2.0, None),
    (300, 512, 512, 64, 0.25, None),              # ragged M
    (200, 1024, 512, 16, 1.0, (512, 256, 256)),   # three adapters
    (2048, 2560, 512, 16, 1.0, None),             # several tiles per CTA pair
    (100, 136, 192, 16, 0.5, None),               # weight rows past N (Y) and reduction rows past N (dX)
    (129, 264, 320, 8, 1.0, None),                # K = 320: dX output columns past K; K % 256 != 0
    (257, 776, 448, 32, 2.0, (512, 264)),         # two adapters, ragged last segment, K % 256 != 0
])
def test_weight_paths_match_bitwise_and_oracle(M, N, K, r, s, seg, monkeypatch):
    li = synth.make_linear(M, N, K, r, s, seg_n=seg, seed=M + N)
    res = {m: _run(li, m, monkeypatch) for m in MODES}
    for m in ("separate", "fused"):
        for k in ("Y", "dX", "dA", "dB", "XA"):
            assert np.array_equal(res[m][k], res["rankr"][k]), (m, k)
    compare(res["rankr"], oracle_full(li), keys=("Y", "dX", "dA", "dB", "XA"))


@pytest.mark.parametrize("M,separate", [(4096, True), (8192, False)])
def test_default_weight_path_follows_token_count(M, separate, monkeypatch):
    """Without a switch, the separate dequantiser below 8192 tokens and the
    Wd written by the rank-r launches from 8192 on; both within the oracle
    bounds."""
    for k in ("QLORA_FUSED_DQ", "QLORA_DQ_IN_RANKR"):
        monkeypatch.delenv(k, raising=False)
    li = synth.make_linear(M, 512, 256, 16, 1.0, seed=M + 3)
    g = GpuLayer(li)
    binding.qlora_profiler_enable(True)
    binding.qlora_profiler_collect()
    g.forward()
    g.backward()
    g.check()
    ran = {name for name, _, _ in binding.qlora_profiler_collect()}
    binding.qlora_profiler_enable(False)
    assert ("dequant4" in ran) == separate, ran
    compare(g.results(), oracle_full(li), keys=("Y", "dX", "dA", "dB", "XA"))


@pytest.mark.slow
@pytest.mark.parametrize("name,which", [("llama3-8b-q_proj-m4096-k4096-n4096-r16", 0),
                                        ("llama3-8b-mlp-m8192-4096x14336-r64", 2)])
def test_fused_dequant_full_size(name, which, monkeypatch):
    """Full size with the in-kernel expansion: the q_proj shape and the
    Llama-3-8B down projection (K = 14336: the dX GEMM reads a column band of
    the packed codes)."""
    label, kw = synth.WORKLOADS[name][which]
    li = synth.make_linear(seed=0, stream=which, **kw)
    check_sampled(li, _run(li, "fused", monkeypatch))


@pytest.mark.parametrize("label", ["gemm_fwd", "gemm_dx"])
def test_fused_dequant_stall_reports_timeout(label, monkeypatch):
    monkeypatch.setenv("QLORA_FUSED_DQ", "1")
    binding.qlora_set_wait_limit_ns(50_000_000)
    try:
        li = synth.make_linear(256, 512, 512, 16, 1.0, seed=78)
        g = GpuLayer(li)
        binding.qlora_debug_stall_next_launch(label)
        g.forward()
        g.backward()
        assert binding.qlora_check_device_error(g.ws) == binding.TIMEOUT
        g.forward()
        g.backward()
        assert binding.qlora_check_device_error(g.ws) == binding.OK
        compare(g.results(), oracle_full(li), keys=("Y", "dX", "dA", "dB", "XA"))
    finally:
        binding.qlora_debug_stall_next_launch(None)
        binding.qlora_set_wait_limit_ns(2_000_000_000)


def _random_shapes(n, seed=2024):
    """Seeded shapes within the call's preconditions: ragged M, N % 8 == 0,
    K % 64 == 0, r in 8..128 (multiple of 8), 1-3 adapter segments (all but
    the last a multiple of 128 columns), n_seg * r <= 256."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        M = int(rng.integers(1, 600))
        K = 64 * int(rng.integers(1, 9))
        n_seg = int(rng.integers(1, 4))
        r = 8 * int(rng.integers(1, 17))
        if n_seg * r > 256:
            continue
        heads = [128 * int(rng.integers(1, 4)) for _ in range(n_seg - 1)]
        last = 8 * int(rng.integers(1, 65))
        seg = tuple(heads + [last]) if n_seg > 1 else None
        N = sum(heads) + last
        out.append((M, N, K, r, float(rng.choice([0.25, 0.5, 2.0])), seg))
    return out


@pytest.mark.parametrize("M,N,K,r,s,seg", _random_shapes(12))
def test_random_shapes_all_weight_paths(M, N, K, r, s, seg, monkeypatch):
    """Seeded random shapes through the three weight paths: bit-identical
    results across them and within the oracle bounds."""
    li = synth.make_linear(M, N, K, r, s, seg_n=seg, seed=M * 7 + N)
    res = {m: _run(li, m, monkeypatch) for m in MODES}
    for m in ("separate", "fused"):
        for k in ("Y", "dX", "dA", "dB", "XA"):
            assert np.array_equal(res[m][k], res["rankr"][k]), (m, k)
    compare(res["rankr"], oracle_full(li), keys=("Y", "dX", "dA", "dB", "XA"))
