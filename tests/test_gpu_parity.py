"""CUDA path vs the CPU oracle, through the C ABI, on seeded inputs.

Bar: dequantisation bit-exact; Y, dX, dA, dB within 1e-2 relative Frobenius
error (bf16 operands, fp32 accumulation, bf16 Y/dX); exact zeros where the
definition gives exact zeros.
"""
import numpy as np
import pytest

import oracle
from qlora_fine_tuning_gb300 import binding, synth

from golden_case import expected_dense, load as load_golden
from harness import GpuLayer, TOL, check_sampled, compare, dev, host_bits, oracle_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.lib()
    yield


# --------------------------------------------------------------------------
# dequantisation: bit-exact
# --------------------------------------------------------------------------

@pytest.mark.parametrize("N,K,kind", [(8, 64, "U"), (1024, 1024, "Q"), (24, 4160, "Q"), (4096, 4096, "Q")])
def test_dequant_bit_exact(N, K, kind):
    import torch
    li = synth.make_linear(1, N, K, 8, 1.0, cb_kind=kind, seed=N + K)
    w = binding.make_w4(dev(li.idx), dev(li.absmax), dev(li.codebook), N, K)
    ob = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    of = torch.empty((N, K), dtype=torch.float32, device="cuda")
    keep = (w,)
    binding.dequant_4bit(w, ob, of)
    torch.cuda.synchronize()
    w32, w16 = oracle.dequant(li.idx, li.absmax, li.codebook, N, K)
    assert np.array_equal(host_bits(ob), w16)
    assert np.array_equal(of.cpu().numpy().view(np.uint32), w32.view(np.uint32))
    del keep


def test_dequant_edge_scales_bit_exact():
    import torch
    cb = synth.codebook("Q")
    vals = [0.0, 1.0, 0.02, 2.0 ** -126, float(np.finfo(np.float32).max), float(np.float32(1e-45)), 3.0, 7.5e-39]
    N, K = len(vals), 64
    codes = np.tile(np.arange(16, dtype=np.uint8), K // 16)
    idx = np.tile(codes[0::2] | (codes[1::2] << 4), (N, 1)).astype(np.uint8)
    absmax = np.array(vals, dtype=np.float32)
    w = binding.make_w4(dev(idx), dev(absmax), dev(cb), N, K)
    ob = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    of = torch.empty((N, K), dtype=torch.float32, device="cuda")
    binding.dequant_4bit(w, ob, of)
    torch.cuda.synchronize()
    w32, w16 = oracle.dequant(idx, absmax, cb, N, K)
    assert np.array_equal(host_bits(ob), w16)
    assert np.array_equal(of.cpu().numpy().view(np.uint32), w32.view(np.uint32))


# --------------------------------------------------------------------------
# hand-worked example: exact
# --------------------------------------------------------------------------

def test_golden_closed_form_exact():
    c = load_golden()
    r = 8  # the ABI's smallest rank: pad the rank-1 example with zero columns/rows
    M, K, N = c["M"], c["K"], c["N"]
    A = np.zeros((K, r), dtype=np.float32)
    A[:, 0] = c["A"][:, 0]
    B = np.zeros((r, N), dtype=np.float32)
    B[0] = c["B"][0]
    li = synth.LinearInputs(M=M, N=N, K=K, r=r, s=c["s"], seg_n=(N,), idx=c["idx"], absmax=c["absmax"],
                            codebook=c["codebook"], X=synth.to_bf16_bits(c["X"]), A=synth.to_bf16_bits(A),
                            B=synth.to_bf16_bits(B), dY=synth.to_bf16_bits(c["dY"]))
    g = GpuLayer(li)
    g.forward()
    g.backward()
    g.check()
    got = g.results()
    e = c["expect"]
    _, dx_exp, da_exp = expected_dense(c)
    assert np.array_equal(got["Y"], e["Y"])
    assert np.array_equal(got["XA"][:, :1], e["XA"]) and np.all(got["XA"][:, 1:] == 0)
    assert np.array_equal(got["dX"], dx_exp)
    assert np.array_equal(got["dA"][:, :1], da_exp) and np.all(got["dA"][:, 1:] == 0)
    assert np.array_equal(got["dB"][:1], e["dB"]) and np.all(got["dB"][1:] == 0)


# --------------------------------------------------------------------------
# small shapes, full comparison
# --------------------------------------------------------------------------

SMALL = [
    # M, N, K, r, s, seg_n
    (256, 1024, 1024, 8, 2.0, None),          # the tiny workload
    (1, 64, 64, 8, 1.0, None),                # single row, single k-block
    (100, 136, 192, 16, 0.5, None),           # ragged M and N tails
    (129, 264, 128, 32, 1.0, None),           # one row past a tile, N past a 256 tile
    (300, 512, 256, 64, 0.25, None),
    (130, 384, 128, 128, 2.0, None),          # largest rank: two 64-wide LoRA blocks
    (200, 320, 128, 16, 1.0, (128, 128, 64)), # three adapters side by side
    (64, 384, 192, 8, 2.0, (256, 128)),       # rank 8 with two adapters
    (2048, 2560, 512, 16, 1.0, None),         # more tiles than CTA pairs; rank-r rounds between tiles
    # 81 pair tiles: one full wave of 76 pairs and a 5-tile tail
    (2304, 2304, 1024, 64, 0.25, (1280, 1024)),  # ... in the forward GEMM (two adapters)
    (2304, 1024, 2304, 16, 1.0, None),           # ... in the dX GEMM
    (37, 8, 128, 8, 1.0, None),                  # the narrowest output: 8 columns of one tile
    (96, 264, 192, 16, 0.0, None),               # s = 0: no adapter term; dA, dB exactly zero
]


@pytest.mark.parametrize("M,N,K,r,s,seg", SMALL)
def test_small_shapes_match_oracle(M, N, K, r, s, seg):
    li = synth.make_linear(M, N, K, r, s, seg_n=seg, seed=M * 7 + N)
    g = GpuLayer(li)
    g.forward()
    g.backward()
    g.check()
    got = g.results()
    ref = oracle_full(li)
    compare(got, ref, keys=("Y", "dX", "dA", "dB", "XA"))
    if s == 0.0:
        assert np.all(got["dA"] == 0.0) and np.all(got["dB"] == 0.0)


@pytest.mark.parametrize("variant", ["w_zero", "b_large", "u_codebook"])
def test_lora_visible_variants(variant):
    """W = 0 makes Y and dX pure LoRA; B ~ N(0,1) makes the LoRA term dominate."""
    kw = dict(M=192, N=256, K=256, r=16, s=2.0, seed=11)
    if variant == "w_zero":
        kw["w_zero"] = True
    elif variant == "b_large":
        kw["b_std"] = 1.0
    else:
        kw["cb_kind"] = "U"
    li = synth.make_linear(**kw)
    g = GpuLayer(li)
    g.forward()
    g.backward()
    g.check()
    compare(g.results(), oracle_full(li), keys=("Y", "dX", "dA", "dB", "XA"))


def test_b_zero_gives_exact_zero_da_and_a_zero_gives_exact_zero_db():
    li = synth.make_linear(160, 256, 128, 16, 1.0, b_zero=True, seed=3)
    g = GpuLayer(li)
    g.forward()
    g.backward()
    g.check()
    got = g.results()
    assert np.all(got["dA"] == 0.0)
    li = synth.make_linear(160, 256, 128, 16, 1.0, a_zero=True, seed=4)
    g = GpuLayer(li)
    g.forward()
    g.backward()
    g.check()
    got = g.results()
    assert np.all(got["dB"] == 0.0) and np.all(got["XA"] == 0.0)


def test_empty_batch():
    import torch
    li = synth.make_linear(1, 64, 64, 8, 1.0)
    g = GpuLayer(li)
    g.dA.fill_(7.0)
    g.dB.fill_(7.0)
    binding.qlora_linear_fwd(g.X, 0, g.w, g.A, g.B, 8, None, 1.0, g.Y, g.XA, g.ws, g.ws_bytes)
    binding.qlora_linear_bwd(g.dY, g.X, g.XA, 0, g.w, g.A, g.B, 8, None, 1.0, g.dX, g.dA, g.dB, g.ws, g.ws_bytes)
    torch.cuda.synchronize()
    assert float(g.dA.abs().max()) == 0.0 and float(g.dB.abs().max()) == 0.0


@pytest.mark.parametrize("M,N,K", [(300, 384, 256), (2304, 2304, 2304)])
def test_deterministic_repeat(M, N, K):
    li = synth.make_linear(M, N, K, 16, 1.0, seed=21)
    g = GpuLayer(li)
    g.forward()
    g.backward()
    a = g.results()
    g.forward()
    g.backward()
    b = g.results()
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_rows_independent_of_batch_split():
    """Packed sequences: a row's Y and dX do not depend on the other rows."""
    li = synth.make_linear(512, 256, 256, 16, 1.0, seed=5, with_lengths=True)
    g = GpuLayer(li)
    g.forward()
    g.backward()
    full = g.results()
    off = 0
    for L in li.lengths[:3]:
        sub = synth.LinearInputs(M=int(L), N=li.N, K=li.K, r=li.r, s=li.s, seg_n=li.seg_n, idx=li.idx,
                                 absmax=li.absmax, codebook=li.codebook, X=li.X[off:off + L], A=li.A, B=li.B,
                                 dY=li.dY[off:off + L])
        gs = GpuLayer(sub)
        gs.forward()
        gs.backward()
        part = gs.results()
        assert np.array_equal(part["Y"], full["Y"][off:off + L])
        assert np.array_equal(part["dX"], full["dX"][off:off + L])
        off += int(L)


# --------------------------------------------------------------------------
# the pages' workloads at full size, sampled outputs
# --------------------------------------------------------------------------

FULL = [
    ("llama3-8b-q_proj-m4096-k4096-n4096-r16", 0),
    ("llama3-8b-qkv-gqa-m8192-k4096-n6144-r16x3", 0),
    ("llama3-8b-mlp-m8192-4096x14336-r64", 0),   # gate
    ("llama3-8b-mlp-m8192-4096x14336-r64", 2),   # down
    ("qwen3-14b-mlp-m16384-5120x17408-r16", 0),  # gate
    ("qwen3-14b-mlp-m16384-5120x17408-r16", 2),  # down (K = 17408, N = 5120)
    ("llama3-8b-mlp-fused-gateup-m8192-4096x2x14336-r64", 0),  # gate and up as one two-adapter call
]


@pytest.mark.slow
@pytest.mark.parametrize("name,which", FULL)
def test_full_size_sampled(name, which):
    """Full size, in the launch configuration the benchmark times; the oracle
    evaluates one row of every 256-row tile (all columns), one row of every
    128-row block of dA and one column of every 128-column block of dB."""
    label, kw = synth.WORKLOADS[name][which]
    li = synth.make_linear(seed=0, stream=which, **kw)
    g = GpuLayer(li)
    g.forward()
    g.backward()
    g.check()
    check_sampled(li, g.results())


# --------------------------------------------------------------------------
# stray writes: every output inside a canary-filled allocation
# --------------------------------------------------------------------------

PAD = 512  # elements before and after each output (keeps 16-byte alignment)


def _canary(shape, dtype):
    import torch
    n = int(np.prod(shape))
    if dtype == torch.bfloat16:
        buf = torch.full((n + 2 * PAD,), 0x7FA5, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    else:
        buf = torch.full((n + 2 * PAD,), 0x7FA5A5A5, dtype=torch.int32, device="cuda").view(torch.float32)
    return buf, buf[PAD:PAD + n].view(*shape)


def _pads_intact(buf):
    import torch
    raw = buf.view(torch.int16) if buf.dtype == torch.bfloat16 else buf.view(torch.int32)
    want = 0x7FA5 if buf.dtype == torch.bfloat16 else 0x7FA5A5A5
    head, tail = raw[:PAD], raw[-PAD:]
    return bool((head == want).all()) and bool((tail == want).all())


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("M,N,K,r,seg", [(300, 264, 192, 16, None), (129, 520, 320, 8, (256, 264)),
                                         (2304, 1032, 2304, 64, None)])
def test_no_writes_outside_the_outputs(M, N, K, r, seg, fused, monkeypatch):
    """Ragged M and N tails (partial row and column tiles, a partial last wave
    of pair tiles): Y, XA, dX, dA and dB sit inside canary-filled buffers; the
    canaries before and after each must be untouched and the outputs correct
    -- with the dequantised weight read by TMA and with the 4-bit weight
    expanded inside the GEMM."""
    import torch
    if fused:
        monkeypatch.setenv("QLORA_FUSED_DQ", "1")
    else:
        monkeypatch.delenv("QLORA_FUSED_DQ", raising=False)
    li = synth.make_linear(M, N, K, r, 1.0, seg_n=seg, seed=M + K)
    g = GpuLayer(li)
    bufs = {}
    for name, shape, dt in (("Y", (M, N), torch.bfloat16), ("XA", (M, li.R), torch.bfloat16),
                            ("dX", (M, K), torch.bfloat16), ("dA", (K, li.R), torch.float32),
                            ("dB", (r, N), torch.float32)):
        buf, view = _canary(shape, dt)
        bufs[name] = buf
        setattr(g, name, view)
    g.forward()
    g.backward()
    g.check()
    torch.cuda.synchronize()
    for name, buf in bufs.items():
        assert _pads_intact(buf), f"a write landed outside {name}"
    compare(g.results(), oracle_full(li), keys=("Y", "dX", "dA", "dB", "XA"))
