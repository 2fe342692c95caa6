"""GPU 4-bit quantiser (quantize_4bit) against the oracle: bit-exact codes and
absmax, fp32 and bf16 weights, through the C ABI."""
import numpy as np
import pytest

import oracle
from qlora_fine_tuning_gb300 import binding, synth

from harness import dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.lib()
    yield


def _gpu_quantize(w: np.ndarray, cb: np.ndarray, as_bf16: bool):
    import torch
    N, K = w.shape
    if as_bf16:
        bits = synth.to_bf16_bits(w)
        W = torch.from_numpy(bits.view(np.int16)).cuda()
        w_ref = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)   # exact widening
    else:
        W = torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32)).cuda()
        w_ref = w
    idx = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
    am = torch.empty((N * K // 64,), dtype=torch.float32, device="cuda")
    c = dev(cb)
    binding.quantize_4bit(W, as_bf16, N, K, c, idx, am)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), am.cpu().numpy(), w_ref


def _check(w, cb, as_bf16):
    idx, am, w_ref = _gpu_quantize(w, cb, as_bf16)
    idx_o, am_o = oracle.quantize(w_ref, cb)
    assert np.array_equal(am.view(np.uint32), am_o.view(np.uint32))
    assert np.array_equal(idx, idx_o)


@pytest.mark.parametrize("as_bf16", [False, True])
@pytest.mark.parametrize("N,K,kind", [(1, 64, "Q"), (3, 192, "U"), (100, 4160, "Q"), (1024, 1024, "U")])
def test_random_weights_bit_exact(N, K, kind, as_bf16):
    rng = np.random.default_rng(N * 131 + K)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    _check(w, synth.codebook(kind), as_bf16)


def test_ties_near_ties_zero_blocks_and_extremes():
    cb = np.array([(i - 8) / 8 for i in range(16)], dtype=np.float32)   # dyadic: exact midpoints
    mids = np.array([(cb[i] + cb[i + 1]) / 2 for i in range(15)], dtype=np.float32)
    w = np.zeros((6, 128), dtype=np.float32)
    w[0, 0] = 1.0
    w[0, 1:16] = mids                                    # exact ties -> lower code
    w[0, 16:31] = np.nextafter(mids, np.float32(np.inf))  # one ulp either side: the double path decides
    w[0, 31:46] = np.nextafter(mids, np.float32(-np.inf))
    w[0, 46:62] = cb                                      # codebook values themselves
    w[0, 62] = -0.0
    w[1, :64] = 0.0                                       # zero block
    w[1, 64:] = np.float32(1e-40) * np.arange(64, dtype=np.float32)  # subnormal block
    w[2, :] = np.float32(3.0e38) * np.sin(np.arange(128, dtype=np.float32))  # near FLT_MAX
    w[3, :] = np.float32(7.0e-39)                         # constant subnormal block (t = 1)
    w[4, :64] = np.float32(0.02)                          # constant block: every t = 1
    w[4, 64:] = np.float32(1.4e-45) * np.arange(64, dtype=np.float32)  # absmax ~9e-44: 1/absmax overflows fp32
    w[5, :] = np.linspace(-1.0, 1.0, 128, dtype=np.float32)
    for as_bf16 in (False, True):
        _check(w, cb, as_bf16)


def test_unsorted_codebook_bit_exact():
    rng = np.random.default_rng(9)
    cb = synth.codebook("Q")[rng.permutation(16)]
    w = (rng.standard_normal((64, 512)) * 0.02).astype(np.float32)
    _check(w, cb, False)


def test_full_size_weight_bit_exact_and_round_trip():
    import torch
    rng = np.random.default_rng(11)
    N, K = 14336, 4096
    w = (rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02))
    cb = synth.codebook("Q")
    idx, am, _ = _gpu_quantize(w, cb, False)
    idx_o, am_o = oracle.quantize(w, cb)
    assert np.array_equal(am, am_o) and np.array_equal(idx, idx_o)
    # the stored form dequantises to the oracle's values (through the product path)
    W4 = binding.make_w4(dev(idx), dev(am), dev(cb), N, K)
    out = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    binding.dequant_4bit(W4, out)
    torch.cuda.synchronize()
    _, w16 = oracle.dequant(idx_o, am_o, cb, N, K)
    assert np.array_equal(out.cpu().view(torch.int16).numpy().view(np.uint16), w16)
