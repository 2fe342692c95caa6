"""The parity comparison itself (no GPU): it accepts the rounding a correct
bf16 kernel makes and rejects a wrong tile or a single wrong element, which
one global Frobenius norm over a large output would hide."""
import numpy as np
import pytest

import oracle
from harness import TILES_FULL, TILES_SAMPLED, compare, sample_indices
from qlora_fine_tuning_gb300 import synth


def _ref(seed=0, shape=(512, 640)):
    return np.random.default_rng(seed).standard_normal(shape)


def _bf16_round(x):
    return oracle.bf16_to_f64(synth.to_bf16_bits(x.astype(np.float32)))


def test_bf16_rounded_output_passes():
    ref = {"Y": _ref(0), "dX": _ref(1)}
    got = {k: _bf16_round(v) for k, v in ref.items()}
    errs = compare(got, ref, keys=("Y", "dX"))
    assert max(errs.values()) < 4e-3


def test_one_wrong_element_fails_although_the_global_norm_passes():
    ref = {"Y": _ref(2)}
    got = {"Y": _bf16_round(ref["Y"])}
    got["Y"][300, 17] += 1.0   # 1/128 of its tile's norm: only the element bound sees it
    assert oracle.rel_fro(got["Y"], ref["Y"]) < 1e-2
    with pytest.raises(AssertionError, match="out of bounds"):
        compare(got, ref, keys=("Y",))


def test_one_wrong_tile_fails_although_the_global_norm_passes():
    ref = {"dX": _ref(3, (2048, 2048))}
    got = {"dX": ref["dX"].copy()}
    got["dX"][128:256, 1024:1152] *= 1.1   # one tile of 256, scaled by 10%
    assert oracle.rel_fro(got["dX"], ref["dX"]) < 1e-2
    with pytest.raises(AssertionError, match="tile"):
        compare(got, ref, keys=("dX",))


def test_zero_reference_tile_needs_exact_zeros():
    ref = {"dA": np.zeros((256, 64))}
    ref["dA"][128:] = _ref(4, (128, 64))
    got = {"dA": ref["dA"].copy()}
    compare(got, ref, keys=("dA",))
    got["dA"][3, 5] = 1e-30
    with pytest.raises(AssertionError):
        compare(got, ref, keys=("dA",))


def test_samples_cover_every_tile():
    li = synth.LinearInputs(M=8192 + 100, N=14336, K=4096, r=64, s=0.25, seg_n=(14336,), idx=None, absmax=None,
                            codebook=None, X=None, A=None, B=None, dY=None)
    rows, kidx, Jidx, cidx, nidx = sample_indices(li)
    assert set(range(0, li.M, 256)) <= set(256 * (m // 256) for m in rows) | {0}
    assert {m // 256 for m in rows} == set(range((li.M + 255) // 256))
    assert {k // 128 for k in kidx} == set(range(li.K // 128))
    assert {n // 128 for n in nidx} == set(range(li.N // 128))
    assert Jidx == list(range(li.R)) and cidx == list(range(li.r))
    assert set(TILES_FULL) == set(TILES_SAMPLED)
