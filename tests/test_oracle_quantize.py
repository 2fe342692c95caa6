"""Pins of the oracle's 4-bit quantiser (the stored form the path starts from).

Definition ("load_in_4bit" storage, block 64, fp32 absmax, 16-entry codebook):
absmax = max |w| over 64 consecutive elements of the row-major flattening;
code = first i minimising |w/absmax - codebook[i]| in double precision
(t = 0 for an all-zero block).  The oracle is checked against a brute-force
Python loop, exact special cases, an independent midpoint formulation and the
dequantise-after-quantise error bound.
"""
import numpy as np
import pytest

import oracle
from qlora_fine_tuning_gb300 import synth


def _codes(idx, N, K):
    c = np.empty((N, K), dtype=np.int64)
    c[:, 0::2] = idx & 0xF
    c[:, 1::2] = idx >> 4
    return c


def _brute(w, cb):
    N, K = w.shape
    flat = w.reshape(-1, 64)
    codes = np.empty(flat.shape, dtype=np.int64)
    am = np.empty(flat.shape[0], dtype=np.float32)
    for b in range(flat.shape[0]):
        a = max(abs(float(v)) for v in flat[b])
        am[b] = a
        for e in range(64):
            t = 0.0 if a == 0.0 else float(flat[b, e]) / a
            best, dbest = 0, None
            for i in range(16):
                d = abs(t - float(cb[i]))
                if dbest is None or d < dbest:
                    best, dbest = i, d
            codes[b, e] = best
    return codes.reshape(N, K), am


@pytest.mark.parametrize("kind", ["Q", "U"])
def test_matches_brute_force(kind):
    rng = np.random.default_rng(7)
    cb = synth.codebook(kind)
    w = (rng.standard_normal((3, 192)) * 0.02).astype(np.float32)
    w[1, 64:128] = 0.0                      # an all-zero block
    w[2, 5] = np.float32(1e-40)             # a subnormal element
    idx, am = oracle.quantize(w, cb)
    codes, am_ref = _brute(w, cb)
    assert np.array_equal(am, am_ref)
    assert np.array_equal(_codes(idx, 3, 192), codes)


def test_codebook_values_map_to_their_own_code():
    cb = synth.codebook("Q")
    for a in (1.0, 0.02, 3.5):
        w = (np.tile(cb, 4) * np.float32(a)).astype(np.float32).reshape(1, 64)
        w[0, 0] = np.float32(a) * np.float32(-1.0)   # keeps absmax = a
        idx, am = oracle.quantize(w, cb)
        assert am[0] == np.float32(a)
        codes = _codes(idx, 1, 64)[0]
        t = w[0].astype(np.float64) / np.float64(a)
        exact = np.array([np.flatnonzero(cb.astype(np.float64) == v) for v in t], dtype=object)
        for e in range(64):
            if len(exact[e]):
                assert codes[e] == exact[e][0]


def test_exact_midpoint_takes_the_lower_code():
    cb = np.array([(i - 8) / 8 for i in range(16)], dtype=np.float32)   # dyadic: midpoints exact
    w = np.zeros((1, 64), dtype=np.float32)
    w[0, 0] = 1.0                                                      # absmax 1
    mids = [(cb[i] + cb[i + 1]) / 2 for i in range(15)]
    w[0, 1:16] = np.array(mids, dtype=np.float32)
    idx, _ = oracle.quantize(w, cb)
    codes = _codes(idx, 1, 64)[0]
    assert list(codes[1:16]) == list(range(15))


def test_zero_block_takes_code_nearest_zero_lower_on_tie():
    cb = np.linspace(-1, 1, 16).astype(np.float32)          # no zero entry: -1/15 and +1/15 tie
    w = np.zeros((2, 64), dtype=np.float32)
    idx, am = oracle.quantize(w, cb)
    assert np.all(am == 0)
    assert np.all(_codes(idx, 2, 64) == 7)
    cb2 = np.array([(i - 8) / 8 for i in range(16)], dtype=np.float32)   # has an exact zero at 8
    idx, _ = oracle.quantize(w, cb2)
    assert np.all(_codes(idx, 2, 64) == 8)


def test_agrees_with_midpoint_formulation_and_unsorted_codebook():
    rng = np.random.default_rng(3)
    cb = synth.codebook("Q")
    w = (rng.standard_normal((32, 512)) * 0.02).astype(np.float32)
    idx, am = oracle.quantize(w, cb)
    idx_g, am_g = synth.quantize_4bit(w, cb)     # searchsorted on midpoints (independent route)
    assert np.array_equal(am, am_g) and np.array_equal(idx, idx_g)
    perm = rng.permutation(16)
    idx_p, _ = oracle.quantize(w, cb[perm])      # codes follow the permutation
    assert np.array_equal(perm[_codes(idx_p, 32, 512)], _codes(idx, 32, 512))


def test_dequantise_after_quantise_within_half_a_gap():
    rng = np.random.default_rng(5)
    cb = synth.codebook("Q")
    w = (rng.standard_normal((8, 256)) * 0.02).astype(np.float32)
    idx, am = oracle.quantize(w, cb)
    w32, _ = oracle.dequant(idx, am, cb, 8, 256)
    half_gap = np.max(np.diff(cb.astype(np.float64))) / 2
    bound = np.repeat(am.astype(np.float64), 64).reshape(8, 256) * half_gap * (1 + 1e-6)
    assert np.all(np.abs(w32.astype(np.float64) - w.astype(np.float64)) <= bound)
