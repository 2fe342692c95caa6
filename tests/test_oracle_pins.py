"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: hand-worked
values, IEEE arithmetic done by numpy / torch, closed forms, the textbook
matrix product (numpy float64 matmul) in the special cases that reduce to it,
the other bracketing of the chain product, and central finite differences of
the scalar <dY, Y>, which are exact up to roundoff because that scalar is
linear in each of X, A and B separately.
"""
import numpy as np
import pytest
import torch

import oracle
from qlora_fine_tuning_gb300 import synth
from golden_case import expected_dense, load as load_golden


def f32_bits(x):
    return np.array([x], dtype=np.float32).view(np.uint32)[0]


def bits_f32(u):
    return float(np.array([u], dtype=np.uint32).view(np.float32)[0])


def torch_bf16_bits(x):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------
# bf16 rounding
# --------------------------------------------------------------------------

@pytest.mark.parametrize("inp,out", [
    (0x3F800000, 0x3F80),  # 1.0 exact
    (0x3F808000, 0x3F80),  # tie, even upper half stays
    (0x3F818000, 0x3F82),  # tie, odd upper half rounds up
    (0x3F808001, 0x3F81),  # just above a tie
    (0x3F807FFF, 0x3F80),  # just below a tie
    (0x80000000, 0x8000),  # -0 keeps its sign
    (0x00000000, 0x0000),
    (0x00000001, 0x0000),  # smallest subnormal rounds to +0
    (0x80008000, 0x8000),  # negative tie toward even (zero)
    (0x7F7FFFFF, 0x7F80),  # FLT_MAX overflows to +inf under RNE
    (0xBF7FFFFF, 0xBF80),  # -0.99999994 -> -1.0
    (0x007FFFFF, 0x0080),  # largest subnormal rounds up to the smallest normal
])
def test_bf16_rne_hand_values(inp, out):
    assert int(oracle.bf16_rne(bits_f32(inp))) == out


def test_bf16_rne_matches_torch_on_random_and_edge_values():
    rng = np.random.default_rng(1)
    u = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    x = u.view(np.float32)
    x = x[np.isfinite(x)]
    edge = np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 1e-45, 1.17549435e-38,
                     0.02, 1.0 / 3.0], dtype=np.float32)
    x = np.concatenate([x[:4000], edge])
    assert np.array_equal(oracle.bf16_rne(x), torch_bf16_bits(x))


# --------------------------------------------------------------------------
# Dequantisation
# --------------------------------------------------------------------------

ABSMAX_SET = [0.0, 1.0, 0.02, 2.0 ** -126, float(np.finfo(np.float32).max), 3.0,
              float(np.float32(1e-45)), 0.5]


@pytest.mark.parametrize("kind", ["Q", "U"])
def test_dequant_exhaustive_codes_times_absmax(kind):
    cb = synth.codebook(kind)
    K = 64
    N = len(ABSMAX_SET) * 16 // 2  # each row holds 64 codes; 16 codes x 4 = 64
    # one row per absmax value; each row cycles through all 16 codes 4 times
    N = len(ABSMAX_SET)
    codes = np.tile(np.arange(16, dtype=np.uint8), K // 16)
    idx = np.tile(codes[0::2] | (codes[1::2] << 4), (N, 1))
    absmax = np.array(ABSMAX_SET, dtype=np.float32)
    w32, w16 = oracle.dequant(idx, absmax, cb, N, K)
    with np.errstate(over="ignore"):
        expect32 = cb[codes][None, :].astype(np.float32) * absmax[:, None].astype(np.float32)
    assert np.array_equal(w32.view(np.uint32), expect32.astype(np.float32).view(np.uint32))
    assert np.array_equal(w16, torch_bf16_bits(expect32))


def test_dequant_nibble_order_and_constant_code():
    cb = synth.codebook("U")
    K, N = 128, 2
    # byte 0xA3: even k -> code 3, odd k -> code 10
    idx = np.full((N, K // 2), 0xA3, dtype=np.uint8)
    absmax = np.ones(N * K // 64, dtype=np.float32)
    w32, _ = oracle.dequant(idx, absmax, cb, N, K)
    assert np.all(w32[:, 0::2] == cb[3]) and np.all(w32[:, 1::2] == cb[10])
    # every code j everywhere gives codebook[j] * absmax
    for j in range(16):
        idx = np.full((N, K // 2), j | (j << 4), dtype=np.uint8)
        am = np.full(N * K // 64, 0.75, dtype=np.float32)
        w32, _ = oracle.dequant(idx, am, cb, N, K)
        assert np.all(w32 == np.float32(cb[j]) * np.float32(0.75))


def test_dequant_block_index_follows_row_major_flattening():
    cb = synth.codebook("U")  # codebook[15] == 1.0 exactly
    N, K = 3, 256
    nb = N * K // 64
    absmax = (2.0 ** -np.arange(nb)).astype(np.float32)
    idx = np.full((N, K // 2), 0xFF, dtype=np.uint8)
    w32, _ = oracle.dequant(idx, absmax, cb, N, K)
    flat = w32.reshape(-1)
    for e in range(N * K):
        assert flat[e] == absmax[e // 64]


# --------------------------------------------------------------------------
# Linear layer
# --------------------------------------------------------------------------

def _rand_problem(M, N, K, r, nseg=1, seed=0, scale_b=1.0):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((M, K))
    Wd = rng.standard_normal((N, K)) * 0.1
    A = rng.standard_normal((K, r * nseg)) * 0.1
    B = rng.standard_normal((r, N)) * scale_b
    dY = rng.standard_normal((M, N))
    return X, Wd, A, B, dY


def test_golden_closed_form():
    c = load_golden()
    e = c["expect"]
    w32, w16 = oracle.dequant(c["idx"], c["absmax"], c["codebook"], c["N"], c["K"])
    wd_exp, dx_exp, da_exp = expected_dense(c)
    wd = oracle.bf16_to_f64(w16)
    assert np.array_equal(wd, wd_exp) and np.array_equal(w32.astype(np.float64), wd_exp)
    out = oracle.linear_full(c["X"], wd, c["A"], c["B"], c["dY"], c["r"], c["s"])
    assert np.array_equal(out["XA"], e["XA"])
    assert np.array_equal(out["Y"], e["Y"])
    assert np.array_equal(out["G"], e["G"])
    assert np.array_equal(out["dX"], dx_exp)
    assert np.array_equal(out["dA"], da_exp)
    assert np.array_equal(out["dB"], e["dB"])


def test_b_zero_reduces_to_textbook_gemm():
    X, Wd, A, B, dY = _rand_problem(5, 24, 64, 4)
    B[:] = 0
    out = oracle.linear_full(X, Wd, A, B, dY, 4, 2.0)
    assert np.allclose(out["Y"], X @ Wd.T, rtol=1e-12, atol=1e-12)
    assert np.allclose(out["dX"], dY @ Wd, rtol=1e-12, atol=1e-12)
    assert np.all(out["dA"] == 0.0)  # G is exactly zero


def test_a_zero_and_w_zero_special_cases():
    X, Wd, A, B, dY = _rand_problem(4, 16, 64, 4, seed=3)
    A0 = np.zeros_like(A)
    out = oracle.linear_full(X, Wd, A0, B, dY, 4, 0.5)
    assert np.allclose(out["Y"], X @ Wd.T, rtol=1e-12, atol=1e-12)
    assert np.all(out["dB"] == 0.0)
    W0 = np.zeros_like(Wd)
    s = 0.25
    out = oracle.linear_full(X, W0, A, B, dY, 4, s)
    # pure LoRA, bracketed the other way: s X (A B)
    assert np.allclose(out["Y"], s * (X @ (A @ B)), rtol=1e-10, atol=1e-12)
    assert np.allclose(out["dX"], s * (dY @ (A @ B).T), rtol=1e-10, atol=1e-12)


def test_bracketing_invariance():
    X, Wd, A, B, dY = _rand_problem(6, 32, 128, 8, seed=4)
    s = 1.5
    out = oracle.linear_full(X, Wd, A, B, dY, 8, s)
    # the oracle computes (X A) B and X^T (dY B^T); compare with X (A B), (X^T dY) B^T
    assert np.allclose(out["Y"] - X @ Wd.T, s * (X @ (A @ B)), rtol=1e-10, atol=1e-12)
    assert np.allclose(out["dA"], s * ((X.T @ dY) @ B.T), rtol=1e-10, atol=1e-12)
    assert np.allclose(out["dB"], s * (A.T @ (X.T @ dY)), rtol=1e-10, atol=1e-12)


def _loss(X, Wd, A, B, dY, r, s, seg_n=None):
    _, y = oracle.forward_rows(X, Wd, A, B, r, s, seg_n=seg_n)
    return float(np.sum(dY * y))


@pytest.mark.parametrize("M,K,N,r,seg_n", [(4, 64, 8, 2, None), (3, 128, 16, 4, (8, 8))])
def test_gradients_match_central_differences(M, K, N, r, seg_n):
    nseg = 1 if seg_n is None else len(seg_n)
    X, Wd, A, B, dY = _rand_problem(M, N, K, r, nseg=nseg, seed=5)
    s = 0.75
    out = oracle.linear_full(X, Wd, A, B, dY, r, s, seg_n=seg_n)
    h = 0.5  # any step is exact for a function linear in the perturbed operand
    for name, T, grad in (("X", X, out["dX"]), ("A", A, out["dA"]), ("B", B, out["dB"])):
        fd = np.zeros_like(T)
        it = np.ndindex(*T.shape)
        for ij in it:
            if name == "X" and M * K > 256 and (ij[1] % 7 != 0):
                fd[ij] = grad[ij]  # subsample the larger case
                continue
            old = T[ij]
            T[ij] = old + h
            lp = _loss(X, Wd, A, B, dY, r, s, seg_n)
            T[ij] = old - h
            lm = _loss(X, Wd, A, B, dY, r, s, seg_n)
            T[ij] = old
            fd[ij] = (lp - lm) / (2 * h)
        scale = max(1.0, float(np.max(np.abs(grad))))
        assert np.max(np.abs(fd - grad)) <= 1e-11 * scale, name


def test_segments_are_independent_adapters():
    seg_n = (16, 8, 8)
    r = 4
    M, K, N = 5, 64, sum(seg_n)
    X, Wd, A, B, dY = _rand_problem(M, N, K, r, nseg=3, seed=6)
    s = 2.0
    full = oracle.linear_full(X, Wd, A, B, dY, r, s, seg_n=seg_n)
    off = 0
    dx_sum = np.zeros((M, K))
    for j, nj in enumerate(seg_n):
        cols = slice(off, off + nj)
        Aj = A[:, j * r:(j + 1) * r]
        part = oracle.linear_full(X, Wd[cols], Aj, B[:, cols], dY[:, cols], r, s)
        assert np.allclose(full["Y"][:, cols], part["Y"], rtol=1e-13, atol=1e-13)
        assert np.allclose(full["dA"][:, j * r:(j + 1) * r], part["dA"], rtol=1e-13, atol=1e-13)
        assert np.allclose(full["dB"][:, cols], part["dB"], rtol=1e-13, atol=1e-13)
        assert np.allclose(full["G"][:, j * r:(j + 1) * r], part["G"], rtol=1e-13, atol=1e-13)
        dx_sum += part["dX"]
        off += nj
    # the base term dY Wd is shared; each part holds its own slice of it
    assert np.allclose(full["dX"], dx_sum, rtol=1e-12, atol=1e-12)


def test_sampled_outputs_equal_full_outputs():
    X, Wd, A, B, dY = _rand_problem(9, 24, 64, 4, seed=7)
    s = 0.5
    full = oracle.linear_full(X, Wd, A, B, dY, 4, s)
    rows = [8, 0, 3]
    xa, y = oracle.forward_rows(X, Wd, A, B, 4, s, rows=rows)
    g, dx = oracle.backward_dx_rows(dY, Wd, A, B, 4, s, rows=rows)
    assert np.array_equal(y, full["Y"][rows]) and np.array_equal(dx, full["dX"][rows])
    da = oracle.backward_da(X, dY, B, 4, s, kidx=[63, 1], Jidx=[3, 0])
    assert np.array_equal(da, full["dA"][np.ix_([63, 1], [3, 0])])
    db = oracle.backward_db(X, dY, A, 4, s, cidx=[2], nidx=[23, 5])
    assert np.array_equal(db, full["dB"][np.ix_([2], [23, 5])])


def test_row_split_rows_identical_and_adapter_grads_add_up():
    X, Wd, A, B, dY = _rand_problem(10, 16, 64, 4, seed=8)
    s = 1.0
    full = oracle.linear_full(X, Wd, A, B, dY, 4, s)
    a = oracle.linear_full(X[:6], Wd, A, B, dY[:6], 4, s)
    b = oracle.linear_full(X[6:], Wd, A, B, dY[6:], 4, s)
    assert np.array_equal(np.vstack([a["Y"], b["Y"]]), full["Y"])
    assert np.array_equal(np.vstack([a["dX"], b["dX"]]), full["dX"])
    assert np.allclose(a["dA"] + b["dA"], full["dA"], rtol=1e-13, atol=1e-14)
    assert np.allclose(a["dB"] + b["dB"], full["dB"], rtol=1e-13, atol=1e-14)


def test_rel_fro_metric():
    assert oracle.rel_fro([3.0, 4.0], [3.0, 4.0]) == 0.0
    assert abs(oracle.rel_fro([3.0, 4.0 + 0.5], [3.0, 4.0]) - 0.1) < 1e-15
    assert oracle.rel_fro([0.0], [0.0]) == 0.0
