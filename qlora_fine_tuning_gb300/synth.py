"""Seeded synthetic inputs for the QLoRA linear layer.

This module is shared by the tests (which feed the same inputs to the CUDA
library and to the CPU oracle) and by the benchmark.  It contains no step of
the layer's own arithmetic: it draws random tensors, rounds them to their
storage types and packs the frozen weight into the 4-bit storage format
offline (the "load_in_4bit" preparation step, which is not part of the
forward/backward path).

Workload shapes follow the pages' fine-tuning examples (Llama-3-8B q_proj,
fused QKV with grouped K/V heads, the Llama-3-8B and Qwen3-14B MLP
projections); value distributions:

  X ~ N(0,1) bf16;  W ~ N(0,0.02) fp32, 4-bit blockwise (64) with fp32 absmax;
  A ~ U(+-1/sqrt(K)) bf16;  B ~ N(0,0.01) bf16;  dY ~ N(0,0.01) bf16.

Random streams come from numpy PCG64 seeded by SeedSequence, spawned in the
fixed order W, X, A, B, dY, lengths.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from statistics import NormalDist
from typing import Optional, Sequence

import numpy as np

BLOCK = 64


# --------------------------------------------------------------------------
# Codebooks (16 sorted fp32 values spanning [-1, 1]; the codebook is an input)
# --------------------------------------------------------------------------

def codebook_uniform() -> np.ndarray:
    """16 evenly spaced values from -1 to 1."""
    return np.linspace(-1.0, 1.0, 16).astype(np.float32)


def codebook_quantile() -> np.ndarray:
    """Normal quantiles at 16 evenly spaced probabilities in [1/32, 31/32],
    divided by the largest magnitude so the values span [-1, 1]."""
    nd = NormalDist()
    p = np.linspace(1.0 / 32.0, 31.0 / 32.0, 16)
    q = np.array([nd.inv_cdf(float(pi)) for pi in p], dtype=np.float64)
    q = q / np.max(np.abs(q))
    return q.astype(np.float32)


def codebook(kind: str = "Q") -> np.ndarray:
    if kind in ("Q", "quantile"):
        return codebook_quantile()
    if kind in ("U", "uniform"):
        return codebook_uniform()
    raise ValueError(f"unknown codebook {kind!r}")


# --------------------------------------------------------------------------
# Storage-type conversions (input preparation)
# --------------------------------------------------------------------------

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def quantize_4bit(w: np.ndarray, cb: np.ndarray, block: int = BLOCK, chunk_rows: int = 256):
    """Pack fp32 W [N,K] as 4-bit codes + fp32 absmax per `block` elements.

    absmax = max |w| over each block of the row-major flattening; each element
    takes the code whose codebook value is nearest w/absmax (fp64 decision,
    the lower code on a tie; a block with absmax 0 takes the code nearest 0).
    Codes are packed two per byte, the even column in the low nibble.
    Requires a sorted codebook.
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    assert K % block == 0 and K % 2 == 0
    cb64 = cb.astype(np.float64)
    assert np.all(np.diff(cb64) > 0), "codebook must be sorted"
    mids = 0.5 * (cb64[1:] + cb64[:-1])
    idx = np.empty((N, K // 2), dtype=np.uint8)
    absmax = np.empty((N * K // block,), dtype=np.float32)
    zero_code = int(np.argmin(np.abs(cb64)))
    for r0 in range(0, N, chunk_rows):
        r1 = min(N, r0 + chunk_rows)
        blk = w[r0:r1].reshape(-1, block)
        am = np.max(np.abs(blk), axis=1)
        absmax[r0 * K // block: r1 * K // block] = am
        am64 = am.astype(np.float64)
        safe = np.where(am64 > 0, am64, 1.0)
        t = blk.astype(np.float64) / safe[:, None]
        codes = np.searchsorted(mids, t, side="left").astype(np.uint8)
        codes[am64 == 0] = zero_code
        codes = codes.reshape(r1 - r0, K)
        idx[r0:r1] = codes[:, 0::2] | (codes[:, 1::2] << np.uint8(4))
    return idx, absmax


# --------------------------------------------------------------------------
# One linear layer's inputs
# --------------------------------------------------------------------------

@dataclass
class LinearInputs:
    M: int
    N: int
    K: int
    r: int
    s: float
    seg_n: tuple
    idx: np.ndarray        # uint8  [N, K/2]
    absmax: np.ndarray     # fp32   [N*K/64]
    codebook: np.ndarray   # fp32   [16]
    X: np.ndarray          # bf16 bits [M, K]
    A: np.ndarray          # bf16 bits [K, nseg*r]
    B: np.ndarray          # bf16 bits [r, N]
    dY: np.ndarray         # bf16 bits [M, N]
    lengths: Optional[np.ndarray] = None
    meta: dict = field(default_factory=dict)

    @property
    def R(self) -> int:
        return self.r * len(self.seg_n)


def _seed_seq(seed: int, stream: int) -> np.random.SeedSequence:
    return np.random.SeedSequence(seed if stream == 0 else [seed, stream])


def packed_lengths(total: int, rng: np.random.Generator, lo: int = 64, hi: int = 2048) -> np.ndarray:
    """Sequence lengths drawn uniformly from [lo, hi] until they cover `total`
    tokens; the last one is truncated so the lengths sum to `total`."""
    out = []
    acc = 0
    while acc < total:
        L = int(rng.integers(lo, hi + 1))
        L = min(L, total - acc)
        out.append(L)
        acc += L
    return np.array(out, dtype=np.int64)


def make_linear(M: int, N: int, K: int, r: int, s: float, seg_n: Optional[Sequence[int]] = None,
                seed: int = 0, stream: int = 0, cb_kind: str = "Q",
                x_std: float = 1.0, w_std: float = 0.02, b_std: float = 0.01,
                dy_std: float = 0.01, w_zero: bool = False, a_zero: bool = False,
                b_zero: bool = False, with_lengths: bool = False, shard: int = 0) -> LinearInputs:
    """One linear's seeded inputs.  `shard` > 0 draws X and dY (the tokens)
    from a stream of their own, keeping W, A and B those of shard 0: the
    token shard of one data-parallel rank."""
    seg = tuple(int(v) for v in (seg_n if seg_n is not None else (N,)))
    assert sum(seg) == N
    R = r * len(seg)
    ss = _seed_seq(seed, stream).spawn(6)
    g_w, g_x, g_a, g_b, g_dy, g_len = (np.random.Generator(np.random.PCG64(s_)) for s_ in ss)
    if shard:
        tx, tdy = np.random.SeedSequence([seed, stream, 1000 + shard]).spawn(2)
        g_x, g_dy = np.random.Generator(np.random.PCG64(tx)), np.random.Generator(np.random.PCG64(tdy))
    cb = codebook(cb_kind)
    if w_zero:
        w = np.zeros((N, K), dtype=np.float32)
    else:
        w = g_w.standard_normal((N, K), dtype=np.float32) * np.float32(w_std)
    idx, absmax = quantize_4bit(w, cb)
    del w
    X = to_bf16_bits(g_x.standard_normal((M, K), dtype=np.float32) * np.float32(x_std))
    bound = 1.0 / np.sqrt(K)
    A = to_bf16_bits(g_a.uniform(-bound, bound, (K, R)).astype(np.float32))
    B = to_bf16_bits(g_b.standard_normal((r, N), dtype=np.float32) * np.float32(b_std))
    dY = to_bf16_bits(g_dy.standard_normal((M, N), dtype=np.float32) * np.float32(dy_std))
    if a_zero:
        A[...] = 0
    if b_zero:
        B[...] = 0
    lengths = packed_lengths(M, g_len) if with_lengths else None
    return LinearInputs(M=M, N=N, K=K, r=r, s=float(s), seg_n=seg, idx=idx, absmax=absmax,
                        codebook=cb, X=X, A=A, B=B, dY=dY, lengths=lengths)


# --------------------------------------------------------------------------
# Workloads (the pages' fine-tuning shapes)
# --------------------------------------------------------------------------

# name -> list of (label, dict of make_linear kwargs)
WORKLOADS = {
    "tiny-m256-k1024-n1024-r8": [
        ("linear", dict(M=256, K=1024, N=1024, r=8, s=2.0)),
    ],
    "llama3-8b-q_proj-m4096-k4096-n4096-r16": [
        ("q_proj", dict(M=4096, K=4096, N=4096, r=16, s=1.0)),
    ],
    "llama3-8b-qkv-gqa-m8192-k4096-n6144-r16x3": [
        ("qkv", dict(M=8192, K=4096, N=6144, r=16, s=1.0, seg_n=(4096, 1024, 1024))),
    ],
    "llama3-8b-mlp-m8192-4096x14336-r64": [
        ("gate", dict(M=8192, K=4096, N=14336, r=64, s=0.25)),
        ("up", dict(M=8192, K=4096, N=14336, r=64, s=0.25)),
        ("down", dict(M=8192, K=14336, N=4096, r=64, s=0.25)),
    ],
    # gate and up as one call: W_gate and W_up stacked, one adapter per half
    "llama3-8b-mlp-fused-gateup-m8192-4096x2x14336-r64": [
        ("gate_up", dict(M=8192, K=4096, N=28672, r=64, s=0.25, seg_n=(14336, 14336))),
        ("down", dict(M=8192, K=14336, N=4096, r=64, s=0.25)),
    ],
    "qwen3-14b-mlp-m16384-5120x17408-r16": [
        ("gate", dict(M=16384, K=5120, N=17408, r=16, s=2.0, with_lengths=True)),
        ("up", dict(M=16384, K=5120, N=17408, r=16, s=2.0, with_lengths=True)),
        ("down", dict(M=16384, K=17408, N=5120, r=16, s=2.0, with_lengths=True)),
    ],
}


def workload(name: str, seed: int = 0, shard: int = 0, **overrides):
    """All linears of a workload; linear i uses random stream i (`shard`: the
    token shard of a data-parallel rank, see make_linear)."""
    out = []
    for i, (label, kw) in enumerate(WORKLOADS[name]):
        kw = dict(kw)
        kw.update(overrides)
        li = make_linear(seed=seed, stream=i, shard=shard, **kw)
        li.meta["label"] = label
        out.append(li)
    return out


def flops_fwd_bwd(M: int, N: int, K: int, r: int, n_seg: int = 1) -> int:
    """Algorithmic FLOPs of one forward + backward (no frozen-weight gradient):
    base 2MNK (Y) + 2MNK (dX); rank side 3 x 2MK(R) (XA, dX term, dA) and
    3 x 2MrN (Y term, G, dB)."""
    R = r * n_seg
    return 4 * M * N * K + 3 * 2 * M * K * R + 3 * 2 * M * r * N
