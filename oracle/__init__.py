"""CPU fp64 oracle for the QLoRA-adapted linear layer -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and
this package imports nothing from the product package.

The arithmetic lives in ``qlora_oracle.c`` (plain loops, double precision,
ascending summation order, no contraction into FMA).  This wrapper only
compiles it, converts bf16 bit patterns to doubles exactly and marshals numpy
arrays.  Definitions followed, by page:

* "Introducing Unsloth: LLM 训练提速 30 倍", section 手动 Autograd -- the
  adapted projection X(W + AB) with W frozen, the derivatives w.r.t. A, B and
  the input, and the rank-r bracketing of the chain product.
* "利用 Unsloth 和 NVIDIA 硬件加速 LLM 训练", section 1 -- the 4-bit weight
  is dequantised to a 16-bit format before the tensor-core product.
* "UnSloth极速微调" -- bf16 is the 16-bit format.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qlora_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, -O2, IEEE semantics kept)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", "-std=c11", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int64
            D = ctypes.c_double
            lib.oracle_bf16_rne.restype = ctypes.c_uint16
            lib.oracle_bf16_rne.argtypes = [ctypes.c_float]
            lib.oracle_dequant.restype = None
            lib.oracle_dequant.argtypes = [P, P, P, I, I, I, P, P]
            lib.oracle_quantize.restype = None
            lib.oracle_quantize.argtypes = [P, I, I, I, P, P, P]
            lib.oracle_forward_rows.restype = None
            lib.oracle_forward_rows.argtypes = [P, P, P, P, I, I, I, I, I, P, D, P, I, P, P]
            lib.oracle_backward_dx_rows.restype = None
            lib.oracle_backward_dx_rows.argtypes = [P, P, P, P, I, I, I, I, I, P, D, P, I, P, P]
            lib.oracle_backward_da.restype = None
            lib.oracle_backward_da.argtypes = [P, P, P, I, I, I, I, I, P, D, P, I, P, I, P]
            lib.oracle_backward_db.restype = None
            lib.oracle_backward_db.argtypes = [P, P, P, I, I, I, I, I, P, D, P, I, P, I, P]
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_num_threads.argtypes = []
            lib.oracle_set_num_threads.restype = None
            lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Worker threads of the following calls (timing only; results do not
    depend on it: every output is one thread's ascending-order sum)."""
    _load().oracle_set_num_threads(int(n))


# --------------------------------------------------------------------------
# bf16 helpers
# --------------------------------------------------------------------------

def bf16_rne(x) -> np.ndarray:
    """fp32 -> bf16 bit patterns (round to nearest, ties to even), elementwise."""
    lib = _load()
    x = np.asarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    flat_in, flat_out = x.reshape(-1), out.reshape(-1)
    for i in range(flat_in.size):
        flat_out[i] = lib.oracle_bf16_rne(float(flat_in[i]))
    return out


def bf16_to_f64(h) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    h = np.asarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# Dequantisation
# --------------------------------------------------------------------------

def dequant(idx, absmax, codebook, N: int, K: int, block: int = 64):
    """Return (W32 float32 [N,K], W16 uint16 bf16 bits [N,K])."""
    lib = _load()
    idx = _c(idx, np.uint8)
    absmax = _c(absmax, np.float32)
    codebook = _c(codebook, np.float32)
    assert idx.size == N * K // 2 and absmax.size == N * K // block and codebook.size == 16
    w32 = np.empty((N, K), dtype=np.float32)
    w16 = np.empty((N, K), dtype=np.uint16)
    lib.oracle_dequant(_p(idx), _p(absmax), _p(codebook), N, K, block, _p(w32), _p(w16))
    return w32, w16


def quantize(w, codebook, block: int = 64):
    """fp32 W [N,K] -> (idx uint8 [N,K/2], absmax float32 [N*K/block]).

    Per block of the row-major flattening: absmax = max |w|; the code of each
    element is the first i minimising |w/absmax - codebook[i]| in double
    precision (t = 0 for a zero block).  Pass bf16 weights widened to fp32.
    """
    lib = _load()
    w = _c(w, np.float32)
    codebook = _c(codebook, np.float32)
    N, K = w.shape
    assert K % block == 0 and codebook.size == 16
    idx = np.empty((N, K // 2), dtype=np.uint8)
    absmax = np.empty((N * K // block,), dtype=np.float32)
    lib.oracle_quantize(_p(w), N, K, block, _p(codebook), _p(idx), _p(absmax))
    return idx, absmax


# --------------------------------------------------------------------------
# Linear layer (operands given as float64 arrays; bf16 inputs widened exactly)
# --------------------------------------------------------------------------

def _segs(N: int, seg_n):
    if seg_n is None:
        seg_n = [N]
    seg = _c(list(seg_n), np.int64)
    assert int(seg.sum()) == N
    return seg


def forward_rows(X, Wd, A, B, r: int, s: float, rows=None, seg_n=None):
    """XA and Y rows; X [M,K], Wd [N,K], A [K,R], B [r,N] as float64."""
    lib = _load()
    X, Wd, A, B = (_c(t, np.float64) for t in (X, Wd, A, B))
    M, K = X.shape
    N = Wd.shape[0]
    seg = _segs(N, seg_n)
    R = r * seg.size
    assert A.shape == (K, R) and B.shape == (r, N) and Wd.shape == (N, K)
    rows = _c(np.arange(M) if rows is None else rows, np.int64)
    xa = np.empty((rows.size, R), dtype=np.float64)
    y = np.empty((rows.size, N), dtype=np.float64)
    lib.oracle_forward_rows(_p(X), _p(Wd), _p(A), _p(B), M, N, K, r, seg.size, _p(seg),
                            float(s), _p(rows), rows.size, _p(xa), _p(y))
    return xa, y


def backward_dx_rows(dY, Wd, A, B, r: int, s: float, rows=None, seg_n=None):
    """G and dX rows; dY [M,N] float64."""
    lib = _load()
    dY, Wd, A, B = (_c(t, np.float64) for t in (dY, Wd, A, B))
    M, N = dY.shape
    K = Wd.shape[1]
    seg = _segs(N, seg_n)
    R = r * seg.size
    assert A.shape == (K, R) and B.shape == (r, N) and Wd.shape == (N, K)
    rows = _c(np.arange(M) if rows is None else rows, np.int64)
    g = np.empty((rows.size, R), dtype=np.float64)
    dx = np.empty((rows.size, K), dtype=np.float64)
    lib.oracle_backward_dx_rows(_p(dY), _p(Wd), _p(A), _p(B), M, N, K, r, seg.size, _p(seg),
                                float(s), _p(rows), rows.size, _p(g), _p(dx))
    return g, dx


def backward_da(X, dY, B, r: int, s: float, kidx=None, Jidx=None, seg_n=None):
    """dA[kidx][:, Jidx] as float64 [len(kidx), len(Jidx)], summed over all rows."""
    lib = _load()
    X, dY, B = (_c(t, np.float64) for t in (X, dY, B))
    M, K = X.shape
    N = dY.shape[1]
    seg = _segs(N, seg_n)
    R = r * seg.size
    kidx = _c(np.arange(K) if kidx is None else kidx, np.int64)
    Jidx = _c(np.arange(R) if Jidx is None else Jidx, np.int64)
    out = np.empty((kidx.size, Jidx.size), dtype=np.float64)
    lib.oracle_backward_da(_p(X), _p(dY), _p(B), M, N, K, r, seg.size, _p(seg), float(s),
                           _p(kidx), kidx.size, _p(Jidx), Jidx.size, _p(out))
    return out


def backward_db(X, dY, A, r: int, s: float, cidx=None, nidx=None, seg_n=None):
    """dB[cidx][:, nidx] as float64 [len(cidx), len(nidx)], summed over all rows."""
    lib = _load()
    X, dY, A = (_c(t, np.float64) for t in (X, dY, A))
    M, K = X.shape
    N = dY.shape[1]
    seg = _segs(N, seg_n)
    cidx = _c(np.arange(r) if cidx is None else cidx, np.int64)
    nidx = _c(np.arange(N) if nidx is None else nidx, np.int64)
    out = np.empty((cidx.size, nidx.size), dtype=np.float64)
    lib.oracle_backward_db(_p(X), _p(dY), _p(A), M, N, K, r, seg.size, _p(seg), float(s),
                           _p(cidx), cidx.size, _p(nidx), nidx.size, _p(out))
    return out


def linear_full(X, Wd, A, B, dY, r: int, s: float, seg_n=None):
    """Every output of one forward + backward: dict of float64 arrays."""
    xa, y = forward_rows(X, Wd, A, B, r, s, seg_n=seg_n)
    g, dx = backward_dx_rows(dY, Wd, A, B, r, s, seg_n=seg_n)
    da = backward_da(X, dY, B, r, s, seg_n=seg_n)
    db = backward_db(X, dY, A, r, s, seg_n=seg_n)
    return {"XA": xa, "Y": y, "G": g, "dX": dx, "dA": da, "dB": db}


def rel_fro(got, ref) -> float:
    """||got - ref||_F / ||ref||_F (0 when both are exactly zero)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.linalg.norm(ref))
    num = float(np.linalg.norm(got - ref))
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return num / den
