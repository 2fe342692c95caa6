"""ctypes binding of libqlora.so -- argument marshalling only.

The functions here carry the C ABI's names and call straight into it: they
turn torch tensors into device pointers, pass torch's current CUDA stream, and
raise ``QloraError`` on a non-OK status.  Every step of the layer runs inside
the library's CUDA kernels; nothing here computes.  If the library is missing
or cannot be loaded the import-time call ``lib()`` raises -- there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from typing import Optional, Sequence

from . import build as _build

_lock = threading.Lock()
_lib = None

STATUS = {
    0: "QLORA_OK",
    1: "QLORA_ERR_INVALID_ARG",
    2: "QLORA_ERR_UNSUPPORTED",
    3: "QLORA_ERR_ALIGNMENT",
    4: "QLORA_ERR_WORKSPACE",
    5: "QLORA_ERR_CUDA",
    6: "QLORA_ERR_TIMEOUT",
}
OK, INVALID_ARG, UNSUPPORTED, ALIGNMENT, WORKSPACE, CUDA, TIMEOUT = range(7)


class QloraError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS.get(self.status, self.status)} "
                         f"({lib().qlora_status_str(self.status).decode()})")


class W4(ctypes.Structure):
    """qlora_w4: the frozen 4-bit weight descriptor."""
    _fields_ = [("idx", ctypes.c_void_p), ("absmax", ctypes.c_void_p), ("codebook", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("block", ctypes.c_int32)]


class KernelStat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_int64), ("total_ms", ctypes.c_double)]


def header_functions() -> list:
    """Names of the functions declared in include/qlora.h."""
    path = os.path.join(_build.ROOT, "include", "qlora.h")
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "for", "sizeof")))


def lib(path: Optional[str] = None):
    """Load (building first if stale) libqlora.so.  Raises if unavailable."""
    global _lib
    with _lock:
        if _lib is None:
            so = path or _build.build()
            L = ctypes.CDLL(so)
            P, I64, I32, F, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
            WP = ctypes.POINTER(W4)
            L.dequant_4bit.restype = ctypes.c_int
            L.dequant_4bit.argtypes = [WP, P, P, P]
            L.qlora_linear_fwd.restype = ctypes.c_int
            L.qlora_linear_fwd.argtypes = [P, I64, WP, P, P, I32, I32, P, F, P, P, P, SZ, P]
            L.qlora_linear_bwd.restype = ctypes.c_int
            L.qlora_linear_bwd.argtypes = [P, P, P, I64, WP, P, P, I32, I32, P, F, P, P, P, P, SZ, P]
            L.qlora_linear_bwd_accumulate.restype = ctypes.c_int
            L.qlora_linear_bwd_accumulate.argtypes = [P, P, P, I64, WP, P, P, I32, I32, P, F, P, P, P, P, SZ, P]
            L.qlora_workspace_bytes.restype = SZ
            L.qlora_workspace_bytes.argtypes = [I64, I64, I64, I32, I32]
            L.qlora_check_device_error.restype = ctypes.c_int
            L.qlora_check_device_error.argtypes = [P, P]
            L.qlora_set_wait_limit_ns.restype = None
            L.qlora_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            L.qlora_status_str.restype = ctypes.c_char_p
            L.qlora_status_str.argtypes = [ctypes.c_int]
            L.qlora_profiler_enable.restype = None
            L.qlora_profiler_enable.argtypes = [ctypes.c_int]
            L.qlora_profiler_collect.restype = ctypes.c_int
            L.qlora_profiler_collect.argtypes = [ctypes.POINTER(KernelStat), ctypes.c_int]
            L.qlora_launch_counter.restype = ctypes.c_uint64
            L.qlora_launch_counter.argtypes = []
            L.qlora_debug_stall_next_launch.restype = None
            L.qlora_debug_stall_next_launch.argtypes = [ctypes.c_char_p]
            L.quantize_4bit.restype = ctypes.c_int
            L.quantize_4bit.argtypes = [P, I32, I64, I64, P, P, P, P]
            L.qlora_linear_xa_static.restype = ctypes.c_int
            L.qlora_linear_xa_static.argtypes = [P, I64, I64, P, I32, P, P]
            L.qlora_linear_xa_static_status.restype = ctypes.c_int
            L.qlora_linear_xa_static_status.argtypes = [P]
            _lib = L
    return _lib


def library_path() -> str:
    return _build.LIB


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------

def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return int(t.data_ptr())


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _check(st: int, where: str):
    if st != OK:
        raise QloraError(st, where)


def make_w4(idx, absmax, codebook, N: int, K: int, block: int = 64) -> W4:
    """Descriptor of a 4-bit weight.  It keeps references to the tensors it
    points at, so their device memory outlives the descriptor."""
    w = W4(_ptr(idx), _ptr(absmax), _ptr(codebook), int(N), int(K), int(block))
    w._keep = (idx, absmax, codebook)
    return w


def _seg_array(seg_n: Optional[Sequence[int]]):
    if seg_n is None:
        return None, 1
    arr = (ctypes.c_int64 * len(seg_n))(*[int(v) for v in seg_n])
    return arr, len(seg_n)


# --------------------------------------------------------------------------
# C ABI, same names
# --------------------------------------------------------------------------

def dequant_4bit(w: W4, out_bf16=None, out_f32=None, stream=None) -> None:
    _check(lib().dequant_4bit(ctypes.byref(w), _ptr(out_bf16), _ptr(out_f32), _stream(stream)), "dequant_4bit")


def quantize_4bit(W, w_is_bf16: bool, N: int, K: int, codebook, idx, absmax, stream=None) -> None:
    _check(lib().quantize_4bit(_ptr(W), 1 if w_is_bf16 else 0, int(N), int(K), _ptr(codebook), _ptr(idx),
                               _ptr(absmax), _stream(stream)), "quantize_4bit")


def qlora_linear_fwd(X, M: int, w: W4, A, B, r: int, seg_n, s: float, Y, XA_save, ws, ws_bytes: int,
                     stream=None) -> None:
    seg, nseg = _seg_array(seg_n)
    st = lib().qlora_linear_fwd(_ptr(X), int(M), ctypes.byref(w), _ptr(A), _ptr(B), int(r), nseg,
                                ctypes.cast(seg, ctypes.c_void_p) if seg is not None else None, float(s),
                                _ptr(Y), _ptr(XA_save), _ptr(ws), int(ws_bytes), _stream(stream))
    _check(st, "qlora_linear_fwd")


def qlora_linear_bwd(dY, X, XA_saved, M: int, w: W4, A, B, r: int, seg_n, s: float, dX, dA, dB, ws,
                     ws_bytes: int, stream=None) -> None:
    seg, nseg = _seg_array(seg_n)
    st = lib().qlora_linear_bwd(_ptr(dY), _ptr(X), _ptr(XA_saved), int(M), ctypes.byref(w), _ptr(A), _ptr(B),
                                int(r), nseg, ctypes.cast(seg, ctypes.c_void_p) if seg is not None else None,
                                float(s), _ptr(dX), _ptr(dA), _ptr(dB), _ptr(ws), int(ws_bytes), _stream(stream))
    _check(st, "qlora_linear_bwd")


def qlora_linear_bwd_accumulate(dY, X, XA_saved, M: int, w: W4, A, B, r: int, seg_n, s: float, dX, dA, dB, ws,
                                ws_bytes: int, stream=None) -> None:
    seg, nseg = _seg_array(seg_n)
    st = lib().qlora_linear_bwd_accumulate(_ptr(dY), _ptr(X), _ptr(XA_saved), int(M), ctypes.byref(w), _ptr(A),
                                           _ptr(B), int(r), nseg,
                                           ctypes.cast(seg, ctypes.c_void_p) if seg is not None else None,
                                           float(s), _ptr(dX), _ptr(dA), _ptr(dB), _ptr(ws), int(ws_bytes),
                                           _stream(stream))
    _check(st, "qlora_linear_bwd_accumulate")


def qlora_workspace_bytes(M: int, N: int, K: int, r: int, n_seg: int = 1) -> int:
    return int(lib().qlora_workspace_bytes(int(M), int(N), int(K), int(r), int(n_seg)))


def qlora_check_device_error(ws, stream=None) -> int:
    return int(lib().qlora_check_device_error(_ptr(ws), _stream(stream)))


def qlora_set_wait_limit_ns(ns: int) -> None:
    lib().qlora_set_wait_limit_ns(int(ns))


def qlora_debug_stall_next_launch(label) -> None:
    lib().qlora_debug_stall_next_launch(None if label is None else label.encode())


def qlora_status_str(status: int) -> str:
    return lib().qlora_status_str(int(status)).decode()


def qlora_profiler_enable(on: bool = True) -> None:
    lib().qlora_profiler_enable(1 if on else 0)


def qlora_profiler_collect() -> list:
    L = lib()
    # collect() resets the records, so ask once with enough room
    buf = (KernelStat * 64)()
    n = L.qlora_profiler_collect(buf, 64)
    return [(buf[i].name.decode(), int(buf[i].launches), float(buf[i].total_ms)) for i in range(min(n, 64))]


def qlora_launch_counter() -> int:
    return int(lib().qlora_launch_counter())


def qlora_linear_xa_static(X, M: int, K: int, A, R: int, XA, stream=None) -> None:
    """XA = X A with the library's static device scratch: for callers that
    cannot allocate device memory, so cannot provide a workspace."""
    st = lib().qlora_linear_xa_static(_ptr(X), int(M), int(K), _ptr(A), int(R), _ptr(XA), _stream(stream))
    _check(st, "qlora_linear_xa_static")


def qlora_linear_xa_static_status(stream=None) -> int:
    """Status of the static-scratch XA calls since the last query (OK or
    TIMEOUT); clears it."""
    return int(lib().qlora_linear_xa_static_status(_stream(stream)))


# --------------------------------------------------------------------------
# torch allocation helpers (device memory only; no arithmetic)
# --------------------------------------------------------------------------

def alloc_workspace(M: int, N: int, K: int, r: int, n_seg: int = 1, device="cuda"):
    """A zeroed workspace of the required size (256-byte aligned by torch)."""
    import torch
    nbytes = qlora_workspace_bytes(M, N, K, r, n_seg)
    if nbytes == 0:
        raise QloraError(INVALID_ARG, "qlora_workspace_bytes")
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=device)
    return ws, nbytes
