"""Host-side checks of libqlora.so that need no GPU: it loads, exports every
function include/qlora.h declares, and rejects bad arguments with the
documented status before launching anything."""
import ctypes

import pytest

from qlora_fine_tuning_gb300 import binding as b


@pytest.fixture(scope="module")
def L():
    return b.lib()


def test_every_header_function_is_exported(L):
    names = b.header_functions()
    assert {"dequant_4bit", "quantize_4bit", "qlora_linear_fwd", "qlora_linear_bwd", "qlora_workspace_bytes",
            "qlora_check_device_error", "qlora_status_str"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for code in range(7):
        assert isinstance(b.qlora_status_str(code), str) and b.qlora_status_str(code)
    assert b.qlora_status_str(99) == "unknown status"


def test_workspace_bytes_monotone_and_rejects_bad_sizes(L):
    small = b.qlora_workspace_bytes(256, 1024, 1024, 8, 1)
    big = b.qlora_workspace_bytes(8192, 14336, 4096, 64, 1)
    assert 0 < small < big
    assert big >= 2 * 14336 * 4096  # holds the dequantised weight
    assert b.qlora_workspace_bytes(-1, 8, 64, 8, 1) == 0
    assert b.qlora_workspace_bytes(8, 0, 64, 8, 1) == 0


FAKE = 0x10000  # 16-byte-aligned dummy address; never dereferenced on these paths


def _w(N=64, K=64, idx=FAKE, block=64):
    return b.make_w4(idx, FAKE, FAKE, N, K, block)


def _fwd(M=16, w=None, r=8, nseg=1, seg=None, X=FAKE, Y=FAKE, ws=FAKE, ws_bytes=1 << 40):
    w = w or _w()
    arr = None
    if seg is not None:
        arr = (ctypes.c_int64 * len(seg))(*seg)
    return b.lib().qlora_linear_fwd(X, M, ctypes.byref(w), FAKE, FAKE, r, nseg,
                                    ctypes.cast(arr, ctypes.c_void_p) if arr is not None else None, 1.0,
                                    Y, FAKE, ws, ws_bytes, None)


def test_forward_argument_errors(L):
    assert _fwd(X=0) == b.INVALID_ARG
    assert _fwd(M=-1) == b.INVALID_ARG
    assert _fwd(w=_w(K=96)) == b.UNSUPPORTED            # K % 64
    assert _fwd(w=_w(N=68)) == b.UNSUPPORTED            # N % 8
    assert _fwd(w=_w(block=32)) == b.INVALID_ARG
    assert _fwd(r=12) == b.INVALID_ARG
    assert _fwd(r=256) == b.INVALID_ARG
    assert _fwd(X=FAKE + 2) == b.ALIGNMENT
    assert _fwd(w=_w(idx=FAKE + 8)) == b.ALIGNMENT
    assert _fwd(ws=0) == b.WORKSPACE
    assert _fwd(ws_bytes=100) == b.WORKSPACE
    assert _fwd(ws=FAKE + 16) == b.ALIGNMENT
    assert _fwd(nseg=2, seg=None) == b.INVALID_ARG
    assert _fwd(w=_w(N=256), nseg=2, seg=[100, 156]) == b.UNSUPPORTED  # inner boundary not /128
    assert _fwd(w=_w(N=256), nseg=2, seg=[128, 64]) == b.INVALID_ARG   # does not sum to N
    assert _fwd(w=_w(N=2048), r=64, nseg=5, seg=[256] * 4 + [1024]) == b.UNSUPPORTED  # R > 256
    assert _fwd(nseg=9, seg=[8] * 9) == b.INVALID_ARG


def test_empty_batch_forward_is_a_no_op_without_launching(L):
    before = b.qlora_launch_counter()
    assert _fwd(M=0) == b.OK
    assert b.qlora_launch_counter() == before


def test_backward_argument_errors(L):
    w = _w()

    def bwd(dY=FAKE, dA=FAKE, dB=FAKE, dX=FAKE, ws_bytes=1 << 40, r=8):
        return L.qlora_linear_bwd(dY, FAKE, FAKE, 16, ctypes.byref(w), FAKE, FAKE, r, 1, None, 1.0, dX, dA, dB,
                                  FAKE, ws_bytes, None)

    assert bwd(dY=0) == b.INVALID_ARG
    assert bwd(dA=0) == b.INVALID_ARG
    assert bwd(dB=0) == b.INVALID_ARG
    assert bwd(dX=FAKE + 4) == b.ALIGNMENT
    assert bwd(ws_bytes=8) == b.WORKSPACE
    assert bwd(r=4) == b.INVALID_ARG


def test_dequant_argument_errors(L):
    assert L.dequant_4bit(None, FAKE, None, None) == b.INVALID_ARG
    w = _w()
    assert L.dequant_4bit(ctypes.byref(w), None, None, None) == b.INVALID_ARG
    assert L.dequant_4bit(ctypes.byref(w), FAKE + 2, None, None) == b.ALIGNMENT
    w = _w(K=100)
    assert L.dequant_4bit(ctypes.byref(w), FAKE, None, None) == b.UNSUPPORTED
    w = _w(N=0)
    assert L.dequant_4bit(ctypes.byref(w), FAKE, None, None) == b.OK  # nothing to do


def test_quantize_argument_errors(L):
    q = L.quantize_4bit
    assert q(FAKE, 0, -1, 64, FAKE, FAKE, FAKE, None) == b.INVALID_ARG
    assert q(FAKE, 0, 4, 0, FAKE, FAKE, FAKE, None) == b.INVALID_ARG
    assert q(FAKE, 0, 4, 96, FAKE, FAKE, FAKE, None) == b.UNSUPPORTED
    assert q(None, 0, 4, 64, FAKE, FAKE, FAKE, None) == b.INVALID_ARG
    assert q(FAKE, 0, 4, 64, None, FAKE, FAKE, None) == b.INVALID_ARG
    assert q(FAKE + 4, 0, 4, 64, FAKE, FAKE, FAKE, None) == b.ALIGNMENT
    assert q(FAKE, 1, 4, 64, FAKE, FAKE + 8, FAKE, None) == b.ALIGNMENT
    assert q(FAKE, 0, 0, 64, None, None, None, None) == b.OK  # nothing to do, nothing launched


def test_profiler_collect_empty(L):
    b.qlora_profiler_enable(True)
    assert b.qlora_profiler_collect() == []
    b.qlora_profiler_enable(False)
