"""Reader for tests/golden/closed_form_tiny.txt (a hand-worked example)."""
import os

import numpy as np

PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "closed_form_tiny.txt")


def load():
    rows = {}
    with open(PATH) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rows.setdefault(key, []).append(vals)
    one = lambda k: rows[k][0]
    M, K, N, r = (int(one(k)[0]) for k in ("M", "K", "N", "r"))
    s = float(one("s")[0])
    cb = np.array([float(v) for v in one("codebook")], dtype=np.float32)
    absmax = np.array([float(v) for v in one("absmax")], dtype=np.float32)
    assert absmax.size == N * K // 64
    bytes_ = [int(v, 16) for v in one("rowbyte")]
    idx = np.array([[b] * (K // 2) for b in bytes_], dtype=np.uint8)
    xrow = [float(v) for v in one("X_row")]
    X = np.array([[xv] * K for xv in xrow], dtype=np.float32)
    A = np.full((K, r), float(one("A_all")[0]), dtype=np.float32)
    B = np.array([[float(v) for v in one("B")]], dtype=np.float32)
    dY = np.array([[float(v) for v in row] for row in rows["dY"]], dtype=np.float32)
    exp = {
        "Wd_row0": [float(v) for v in one("expect_Wd_row0")],
        "Wd_row1": [float(v) for v in one("expect_Wd_row1")],
        "XA": np.array([float(v) for v in one("expect_XA")]).reshape(M, r),
        "Y": np.array([[float(v) for v in row] for row in rows["expect_Y"]]),
        "G": np.array([float(v) for v in one("expect_G")]).reshape(M, r),
        "dX_row0": [float(v) for v in one("expect_dX_row0")],
        "dX_row1": [float(v) for v in one("expect_dX_row1")],
        "dA_all": float(one("expect_dA_all")[0]),
        "dB": np.array([[float(v) for v in one("expect_dB")]]),
    }
    return dict(M=M, K=K, N=N, r=r, s=s, codebook=cb, absmax=absmax, idx=idx, X=X, A=A, B=B,
                dY=dY, expect=exp)


def expected_dense(case):
    """Expand the per-row patterns of the expected Wd and dX to full arrays."""
    K, N, M = case["K"], case["N"], case["M"]
    e = case["expect"]
    wd = np.zeros((N, K))
    wd[0, :] = e["Wd_row0"][0]
    wd[1, 0::2] = e["Wd_row1"][0]
    wd[1, 1::2] = e["Wd_row1"][1]
    dx = np.zeros((M, K))
    dx[0, :] = e["dX_row0"][0]
    dx[1, 0::2] = e["dX_row1"][0]
    dx[1, 1::2] = e["dX_row1"][1]
    da = np.full((K, case["r"]), e["dA_all"])
    return wd, dx, da
