"""Test helpers: run the CUDA path through the C ABI and the oracle on the same
seeded inputs, and compare."""
from __future__ import annotations

import numpy as np

import oracle
from qlora_fine_tuning_gb300 import binding, synth

TOL = 1e-2  # relative Frobenius error bound on Y, dX, dA, dB (bf16 in, fp32 accumulate)


def dev_bf16(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def dev(arr: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(arr)).cuda()


def host_bits(t) -> np.ndarray:
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


class GpuLayer:
    """Device copies of one linear layer's inputs plus its outputs/workspace."""

    def __init__(self, li: synth.LinearInputs):
        import torch
        self.li = li
        self.idx = dev(li.idx)
        self.absmax = dev(li.absmax)
        self.codebook = dev(li.codebook)
        self.X = dev_bf16(li.X)
        self.A = dev_bf16(li.A)
        self.B = dev_bf16(li.B)
        self.dY = dev_bf16(li.dY)
        M, N, K, R = li.M, li.N, li.K, li.R
        self.w = binding.make_w4(self.idx, self.absmax, self.codebook, N, K)
        self.Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        self.XA = torch.empty((max(M, 1), R), dtype=torch.bfloat16, device="cuda")
        self.dX = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
        self.dA = torch.empty((K, R), dtype=torch.float32, device="cuda")
        self.dB = torch.empty((li.r, N), dtype=torch.float32, device="cuda")
        self.ws, self.ws_bytes = binding.alloc_workspace(M, N, K, li.r, len(li.seg_n))
        self.seg = None if len(li.seg_n) == 1 else list(li.seg_n)

    def forward(self):
        li = self.li
        binding.qlora_linear_fwd(self.X, li.M, self.w, self.A, self.B, li.r, self.seg, li.s, self.Y, self.XA,
                                 self.ws, self.ws_bytes)

    def backward(self, with_dx=True):
        li = self.li
        binding.qlora_linear_bwd(self.dY, self.X, self.XA, li.M, self.w, self.A, self.B, li.r, self.seg, li.s,
                                 self.dX if with_dx else None, self.dA, self.dB, self.ws, self.ws_bytes)

    def check(self):
        st = binding.qlora_check_device_error(self.ws)
        assert st == binding.OK, binding.STATUS.get(st)

    def results(self) -> dict:
        import torch
        torch.cuda.synchronize()
        return {
            "Y": oracle.bf16_to_f64(host_bits(self.Y)),
            "XA": oracle.bf16_to_f64(host_bits(self.XA))[: self.li.M],
            "dX": oracle.bf16_to_f64(host_bits(self.dX)),
            "dA": self.dA.cpu().numpy().astype(np.float64),
            "dB": self.dB.cpu().numpy().astype(np.float64),
        }


def oracle_operands(li: synth.LinearInputs):
    _, w16 = oracle.dequant(li.idx, li.absmax, li.codebook, li.N, li.K)
    return (oracle.bf16_to_f64(li.X), oracle.bf16_to_f64(w16), oracle.bf16_to_f64(li.A),
            oracle.bf16_to_f64(li.B), oracle.bf16_to_f64(li.dY))


def oracle_full(li: synth.LinearInputs) -> dict:
    X, Wd, A, B, dY = oracle_operands(li)
    seg = None if len(li.seg_n) == 1 else li.seg_n
    return oracle.linear_full(X, Wd, A, B, dY, li.r, li.s, seg_n=seg)


def sample_indices(li: synth.LinearInputs, seed: int = 0, row_tile: int = 256, col_block: int = 128):
    """Output indices the oracle evaluates at full size, chosen so that every
    tile the kernels produce is looked at:

    * rows of Y, dX and XA: one random row inside every 256-row tile (the pair
      GEMM's row tile, so every tile row of the persistent walk, including the
      partial last one), plus rows 0, M/2 and M-1; each sampled row is compared
      over all its columns, which covers every column tile;
    * dA: one random row k inside every 128-row block of dA, plus 0 and K-1,
      every column J;
    * dB: one random column n inside every 128-column block of dB, plus 0 and
      N-1, every row c.
    """
    rng = np.random.default_rng(seed)
    M, N, K, R, r = li.M, li.N, li.K, li.R, li.r

    def one_per(n, t):
        return [int(rng.integers(a, min(a + t, n))) for a in range(0, n, t)]

    rows = sorted(set([0, M - 1, M // 2] + one_per(M, row_tile)))
    kidx = sorted(set([0, K - 1] + one_per(K, col_block)))
    nidx = sorted(set([0, N - 1] + one_per(N, col_block)))
    Jidx = list(range(R))
    cidx = list(range(r))
    return rows, kidx, Jidx, cidx, nidx


def oracle_sampled(li: synth.LinearInputs, idx) -> dict:
    rows, kidx, Jidx, cidx, nidx = idx
    X, Wd, A, B, dY = oracle_operands(li)
    seg = None if len(li.seg_n) == 1 else li.seg_n
    xa, y = oracle.forward_rows(X, Wd, A, B, li.r, li.s, rows=rows, seg_n=seg)
    g, dx = oracle.backward_dx_rows(dY, Wd, A, B, li.r, li.s, rows=rows, seg_n=seg)
    da = oracle.backward_da(X, dY, B, li.r, li.s, kidx=kidx, Jidx=Jidx, seg_n=seg)
    db = oracle.backward_db(X, dY, A, li.r, li.s, cidx=cidx, nidx=nidx, seg_n=seg)
    return {"XA": xa, "Y": y, "dX": dx, "dA": da, "dB": db}


# Tile shapes of the per-tile checks on full outputs: the GEMMs' output tiles
# (128-row TMEM lanes x 128 columns) for Y and dX, 128-row blocks of XA and dA,
# 128-column blocks of dB.
TILES_FULL = {"Y": (128, 128), "dX": (128, 128), "XA": (128, 256), "G": (128, 256), "dA": (128, 256),
              "dB": (128, 128)}
# On sampled outputs each sampled row (column for dB) comes from a different
# tile: check it in 128-column (row) pieces.
TILES_SAMPLED = {"Y": (1, 128), "dX": (1, 128), "XA": (1, 256), "G": (1, 256), "dA": (1, 256), "dB": (128, 1)}
TILE_TOL = 2e-2   # relative Frobenius error bound of every tile
ELEM_REL = 2e-2   # per element: |got - ref| <= ELEM_REL |ref| + ELEM_RMS rms(ref tile)
ELEM_RMS = 5e-2


def tile_errors(got, ref, tile) -> list:
    """[(row0, col0, tile rel. Frobenius error, worst element excess)] for
    every tile of a 2-D comparison.  The element excess is the largest
    |got - ref| / (ELEM_REL |ref| + ELEM_RMS rms(ref tile)); above 1 means an
    element is out of bounds (for an all-zero reference tile any nonzero
    element gives inf)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if got.ndim == 1:
        got, ref = got[None, :], ref[None, :]
    th, tw = tile
    out = []
    for i in range(0, ref.shape[0], th):
        for j in range(0, ref.shape[1], tw):
            g = got[i:i + th, j:j + tw]
            f = ref[i:i + th, j:j + tw]
            rel = oracle.rel_fro(g, f)
            bound = ELEM_REL * np.abs(f) + ELEM_RMS * float(np.sqrt(np.mean(f * f)))
            diff = np.abs(g - f)
            with np.errstate(divide="ignore", invalid="ignore"):
                ex = np.where(diff == 0.0, 0.0, diff / bound)
            out.append((i, j, rel, float(np.max(ex)) if ex.size else 0.0))
    return out


def compare(got: dict, ref: dict, keys=("Y", "dX", "dA", "dB"), tol=TOL, tiles=None) -> dict:
    """Relative Frobenius error of every tensor (<= tol), of every tile of it
    (<= TILE_TOL) and a bound on every element; returns the tensor errors.

    `tiles` maps a key to its tile shape (default TILES_FULL; pass
    TILES_SAMPLED for outputs gathered by sample_indices)."""
    tiles = TILES_FULL if tiles is None else tiles
    errs = {k: oracle.rel_fro(got[k], ref[k]) for k in keys}
    bad = {k: v for k, v in errs.items() if not (v <= tol)}
    assert not bad, f"relative Frobenius error above {tol}: {errs}"
    for k in keys:
        te = tile_errors(got[k], ref[k], tiles[k])
        worst_rel = max(te, key=lambda e: e[2])
        worst_el = max(te, key=lambda e: e[3])
        assert worst_rel[2] <= TILE_TOL, f"{k}: tile at {worst_rel[:2]} has relative error {worst_rel[2]:.3g}"
        assert worst_el[3] <= 1.0, f"{k}: an element of tile {worst_el[:2]} is out of bounds ({worst_el[3]:.3g}x)"
    return errs


def check_sampled(li: synth.LinearInputs, got: dict, seed: int = 0) -> dict:
    """Compare a full-size run with the oracle on the outputs sample_indices
    picks (every row tile, every 128-row block of dA, every 128-column block
    of dB), with the tensor, tile and element bounds of compare()."""
    idx = sample_indices(li, seed)
    rows, kidx, Jidx, cidx, nidx = idx
    ref = oracle_sampled(li, idx)
    sub = {"Y": got["Y"][rows], "dX": got["dX"][rows], "XA": got["XA"][rows],
           "dA": got["dA"][np.ix_(kidx, Jidx)], "dB": got["dB"][np.ix_(cidx, nidx)]}
    return compare(sub, ref, keys=("Y", "dX", "dA", "dB", "XA"), tiles=TILES_SAMPLED)
