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


def sample_indices(li: synth.LinearInputs, seed: int = 0, nrows: int = 12, ncols: int = 16, nj: int = 4):
    rng = np.random.default_rng(seed)
    M, N, K, R, r = li.M, li.N, li.K, li.R, li.r
    rows = sorted(set([0, M - 1, M // 2] + list(rng.integers(0, M, nrows))))
    kidx = sorted(set([0, K - 1] + list(rng.integers(0, K, ncols))))
    Jidx = sorted(set([0, R - 1] + list(rng.integers(0, R, nj))))
    cidx = sorted(set([0, r - 1] + list(rng.integers(0, r, nj))))
    nidx = sorted(set([0, N - 1] + list(rng.integers(0, N, ncols))))
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


def compare(got: dict, ref: dict, keys=("Y", "dX", "dA", "dB"), tol=TOL) -> dict:
    errs = {k: oracle.rel_fro(got[k], ref[k]) for k in keys}
    bad = {k: v for k, v in errs.items() if not (v <= tol)}
    assert not bad, f"relative Frobenius error above {tol}: {errs}"
    return errs
