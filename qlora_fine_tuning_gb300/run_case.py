"""Run one linear of a workload through the C ABI a few times.

A small driver for profilers (ncu) and for quick timing of a single call:

    python -m qlora_fine_tuning_gb300.run_case --workload llama3-8b-mlp-m8192-4096x14336-r64 \
        --linear 0 --rows 4096 --op fwd --iters 3

--rows overrides M (the number of tokens) to keep a capture small.  --op quantize
quantises a seeded fp32 weight of the linear's shape (into the linear's
code and absmax buffers).
Prints the per-iteration CUDA-event time of the requested call.
"""
from __future__ import annotations

import argparse

import numpy as np


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--workload", default="llama3-8b-mlp-m8192-4096x14336-r64")
    p.add_argument("--linear", type=int, default=0)
    p.add_argument("--rows", type=int, default=0)
    p.add_argument("--op", default="fwd", choices=["fwd", "bwd", "both", "dequant", "quantize"])
    p.add_argument("--iters", type=int, default=3)
    a = p.parse_args()

    import torch
    from . import binding, synth

    label, kw = synth.WORKLOADS[a.workload][a.linear]
    kw = dict(kw)
    if a.rows:
        kw["M"] = a.rows
    li = synth.make_linear(seed=0, stream=a.linear, **kw)
    binding.lib()

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)

    idx, absmax, cb = (torch.from_numpy(t).cuda() for t in (li.idx, li.absmax, li.codebook))
    w = binding.make_w4(idx, absmax, cb, li.N, li.K)
    X, A, B, dY = bf(li.X), bf(li.A), bf(li.B), bf(li.dY)
    Y = torch.empty((li.M, li.N), dtype=torch.bfloat16, device="cuda")
    XA = torch.empty((li.M, li.R), dtype=torch.bfloat16, device="cuda")
    dX = torch.empty((li.M, li.K), dtype=torch.bfloat16, device="cuda")
    dA = torch.empty((li.K, li.R), dtype=torch.float32, device="cuda")
    dB = torch.empty((li.r, li.N), dtype=torch.float32, device="cuda")
    Wd = torch.empty((li.N, li.K), dtype=torch.bfloat16, device="cuda")
    ws, ws_bytes = binding.alloc_workspace(li.M, li.N, li.K, li.r, len(li.seg_n))
    seg = None if len(li.seg_n) == 1 else list(li.seg_n)
    if a.op == "quantize":  # a seeded fp32 weight of the linear's shape, quantised on the GPU
        gq = torch.Generator(device="cuda")
        gq.manual_seed(0)
        Wf = torch.randn((li.N, li.K), generator=gq, device="cuda", dtype=torch.float32) * 0.02

    def call():
        if a.op == "quantize":
            binding.quantize_4bit(Wf, False, li.N, li.K, cb, idx, absmax)
            return
        if a.op == "dequant":
            binding.dequant_4bit(w, Wd)
            return
        if a.op in ("fwd", "both") or a.op == "bwd":
            binding.qlora_linear_fwd(X, li.M, w, A, B, li.r, seg, li.s, Y, XA, ws, ws_bytes)
        if a.op in ("bwd", "both"):
            binding.qlora_linear_bwd(dY, X, XA, li.M, w, A, B, li.r, seg, li.s, dX, dA, dB, ws, ws_bytes)

    times = []
    for _ in range(a.iters):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    st = binding.qlora_check_device_error(ws)
    assert st == binding.OK, binding.STATUS[st]
    print(f"{label} M={li.M} K={li.K} N={li.N} r={li.r} op={a.op}: "
          + ", ".join(f"{t:.3f}" for t in times) + " ms")


if __name__ == "__main__":
    main()
