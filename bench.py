#!/usr/bin/env python3
"""Benchmark: QLoRA linear forward + backward TFLOP/s on one GB300.

One step = the forward of every linear of the workload, then the backward of
each in reverse order (a training step's pass over these layers), on seeded
synthetic inputs already resident in HBM.  Default workload: the Llama-3-8B
MLP projections (gate and up 4096->14336, down 14336->4096) at 8192 packed
tokens, rank 64, s = 0.25.  FLOPs counted per linear: 4MNK + 6Mr(K+N)
(no frozen-weight gradient; dequantisation not counted).

Prints one JSON line.  `--impl reference` times the CPU fp64 oracle instead,
on a bounded sample of the same workload (that arm is a deliberately slow
baseline, not a target).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from qlora_fine_tuning_gb300 import synth  # noqa: E402

DEFAULT_WORKLOAD = "llama3-8b-mlp-m8192-4096x14336-r64"
METRIC = "QLoRA linear fwd+bwd TFLOP/s on 1 GB300; % of BF16 dense tensor peak"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-graph", action="store_true", help="launch every step instead of replaying a CUDA graph")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU time of the oracle sample")
    return p.parse_args()


def workload_flops(lins) -> int:
    return sum(synth.flops_fwd_bwd(li.M, li.N, li.K, li.r, len(li.seg_n)) for li in lins)


def config_of(name, lins, n_gpus):
    return {
        "workload": name,
        "linears": [{"label": li.meta.get("label"), "M": li.M, "K": li.K, "N": li.N, "r": li.r, "s": li.s,
                     "n_seg": len(li.seg_n)} for li in lins],
        "weights": "4-bit codebook indices + fp32 absmax per 64 (quantile codebook)",
        "parallelism": (f"data parallel x{n_gpus}: each rank its own {lins[0].M}-token shard per linear, "
                        "W/A/B replicated, one sum all-reduce of dA and dB per linear on a reduce stream")
                       if n_gpus > 1 else "single GPU",
        "l2": "inputs larger than L2 (per-step working set >> 129 MB), no flush",
    }


# --------------------------------------------------------------------------
# distributed plumbing (barrier + max over ranks only)
# --------------------------------------------------------------------------

def relaunch(n_gpus: int) -> int:
    """--gpus N > 1 without a launcher: start N ranks of this script under
    torch.distributed.run on this node (one per GPU) and return its exit code."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    env = dict(os.environ)
    env.setdefault("NCCL_DEBUG", "INFO")          # communicator set-up lines (ranks, nranks) on stderr
    env.setdefault("NCCL_DEBUG_SUBSYS", "INIT")
    env.setdefault("NCCL_DEBUG_FILE", "/dev/stderr")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n_gpus}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd, env=env)


def dist_init(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl"
        import torch
        if not torch.cuda.is_available():
            backend = "gloo"
        os.environ.setdefault("NCCL_DEBUG", "INFO")
        os.environ.setdefault("NCCL_DEBUG_SUBSYS", "INIT")
        os.environ.setdefault("NCCL_DEBUG_FILE", "/dev/stderr")
        dist.init_process_group(backend=backend)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------
# clocks
# --------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=0):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# --------------------------------------------------------------------------
# our CUDA path
# --------------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


PAIR_TRAFFIC = os.path.join(ROOT, "profiles", "gemm_pair_traffic.json")


def strip_comments(src: str) -> str:
    """C/C++ source without its comments and trailing blanks (string literals
    in these files hold PTX, which has no comment markers)."""
    import re
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def pair_sources_sha256(csrc: str = None) -> str:
    """sha256 of what decides the pair GEMM's DRAM traffic: its kernel source,
    the PTX wrappers and the host's tile-order choice (pair_group()), with
    comments removed (a comment edit does not change the traffic)."""
    import hashlib
    import re
    csrc = csrc or os.path.join(ROOT, "qlora_fine_tuning_gb300", "csrc")
    h = hashlib.sha256()
    for f in ("gemm_pair.cuh", "ptx.cuh"):
        with open(os.path.join(csrc, f)) as fh:
            h.update(strip_comments(fh.read()).encode())
    with open(os.path.join(csrc, "qlora_api.cu")) as fh:
        m = re.search(r"int pair_group\(.*?\n}\n", fh.read(), re.S)
    h.update(strip_comments(m.group(0)).encode() if m else b"")
    return h.hexdigest()


def pair_traffic(workload: str):
    """(bytes per launch, note): the stored ncu capture of the pair GEMM's DRAM
    bytes (a figure taken by an earlier ncu run, not by this run), reported
    only for the workload it was taken on and while the sources still hash to
    the captured state; else (None, why)."""
    try:
        with open(PAIR_TRAFFIC) as fh:
            d = json.load(fh)
        val = int(d["traffic_bytes_per_launch"])
        sha = str(d["sources_sha256"])
        wl = str(d["workload"])
    except (OSError, KeyError, ValueError, TypeError):
        return None, "no stored capture"
    if workload != wl:
        return None, f"stored capture is for the {wl} workload only"
    if sha != pair_sources_sha256():
        return None, "kernel or tile order changed since the stored ncu capture"
    return val, ("stored ncu capture (not measured by this run): " + d.get("what", "") +
                 f"; {os.path.relpath(PAIR_TRAFFIC, ROOT)}")


def reload_measure(layers, ws, ws_bytes, stream, reps=5):
    """Backward pass of every linear with X and dY reloaded per layer through
    LayerReload (1 and 2 buffer sets), and the per-layer copy and compute
    times the pages' model takes."""
    import torch
    from qlora_fine_tuning_gb300 import binding
    from qlora_fine_tuning_gb300.reload import LayerReload, model_double_buffer, model_single_buffer

    def pinned(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).pin_memory()

    host = [[pinned(L["li"].X), pinned(L["li"].dY)] for L in layers]
    order = list(reversed(range(len(layers))))
    for L in layers:  # XA of every layer, resident
        li = L["li"]
        binding.qlora_linear_fwd(L["X"], li.M, L["w"], L["A"], L["B"], li.r, L["seg"], li.s, L["Y"], L["XA"], ws,
                                 ws_bytes, stream)

    def bwd(i, dev):
        L = layers[i]
        li = L["li"]
        binding.qlora_linear_bwd(dev[1], dev[0], L["XA"], li.M, L["w"], L["A"], L["B"], li.r, L["seg"], li.s,
                                 L["dX"], L["dA"], L["dB"], ws, ws_bytes, stream)

    def timed(fn, on=None):
        s = stream if on is None else on
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        fn()
        b.record(s)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    shapes = [[(L["li"].M, L["li"].K), (L["li"].M, L["li"].N)] for L in layers]
    out = {}
    for nbuf in (1, 2):
        rl = LayerReload(shapes, torch.bfloat16, buffers=nbuf)
        times = []
        for _ in range(reps + 1):
            def one():
                start = torch.cuda.Event()
                start.record(stream)
                rl.copy_stream.wait_event(start)
                rl.run(host, bwd, order=order, stream=stream)
            times.append(timed(one))
        out[nbuf] = statistics.median(times[1:])
        del rl
    # per-layer copy (alone, on a side stream) and compute (alone, inputs resident)
    side = torch.cuda.Stream()
    c_ms, g_ms = [], []
    for i in order:
        L = layers[i]
        dX_, dY_ = torch.empty_like(L["X"]), torch.empty_like(L["dY"])
        c_ms.append(statistics.median([_copy_time(side, dX_, dY_, host[i]) for _ in range(reps)]))
        g_ms.append(statistics.median([timed(lambda: bwd(i, [L["X"], L["dY"]])) for _ in range(reps)]))
        del dX_, dY_
    h2d = sum(int(h.numel()) * 2 for pair in host for h in pair)
    return {"what": "backward of every linear in reverse order, X and dY copied per layer from pinned host memory",
            "t_single_ms": round(out[1], 4), "t_double_ms": round(out[2], 4),
            "saved_ms": round(out[1] - out[2], 4),
            "model_single_ms": round(model_single_buffer(c_ms, g_ms), 4),
            "model_double_ms": round(model_double_buffer(c_ms, g_ms), 4),
            "model_saved_ms": round(model_single_buffer(c_ms, g_ms) - model_double_buffer(c_ms, g_ms), 4),
            "copy_ms": [round(v, 4) for v in c_ms], "compute_ms": [round(v, 4) for v in g_ms],
            "h2d_bytes": h2d, "h2d_gbs": round(h2d / (sum(c_ms) * 1e-3) / 1e9, 1)}


def _copy_time(side, d0, d1, host_pair):
    import torch
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(side):
        a.record(side)
        d0.copy_(host_pair[0], non_blocking=True)
        d1.copy_(host_pair[1], non_blocking=True)
        b.record(side)
    torch.cuda.synchronize()
    return a.elapsed_time(b)


def hbm_bytes_per_step(lins, wd_in_rankr: bool) -> dict:
    """Algorithmic bytes per step of the HBM-bound launches (each operand read
    and each output written once; bf16 = 2 B, fp32 = 4 B).  The Wd expansion
    (codes 0.5 B + absmax 4/64 B read, 2 B written, per weight, once in the
    forward and once in the backward) counts in the XA / G launches when they
    write Wd, else in the dequant4 launches."""
    wd = sum(li.N * li.K * (0.5 + 4 / 64 + 2) for li in lins)
    return {
        "gemm_xa": sum(2 * li.M * li.K + 2 * li.K * li.R + 4 * li.M * li.R for li in lins)
        + (wd if wd_in_rankr else 0),
        "gemm_g": sum(2 * li.M * li.N + 2 * li.r * li.N + 4 * li.M * li.R for li in lins)
        + (wd if wd_in_rankr else 0),
        "gemm_dadb": sum(2 * li.M * li.K + 2 * li.M * li.N + 4 * li.M * li.R + 4 * li.K * li.R + 4 * li.r * li.N
                         for li in lins),
        "dequant4": 0 if wd_in_rankr else 2 * wd,
    }


def hbm_bound_rows(lins, ktimes, prof_steps, hbm_peak):
    """Per HBM-bound kernel of the step: launches, algorithmic bytes, event
    time, GB/s and fraction of the measured copy bandwidth; `ktimes` maps a
    kernel label to (launches, total ms) over `prof_steps` steps.  Without a
    dequant4 launch in the step, Wd was written by the rank-r launches."""
    wd_in_rankr = ktimes.get("dequant4", (0, 0.0))[0] == 0
    rows = {}
    for name, b in hbm_bytes_per_step(lins, wd_in_rankr).items():
        n, ms = ktimes.get(name, (0, 0.0))
        if n == 0 or ms <= 0:
            continue
        gbs = b * prof_steps / (ms * 1e-3) / 1e9
        rows[name] = {"launches_per_step": n // prof_steps, "algorithmic_bytes_per_step": int(b),
                      "ms_per_step": round(ms / prof_steps, 4), "achieved": round(gbs, 1),
                      "frac": round(gbs / hbm_peak, 4)}
    hbm_ms = sum(ktimes.get(k, (0, 0.0))[1] for k in ("gemm_xa", "gemm_g", "gemm_dadb", "dequant4"))
    return rows, wd_in_rankr, hbm_ms


def run_ours(args, rank, world):
    import torch
    from qlora_fine_tuning_gb300 import binding
    from qlora_fine_tuning_gb300.dp import AdapterGradReducer, data_parallel_step

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    binding.lib()
    lins = synth.workload(args.workload, seed=0, shard=rank)
    M_all = sum(li.M for li in lins)
    flops = workload_flops(lins)

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)

    ws_bytes = max(binding.qlora_workspace_bytes(li.M, li.N, li.K, li.r, len(li.seg_n)) for li in lins)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    layers = []
    for li in lins:
        L = {"li": li}
        L["idx"] = torch.from_numpy(li.idx).cuda()
        L["absmax"] = torch.from_numpy(li.absmax).cuda()
        L["codebook"] = torch.from_numpy(li.codebook).cuda()
        L["w"] = binding.make_w4(L["idx"], L["absmax"], L["codebook"], li.N, li.K)
        L["X"], L["A"], L["B"], L["dY"] = bf(li.X), bf(li.A), bf(li.B), bf(li.dY)
        L["Y"] = torch.empty((li.M, li.N), dtype=torch.bfloat16, device="cuda")
        L["XA"] = torch.empty((li.M, li.R), dtype=torch.bfloat16, device="cuda")
        L["dX"] = torch.empty((li.M, li.K), dtype=torch.bfloat16, device="cuda")
        L["dA"] = torch.empty((li.K, li.R), dtype=torch.float32, device="cuda")
        L["dB"] = torch.empty((li.r, li.N), dtype=torch.float32, device="cuda")
        L["seg"] = None if len(li.seg_n) == 1 else list(li.seg_n)
        layers.append(L)
    stream = torch.cuda.current_stream()

    reducer = AdapterGradReducer() if world > 1 else None

    def step():
        cur = torch.cuda.current_stream()  # the capture stream while a graph is recorded

        def fwd(i):
            L = layers[i]
            li = L["li"]
            binding.qlora_linear_fwd(L["X"], li.M, L["w"], L["A"], L["B"], li.r, L["seg"], li.s, L["Y"], L["XA"],
                                     ws, ws_bytes, cur)

        def bwd(i):
            L = layers[i]
            li = L["li"]
            binding.qlora_linear_bwd(L["dY"], L["X"], L["XA"], li.M, L["w"], L["A"], L["B"], li.r, L["seg"], li.s,
                                     L["dX"], L["dA"], L["dB"], ws, ws_bytes, cur)

        data_parallel_step(len(layers), fwd, bwd, lambda i: [layers[i]["dA"], layers[i]["dB"]], reducer)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = binding.qlora_check_device_error(ws)
    if st != binding.OK:
        raise RuntimeError(f"device error after warm-up: {binding.STATUS[st]}")

    # One step recorded as a CUDA graph (the library's launches are plain
    # stream launches, so they capture as they are); replaying it removes the
    # host launch path from the timed region.
    graph = None
    per_step_launches = None
    if not args.no_graph and world == 1:  # with ranks, the collectives run outside a graph
        c0 = binding.qlora_launch_counter()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        per_step_launches = binding.qlora_launch_counter() - c0
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()

    # ---- timed region: device-resident inputs ----
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    time.sleep(0.3)
    launches0 = binding.qlora_launch_counter()
    barrier(world)
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    launches = binding.qlora_launch_counter() - launches0
    if graph is not None:
        launches = per_step_launches * args.steps
    ms_total = ev0.elapsed_time(ev1)
    clk = clocks.stop()
    # ---- the same steps again with CUDA events around every library launch ----
    # (kept out of the timed region above: an event between two launches
    # stops the second from overlapping the first one's tail)
    binding.qlora_profiler_enable(True)
    binding.qlora_profiler_collect()
    prof_steps = max(1, min(args.steps, 50))
    torch.cuda.synchronize()
    pt0 = time.perf_counter()
    for _ in range(prof_steps):
        step()
    torch.cuda.synchronize()
    prof_ms = (time.perf_counter() - pt0) * 1e3
    kstats = binding.qlora_profiler_collect()
    binding.qlora_profiler_enable(False)
    st = binding.qlora_check_device_error(ws)
    if st != binding.OK:
        raise RuntimeError(f"device error in timed region: {binding.STATUS[st]}")
    ms_total = max_over_ranks(ms_total, world)
    ms_step = ms_total / args.steps
    value = flops * world / (ms_step * 1e-3) / 1e12

    # ---- the same step with L2 flushed before each one (every input cold) ----
    # The main figure needs no flush (each linear's X and dY, 67-235 MB, are
    # larger than the 129 MB L2); this one also evicts the weights and the
    # adapters: a 256 MB buffer is written before every step, outside the
    # events that time the step.
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    fl_steps = max(3, min(args.steps, 30))
    fl_ev = []
    for _ in range(fl_steps):
        flush.fill_(1)
        fa, fb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        fa.record(stream)
        if graph is not None:
            graph.replay()
        else:
            step()
        fb.record(stream)
        fl_ev.append((fa, fb))
    torch.cuda.synchronize()
    fl_ms = statistics.median(a.elapsed_time(b) for a, b in fl_ev)
    fl_ms = max_over_ranks(fl_ms, world)
    del flush
    l2f = {"value": round(flops * world / (fl_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
           "ms_per_step": round(fl_ms, 4), "steps": fl_steps,
           "how": "median of single steps, each preceded by a 256 MB write (2x L2) outside its CUDA events"}

    # ---- roofline of the dominant kernel (the tcgen05 base GEMM) ----
    peaks, peak_src = measured_peaks()
    ktimes = {name: (n, ms) for name, n, ms in kstats}
    main_flops_step = 0
    for li in lins:
        main_flops_step += 2 * li.M * li.N * li.K + 2 * li.M * li.r * li.N      # forward GEMM + rank-r steps
        main_flops_step += 2 * li.M * li.N * li.K + 2 * li.M * li.R * li.K      # dX GEMM + rank-r steps
    main_ms = sum(ktimes.get(k, (0, 0.0))[1] for k in ("gemm_fwd", "gemm_dx"))
    main_launches = sum(ktimes.get(k, (0, 0.0))[0] for k in ("gemm_fwd", "gemm_dx"))
    achieved = main_flops_step * prof_steps / (main_ms * 1e-3) / 1e12 if main_ms > 0 else None
    peak = float(peaks.get("bf16_tflops", 1900.0))
    peak_sus = float(peaks.get("bf16_tflops_sustained", peak))
    traffic, traffic_note = pair_traffic(args.workload)
    # A, B and C once per launch, averaged over the step's launches: with the
    # bf16 dequantised weight the kernel reads (2 B per weight), and with the
    # stored 4-bit weight (codes 0.5 B + absmax 4/64 B per weight)
    nl2 = 2 * len(lins)
    alg_bytes = sum(2 * (2 * li.M * li.K + 2 * li.N * li.K + 2 * li.M * li.N) for li in lins) / nl2
    alg_bytes_4bit = sum(2 * (2 * li.M * li.K + li.N * li.K * (0.5 + 4 / 64) + 2 * li.M * li.N) for li in lins) / nl2
    roofline = {
        "kernel": "gemm_pair_kernel (forward Y and backward dX instances)",
        "bound": "tensor",
        "achieved": round(achieved, 2) if achieved else None,
        "peak": peak,
        "peak_source": f"{peak_src} bf16_tflops (burst: a cuBLAS bf16 GEMM timed alone)",
        "unit": "TFLOP/s",
        "frac": round(achieved / peak, 4) if achieved else None,
        "frac_sustained": round(achieved / peak_sus, 4) if achieved else None,
        "peak_sustained": peak_sus,
        "traffic": traffic,
        "traffic_note": traffic_note,
        "algorithmic_bytes_per_launch": int(alg_bytes),
        "algorithmic_bytes_per_launch_4bit_weight": int(alg_bytes_4bit),
        "launches": main_launches,
        "avg_launch_ms": round(main_ms / max(1, main_launches), 4),
        "timing": f"CUDA events around each launch on the launching stream, {prof_steps} steps "
                  f"({prof_ms / 1e3:.2f} s) run right after the timed region",
    }
    total_kernel_ms = sum(ms for _, _, ms in kstats)
    breakdown = {name: {"launches": n, "ms_per_step": round(ms / prof_steps, 4),
                        "share": round(ms / total_kernel_ms, 4) if total_kernel_ms else None}
                 for name, n, ms in kstats}

    # ---- end to end: pinned host inputs -> device, result gradients back ----
    # Host-to-device copies of the next inputs overlap compute (a copy stream
    # and two alternating sets of device input buffers), as in the pages'
    # double-buffered asynchronous reload; dA / dB go back on a third stream.
    e2e = None
    if not args.no_e2e:
        nl = len(layers)
        hX = [torch.from_numpy(np.ascontiguousarray(L["li"].X).view(np.int16)).view(torch.bfloat16).pin_memory()
              for L in layers]
        hdY = [torch.from_numpy(np.ascontiguousarray(L["li"].dY).view(np.int16)).view(torch.bfloat16).pin_memory()
               for L in layers]
        bufX = [[torch.empty_like(L["X"]) for L in layers] for _ in range(2)]
        bufdY = [[torch.empty_like(L["dY"]) for L in layers] for _ in range(2)]
        hdA = [torch.empty(L["dA"].shape, dtype=torch.float32).pin_memory() for L in layers]
        hdB = [torch.empty(L["dB"].shape, dtype=torch.float32).pin_memory() for L in layers]
        h2d = sum(t.numel() * 2 for t in hX) + sum(t.numel() * 2 for t in hdY)
        d2h = sum(t.numel() * 4 for t in hdA) + sum(t.numel() * 4 for t in hdB)
        up = torch.cuda.Stream()
        down = torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()  # noqa: E731
        ev_x = [[ev() for _ in range(nl)] for _ in range(2)]
        ev_dy = [[ev() for _ in range(nl)] for _ in range(2)]
        ev_free = [[None] * nl for _ in range(2)]   # compute finished with buffer set b, linear i
        ev_bwd = [ev() for _ in range(nl)]
        ev_back = [None] * nl                        # dA/dB of linear i copied back

        def e2e_step(sidx):
            b = sidx % 2
            with torch.cuda.stream(up):
                for i in range(nl):
                    if ev_free[b][i] is not None:
                        up.wait_event(ev_free[b][i])
                    bufX[b][i].copy_(hX[i], non_blocking=True)
                    ev_x[b][i].record(up)
                for i in reversed(range(nl)):
                    bufdY[b][i].copy_(hdY[i], non_blocking=True)
                    ev_dy[b][i].record(up)
            for i, L in enumerate(layers):
                li = L["li"]
                stream.wait_event(ev_x[b][i])
                binding.qlora_linear_fwd(bufX[b][i], li.M, L["w"], L["A"], L["B"], li.r, L["seg"], li.s, L["Y"],
                                         L["XA"], ws, ws_bytes, stream)
            for i in reversed(range(nl)):
                L = layers[i]
                li = L["li"]
                stream.wait_event(ev_dy[b][i])
                if ev_back[i] is not None:
                    stream.wait_event(ev_back[i])   # previous dA/dB of this linear copied out
                binding.qlora_linear_bwd(bufdY[b][i], bufX[b][i], L["XA"], li.M, L["w"], L["A"], L["B"], li.r,
                                         L["seg"], li.s, L["dX"], L["dA"], L["dB"], ws, ws_bytes, stream)
                if reducer is not None:  # summed over the ranks before they go back to the host
                    reducer.submit([L["dA"], L["dB"]], after=stream)
                ev_bwd[i].record(stream)
                fr = ev()
                fr.record(stream)
                ev_free[b][i] = fr
                with torch.cuda.stream(down):
                    down.wait_event(ev_bwd[i])
                    if reducer is not None:
                        reducer.wait()  # the copy stream waits for the sums
                    hdA[i].copy_(L["dA"], non_blocking=True)
                    hdB[i].copy_(L["dB"], non_blocking=True)
                    bk = ev()
                    bk.record(down)
                    ev_back[i] = bk

        for w_ in range(2):
            e2e_step(w_)
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(up)
        stream.wait_event(e0)
        down.wait_event(e0)
        for k in range(args.steps):
            e2e_step(k)
        done_c = ev()
        done_c.record(stream)
        down.wait_event(done_c)
        down.wait_event(up.record_event())
        e1.record(down)
        torch.cuda.synchronize()
        barrier(world)
        ems = max_over_ranks(e0.elapsed_time(e1), world) / args.steps
        e2e = {"value": round(flops * world / (ems * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
               "ms_per_step": round(ems, 4), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "what": "per step: X and dY of every linear copied from pinned host memory (copy stream, "
                       "double-buffered, overlapping compute), fwd+bwd through the C ABI, dA and dB copied back"}
        st = binding.qlora_check_device_error(ws)
        if st != binding.OK:
            raise RuntimeError(f"device error in e2e region: {binding.STATUS[st]}")

    # ---- saved activations reloaded per layer (the pages' double buffer) ----
    # The backward pass of every linear, in reverse order, with X and dY coming
    # from pinned host memory through qlora_fine_tuning_gb300.reload (XA stays
    # resident from a forward pass): one buffer set (copy, then compute) against
    # two (the copy of the next layer under the compute of this one), beside
    # the pages' model built from each layer's copy time c and compute time g
    # measured alone.
    reload_row = None
    if not args.no_e2e:
        reload_row = reload_measure(layers, ws, ws_bytes, stream)

    # ---- the storage step that feeds the path: GPU 4-bit quantisation ----
    # HBM-bound: reads 4 B (fp32 W) and writes 0.5 B of codes + 4/64 B of
    # absmax per weight.  Timed alone on the largest weight of the workload
    # (fresh seeded fp32 W on the device), against the measured copy bandwidth.
    qli = max(lins, key=lambda li: li.N * li.K)
    gq = torch.Generator(device="cuda")
    gq.manual_seed(1234 + rank)
    Wq = torch.randn((qli.N, qli.K), generator=gq, device="cuda", dtype=torch.float32) * 0.02
    q_idx = torch.empty((qli.N, qli.K // 2), dtype=torch.uint8, device="cuda")
    q_am = torch.empty((qli.N * qli.K // 64,), dtype=torch.float32, device="cuda")
    q_cb = layers[0]["codebook"]
    for _ in range(3):
        binding.quantize_4bit(Wq, False, qli.N, qli.K, q_cb, q_idx, q_am, stream)
    q_reps = 20
    torch.cuda.synchronize()
    # per-launch CUDA events (the library profiler), as for the step's kernels
    binding.qlora_profiler_enable(True)
    binding.qlora_profiler_collect()
    for _ in range(q_reps):
        binding.quantize_4bit(Wq, False, qli.N, qli.K, q_cb, q_idx, q_am, stream)
    torch.cuda.synchronize()
    q_stats = {n: (c, ms) for n, c, ms in binding.qlora_profiler_collect()}
    binding.qlora_profiler_enable(False)
    q_ms = q_stats["quantize4"][1] / q_stats["quantize4"][0]
    q_bytes = qli.N * qli.K * (4 + 0.5 + 4 / 64)
    q_gbs = q_bytes / (q_ms * 1e-3) / 1e9
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    hbm_rows, wd_in_rankr, hbm_ms = hbm_bound_rows(lins, ktimes, prof_steps, hbm_peak)
    other_rows = {
        "quantize_4bit": {"shape": f"{qli.N}x{qli.K} fp32", "ms": round(q_ms, 4), "bound": "hbm",
                          "achieved": round(q_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                          "frac": round(q_gbs / hbm_peak, 4),
                          "algorithmic_bytes": int(q_bytes),
                          "timing": f"CUDA events around each of {q_reps} launches"},
        "hbm_bound_kernels": {"bound": "hbm", "peak": hbm_peak, "unit": "GB/s", "kernels": hbm_rows,
                              "wd_written_by": "gemm_xa / gemm_g" if wd_in_rankr else "dequant4",
                              "share_of_kernel_time": round(hbm_ms / total_kernel_ms, 4) if total_kernel_ms else None,
                              "timing": "CUDA events around each launch inside the profiled steps"},
    }
    del Wq

    out = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded numpy PCG64; shapes and value distributions of the pages' workloads)",
        "config": config_of(args.workload, lins, world),
        "pct_of_bf16_peak": round(100.0 * value / world / peak, 2),
        "pct_of_bf16_peak_sustained": round(100.0 * value / world / peak_sus, 2),
        "l2_flushed": l2f,
        "roofline": roofline,
        "kernels": breakdown,
        "gpu_launches": int(launches),
        "cuda_graph": graph is not None,
        "clocks": clk,
        "e2e": e2e,
        "other_rows": other_rows,
        "reload": reload_row,
    }
    return out, lins


# --------------------------------------------------------------------------
# the CPU oracle (baseline arm / reference arm)
# --------------------------------------------------------------------------

def oracle_sample_run(lins, rows_per_linear):
    """fwd + bwd of every linear on its first `rows` tokens, fp64 oracle."""
    import oracle
    flops = 0
    t0 = time.perf_counter()
    for li in lins:
        m = min(rows_per_linear, li.M)
        _, w16 = oracle.dequant(li.idx, li.absmax, li.codebook, li.N, li.K)
        X = oracle.bf16_to_f64(li.X[:m])
        dY = oracle.bf16_to_f64(li.dY[:m])
        seg = None if len(li.seg_n) == 1 else li.seg_n
        oracle.linear_full(X, oracle.bf16_to_f64(w16), oracle.bf16_to_f64(li.A), oracle.bf16_to_f64(li.B), dY,
                           li.r, li.s, seg_n=seg)
        flops += synth.flops_fwd_bwd(m, li.N, li.K, li.r, len(li.seg_n))
    return flops, time.perf_counter() - t0


def host_cpu() -> dict:
    """The host's cores as the OS reports them (nproc, lscpu)."""
    info = {"nproc": len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count(),
            "logical_cpus": os.cpu_count()}
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            key, _, val = line.partition(":")
            key = key.strip()
            if key in ("Architecture", "Model name", "Socket(s)", "Core(s) per socket", "Thread(s) per core"):
                info[key.lower().replace("(s)", "s").replace(" ", "_")] = val.strip()
    except (OSError, subprocess.SubprocessError):
        info["lscpu"] = "unavailable"
    return info


def oracle_single_thread():
    """The oracle on one core: the tiny workload in full and a row sample of
    the Llama-3-8B q_proj workload (GFLOP/s, dequant included in the time)."""
    import oracle
    nt = oracle.num_threads()
    out = {}
    try:
        oracle.set_num_threads(1)
        for name, rows in (("tiny-m256-k1024-n1024-r8", 256), ("llama3-8b-q_proj-m4096-k4096-n4096-r16", 16)):
            lins = synth.workload(name, seed=0)
            f, t = oracle_sample_run(lins, rows)
            out[name] = {"rows": min(rows, lins[0].M), "of": lins[0].M, "gflop": round(f / 1e9, 3),
                         "seconds": round(t, 3), "gflops": round(f / t / 1e9, 3)}
    finally:
        oracle.set_num_threads(nt)
    return out


def cpu_baseline(lins, target_s):
    import oracle
    oracle.build()
    # calibration: the dequant of every weight is a fixed cost, the rows add linearly
    # (rows >= the thread count, so both calibration runs keep every core busy)
    nt = max(1, oracle.num_threads())
    r1, r2 = nt, 2 * nt
    _, t1 = oracle_sample_run(lins, r1)
    _, t2 = oracle_sample_run(lins, r2)
    per_row = max((t2 - t1) / (r2 - r1), 1e-4)
    rows = int(max(r1, min(1024, r1 + (target_s - t1) / per_row)))
    f, t = oracle_sample_run(lins, rows)
    rows = min(rows, lins[0].M)
    return {"value": round(f / t / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"fwd+bwd of every linear on its first {rows} tokens (of {lins[0].M}); "
                      f"{f / 1e9:.1f} GFLOP in {t:.1f} s, fp64, dequant included in the time",
            "seconds": round(t, 2), "host": host_cpu(), "single_thread": oracle_single_thread()}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    lins = synth.workload(args.workload, seed=0)
    import oracle
    oracle.build()
    # one step = the oracle's fwd+bwd over a bounded sample of the workload
    f1, t1 = oracle_sample_run(lins, 2)
    total_budget = 150.0
    per_step = total_budget / max(1, args.steps + args.warmup)
    rows = int(max(1, min(128, 2 * per_step / max(t1, 1e-3))))
    for _ in range(args.warmup):
        oracle_sample_run(lins, rows)
    times, fl = [], 0
    for _ in range(args.steps):
        f, t = oracle_sample_run(lins, rows)
        times.append(t)
        fl = f
    tot = sum(times)
    value = fl * args.steps / tot / 1e12
    ms_step = tot / args.steps * 1e3
    sample = f"fwd+bwd of every linear on its first {rows} tokens (of {lins[0].M}), fp64 oracle"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(args.workload, lins, world),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample, "host": host_cpu()},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    if args.warmup < 3:
        args.warmup = 3
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(relaunch(args.gpus))
    rank, world = dist_init(args.gpus)
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if rank == 0 and out is not None:
            print(json.dumps(out), flush=True)
        return
    out, lins = run_ours(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            out["cpu_baseline"] = cpu_baseline(lins, args.cpu_seconds)
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
