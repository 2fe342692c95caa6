"""Host-side checks of bench.py's bookkeeping (no GPU): the FLOP count of the
default workload, the DRAM-traffic figure it reports from the stored ncu
capture only while the captured sources are unchanged, and the host-core
description of the CPU baseline."""
import bench
from qlora_fine_tuning_gb300 import synth


def test_default_workload_flops():
    lins = [synth.LinearInputs(M=kw["M"], N=kw["N"], K=kw["K"], r=kw["r"], s=kw["s"],
                               seg_n=tuple(kw.get("seg_n", (kw["N"],))), idx=None, absmax=None, codebook=None,
                               X=None, A=None, B=None, dY=None)
            for _, kw in synth.WORKLOADS[bench.DEFAULT_WORKLOAD]]
    # 4MNK + 6Mr(K+N) per linear: 5.946 TFLOP for the Llama-3-8B MLP step
    assert bench.workload_flops(lins) == sum(4 * l.M * l.N * l.K + 6 * l.M * l.r * (l.K + l.N) for l in lins)
    assert abs(bench.workload_flops(lins) / 1e12 - 5.946) < 1e-3


def test_traffic_reported_only_for_the_captured_sources():
    import json
    val, note = bench.pair_traffic(bench.DEFAULT_WORKLOAD)
    with open(bench.PAIR_TRAFFIC) as f:
        matches = json.load(f)["sources_sha256"] == bench.pair_sources_sha256()
    if matches:   # the stored capture was taken with these sources
        assert isinstance(val, int) and val > 0, note
        assert "not measured by this run" in note
    else:         # the kernel changed since: no figure rather than a stale one
        assert val is None
    assert bench.pair_traffic("tiny-m256-k1024-n1024-r8")[0] is None


def test_traffic_is_withdrawn_when_the_kernel_source_changes(tmp_path, monkeypatch):
    import json
    d = json.load(open(bench.PAIR_TRAFFIC))
    d["sources_sha256"] = "0" * 64
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps(d))
    monkeypatch.setattr(bench, "PAIR_TRAFFIC", str(p))
    val, note = bench.pair_traffic(bench.DEFAULT_WORKLOAD)
    assert val is None and "changed" in note


def test_host_cpu_reports_the_core_count():
    info = bench.host_cpu()
    assert info["nproc"] >= 1 and info["logical_cpus"] >= info["nproc"]


def test_traffic_survives_a_comment_edit_but_not_a_code_edit(tmp_path):
    import shutil
    src = tmp_path / "csrc"
    shutil.copytree(bench.os.path.join(bench.ROOT, "qlora_fine_tuning_gb300", "csrc"), src)
    base = bench.pair_sources_sha256(str(src))
    p = src / "gemm_pair.cuh"
    text = p.read_text()
    p.write_text(text.replace("#pragma once", "// a new comment line\n#pragma once", 1))
    assert bench.pair_sources_sha256(str(src)) == base
    p.write_text(text.replace("kDqAhead = 4", "kDqAhead = 5", 1))
    assert bench.pair_sources_sha256(str(src)) != base


def _lin(M, N, K, r, seg=None):
    return synth.LinearInputs(M=M, N=N, K=K, r=r, s=1.0, seg_n=tuple(seg or (N,)), idx=None, absmax=None,
                              codebook=None, X=None, A=None, B=None, dY=None)


def test_hbm_bytes_per_step():
    """The gate linear (M 8192, K 4096, N 14336, r 64) worked by hand: XA reads
    X (2MK) and A (2KR) and writes XA and s*XA (4MR); the Wd expansion reads
    0.5 + 4/64 B and writes 2 B per weight; moving the expansion between
    launches leaves the step's total unchanged."""
    gate = _lin(8192, 14336, 4096, 64)
    with_wd = bench.hbm_bytes_per_step([gate], True)
    assert with_wd["gemm_xa"] == 67108864 + 524288 + 2097152 + 150470656
    assert with_wd["gemm_g"] == 2 * 8192 * 14336 + 2 * 64 * 14336 + 2097152 + 150470656
    assert with_wd["dequant4"] == 0
    sep = bench.hbm_bytes_per_step([gate], False)
    assert sep["dequant4"] == 2 * 150470656
    assert sum(sep.values()) == sum(with_wd.values())
    lins = [_lin(**dict(M=kw["M"], N=kw["N"], K=kw["K"], r=kw["r"]))
            for _, kw in synth.WORKLOADS[bench.DEFAULT_WORKLOAD]]
    assert abs(sum(bench.hbm_bytes_per_step(lins, True).values()) / 1e9 - 2.755) < 1e-3


def test_hbm_bound_rows_from_kernel_times():
    gate = _lin(8192, 14336, 4096, 64)
    steps = 10
    # labels as the library profiler reports them: (launches, total ms)
    kt = {"gemm_xa": (steps, 0.05 * steps), "gemm_g": (steps, 0.07 * steps), "gemm_dadb": (steps, 0.06 * steps),
          "gemm_fwd": (steps, 0.5 * steps)}
    rows, wd_in_rankr, hbm_ms = bench.hbm_bound_rows([gate], kt, steps, 6784.5)
    assert wd_in_rankr and set(rows) == {"gemm_xa", "gemm_g", "gemm_dadb"}
    b = bench.hbm_bytes_per_step([gate], True)["gemm_xa"]
    assert rows["gemm_xa"]["launches_per_step"] == 1
    assert abs(rows["gemm_xa"]["achieved"] - b / 0.05e-3 / 1e9) < 0.1
    assert abs(rows["gemm_xa"]["frac"] - b / 0.05e-3 / 1e9 / 6784.5) < 1e-4
    assert abs(hbm_ms - 0.18 * steps) < 1e-9
    kt["dequant4"] = (2 * steps, 0.048 * steps)
    rows, wd_in_rankr, _ = bench.hbm_bound_rows([gate], kt, steps, 6784.5)
    assert not wd_in_rankr and rows["dequant4"]["launches_per_step"] == 2
