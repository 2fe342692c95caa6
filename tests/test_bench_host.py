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
