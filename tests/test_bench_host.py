"""Host-side checks of bench.py's bookkeeping (no GPU): the FLOP count of the
default workload, and the DRAM-traffic figure it reports from the committed
ncu capture only while the captured sources are unchanged."""
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
    val, note = bench.pair_traffic(bench.DEFAULT_WORKLOAD)
    with open(bench.PAIR_PROFILE) as f:
        matches = bench.pair_sources_sha256() in f.read()
    if matches:   # the committed capture was taken with these sources
        assert isinstance(val, int) and val > 0, note
    else:         # the kernel changed since: no figure rather than a stale one
        assert val is None
    assert bench.pair_traffic("tiny-m256-k1024-n1024-r8")[0] is None


def test_traffic_is_withdrawn_when_the_kernel_source_changes(tmp_path, monkeypatch):
    text = open(bench.PAIR_PROFILE).read().replace(bench.pair_sources_sha256(), "0" * 64)
    p = tmp_path / "profile.md"
    p.write_text(text)
    monkeypatch.setattr(bench, "PAIR_PROFILE", str(p))
    val, note = bench.pair_traffic(bench.DEFAULT_WORKLOAD)
    assert val is None and "changed" in note
