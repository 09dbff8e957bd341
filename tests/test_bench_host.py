"""Host logic of the benchmark (no GPU): the DRAM-traffic figure is reported only while it was
taken on the current kernel sources, the peak's provenance, the workload's name and the job
throughput of replicas."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from block_scaled_bit_gb300 import synth  # noqa: E402


def test_traffic_is_reported_only_for_the_kernel_it_was_taken_on(monkeypatch):
    key = f"config{bench.WORKLOAD_CONFIG}"  # the default workload's record
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)[key]
    assert rec["dram_bytes_per_launch"] >= rec["algorithmic_bytes_per_launch"] * 0.95
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: rec["kernel_hash"])
    assert bench.recorded_traffic(key) == float(rec["dram_bytes_per_launch"])
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)  # sources changed since
    assert bench.recorded_traffic(key) is None
    assert bench.recorded_traffic("no such workload") is None


def test_peak_provenance(tmp_path, monkeypatch):
    value, kind = bench.hbm_peak()
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        assert kind == "measured" and value > 1000
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))  # no measured peaks there
    assert bench.hbm_peak() == (bench.FALLBACK_HBM_GBS, "fallback")


def test_workload_name_and_job_throughput():
    shapes = synth.config_shapes(2)
    name = bench.workload_name(2, shapes, 1)
    assert name.startswith("int8 MatMulNBits GEMV with zero points")
    assert all(f"{s.K}x{s.N} bs{s.block_size}" in name for s in shapes) and "M=1" in name
    # replicas: every rank's bytes over the slowest rank's time
    assert bench.job_throughput_gbps(4, 100, 10 ** 9, 2.0) == 200.0
    assert bench.job_throughput_gbps(1, 100, 10 ** 9, 2.0) == 50.0


def test_default_workload_is_the_int4_M_sweep():
    shapes = synth.config_shapes(bench.WORKLOAD_CONFIG)
    name = bench.workload_name(bench.WORKLOAD_CONFIG, shapes, [1, 2, 4, 8, 16])
    assert name.startswith("int4 MatMulNBits GEMV (zero point fixed at 8)")
    for kn in ("4096x4096", "4096x12288", "12288x4096", "4096x151936"):
        assert f"{kn} bs32" in name and name.count(kn + " ") == 1
    assert "M=1,2,4,8,16" in name and name.endswith("fp16 and bf16")
    assert bench.workload_dtype(shapes) == "u4 weights, bf16 and f16 activations, f32 accumulate"


def test_graphs_cover_exactly_the_requested_steps():
    for steps in (1, 3, 20, 23, 24, 25, 48, 100, 1000):
        S, full, rem = bench.graph_plan(steps)
        assert S * full + rem == steps and 0 <= rem < S and S <= bench.GRAPH_STEPS
    assert bench.GRAPH_STEPS % 2 == 0  # weight copies alternate across graph replays
