"""The benchmark's reporting helpers, on the CPU: the algorithmic byte count
of the roofline, the gate that keeps ncu traffic only for the captured build,
and the clock summary that decides whether a run is kept."""
import os

import bench
import workloads as wl


def test_algorithmic_bytes_of_the_skinny_step():
    # A 256x2048 + B 7168x2048 bytes, SFA 256x16 and SFB 56x16 fp32, D 256x7168 bf16
    w = wl.WORKLOADS["skinny"]
    expect = 256 * 2048 + 7168 * 2048 + 256 * 16 * 4 + 56 * 16 * 4 + 256 * 7168 * 2
    assert bench.algorithmic_bytes(w) == expect == 18894336


def test_algorithmic_bytes_count_only_useful_rows_and_active_experts():
    w = wl.WORKLOADS["masked"]
    mm = wl.masked_counts(w.G, w.max_m, w.seed)
    useful, active = int(mm.sum()), int((mm > 0).sum())
    KB, NB = w.K // 128, -(-w.N // 128)
    expect = useful * w.K + active * w.N * w.K + useful * KB * 4 + active * NB * KB * 4 + useful * w.N * 2
    assert bench.algorithmic_bytes(w) == expect
    rows, useful_c, N, K, G = bench.gemm_shape(wl.WORKLOADS["contig"])
    assert rows % 128 == 0 and useful_c == wl.WORKLOADS["contig"].tokens and G == 8


def test_traffic_is_used_only_for_the_captured_build(tmp_path, monkeypatch):
    # a summary taken from other kernel sources is ignored
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "x.md").write_text("# x\n\nsource_sha256: 0123456789abcdef\ndram_bytes_per_launch: 5\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "gemm_source_hash", lambda: "fedcba9876543210")
    assert bench.measured_traffic("x.md") is None
    monkeypatch.setattr(bench, "gemm_source_hash", lambda: "0123456789abcdef")
    assert bench.measured_traffic("x.md") == 5
    assert bench.measured_traffic("missing.md") is None


def test_clock_summary_reports_median_and_active_reasons():
    c = bench.ClockSampler(0)
    c.lines = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
               "0, 1965, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
               "0, 2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
               "garbage line"]
    s = c.summary()
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    c.lines = ["0, 1500, 2070, 900, 0x8, Active, Not Active, Not Active, Not Active"]
    assert c.summary()["reasons"] == ["hw_slowdown"]
    c.lines = []
    assert c.summary()["reasons"] == ["unavailable"]
