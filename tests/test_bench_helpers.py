"""The benchmark's reporting helpers, on the CPU: the algorithmic byte and
FLOP counts of the roofline, the bound it picks, the gate that keeps ncu
traffic only for the captured build, the clock summary that decides whether
a run is kept, and the default workload of the bench line."""
import os

import pytest

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


def test_useful_flops_exclude_padding_rows_and_masked_tails():
    w = wl.WORKLOADS["contig"]
    assert bench.useful_flops(w) == 2.0 * w.tokens * w.N * w.K
    w = wl.WORKLOADS["masked"]
    assert bench.useful_flops(w) == 2.0 * int(wl.masked_counts(w.G, w.max_m, w.seed).sum()) * w.N * w.K
    w = wl.WORKLOADS["sweep_n7168_k18432"]
    assert bench.useful_flops(w) == 2.0 * 4096 * 7168 * 18432


def test_roofline_picks_the_slower_of_compute_and_bytes():
    # the contiguous MoE GEMM is tensor-bound, the skinny and masked ones HBM-bound
    hbm, fp8 = 6797.2, 3791.4
    for name, bound in [("contig", "tensor"), ("sweep_n2112_k7168", "tensor"), ("skinny", "hbm"), ("masked", "hbm")]:
        w = wl.WORKLOADS[name]
        r = bench.roofline(bench.useful_flops(w), bench.algorithmic_bytes(w), 1e-3, hbm, fp8)
        assert r["bound"] == bound, name
        assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    r = bench.roofline(2e12, 1e6, 1e-3, hbm, fp8)
    assert r["unit"] == "TFLOP/s" and r["achieved"] == pytest.approx(2000.0)
    r = bench.roofline(1e6, 5e9, 1e-3, hbm, fp8)
    assert r["unit"] == "GB/s" and r["achieved"] == pytest.approx(5000.0)


def test_quantiser_bytes():
    # fp32 in, one code byte out and one fp32 scale per 128 values
    assert bench.quant_bytes(256, 2048) == 256 * 2048 * 5 + 256 * 16 * 4


def test_default_bench_line_is_the_contiguous_moe_workload():
    args = bench.parse([])
    assert args.workload == "contig" and args.gpus == 1 and args.warmup >= 3
    w = wl.WORKLOADS[args.workload]
    assert (w.layout, w.G, w.tokens, w.N, w.K) == ("contiguous", 8, 32768, 4096, 7168)
    # every other workload is measured in the same run
    assert set(bench.EXTRA) | {"contig"} == set(wl.WORKLOADS)


def test_reduced_token_count_is_a_profiling_variant_only():
    w = bench.with_tokens(wl.WORKLOADS["contig"], 4096)
    assert w.tokens == 4096 and w.name != "contig" and w.N == 4096 and w.K == 7168
    assert bench.with_tokens(wl.WORKLOADS["skinny"], 4096) is wl.WORKLOADS["skinny"]


def test_both_arms_print_the_same_config():
    """The reference arm's config is the GPU arm's: same workload text, L2
    note and input fingerprints, computed from the same seeded host inputs."""
    w = wl.WORKLOADS["skinny"]
    x, wt, meta = bench.host_inputs(w)
    cfg = bench.run_config(w, x, wt, meta, 1)
    assert set(cfg) == {"workload", "l2", "inputs_sha256", "parallelism"}
    assert cfg == bench.run_config(w, *bench.host_inputs(w), 1)          # deterministic
    set_bytes, n_sets = bench.input_sets(w, x.nbytes)
    assert n_sets * set_bytes >= 2 * bench.L2_BYTES and cfg["l2"] == bench.l2_note(set_bytes, n_sets)
    assert cfg["parallelism"] == "single GPU" and bench.run_config(w, x, wt, meta, 2)["parallelism"] == "replicas"
    # a different seed changes the fingerprints
    x2, wt2 = wl.dense_inputs(w.M, w.N, w.K, w.seed + 1, w.outliers)
    assert bench.input_fingerprints(x2, wt2, None) != cfg["inputs_sha256"]
