"""Benchmark of the FP8 fine-grained-scaled GEMM hot path on GB300.

One step = the whole path over one batch: 1x128 quantisation of the fp32
activations (dg_quant_act_1x128) followed by the FP8 GEMM with two-level
accumulation and bf16 output (dg_fp8_gemm_nt); the weights are quantised once,
offline, before timing (dg_quant_weight_128x128).  Default workload: the
skinny dense GEMM M=256, N=7168, K=2048 with 1% x20 outliers in A.

Prints ONE JSON line (rank 0).  --impl reference times the CPU oracle on the
host cores instead (a bounded row sample of the same workload).
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

import workloads as wl  # noqa: E402

METRIC = "FP8 GEMM TFLOPS (2MNK) and fraction of GB300 FP8/HBM roofline, 1 GPU"
UNIT = "TFLOP/s"
FP8_PER_BF16 = 2.0           # nominal dense fp8 : bf16 tensor ratio (4.5 : 2.25 PFLOP/s)
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129 * 2 ** 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="dg", choices=["dg", "reference"])
    ap.add_argument("--workload", default="skinny", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--shape", default="", help="M,N,K: a dense problem of this shape instead of the workload "
                                                 "(profiling aid; not a bench line)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# ---------------------------------------------------------------- clocks --
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = max(smax, float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- workload ---
def describe(w: wl.Workload) -> str:
    if w.layout == "dense":
        return (f"dense NT FP8 GEMM M={w.M} N={w.N} K={w.K}" + (" (1% x20 outliers in A)" if w.outliers else "")
                + "; step = 1x128 activation quantisation + GEMM")
    if w.layout == "contiguous":
        return f"MoE contiguous FP8 GEMM G={w.G} tokens={w.tokens} N={w.N} K={w.K}; step = quantisation + GEMM"
    return f"MoE masked FP8 GEMM G={w.G} max_m={w.max_m} N={w.N} K={w.K}; step = quantisation + GEMM"


def gemm_shape(w: wl.Workload):
    """(rows of A, useful rows, N, K, G)."""
    if w.layout == "dense":
        return w.M, w.M, w.N, w.K, 1
    if w.layout == "contiguous":
        counts, m_indices, _ = wl.contiguous_routing(w.G, w.tokens, w.seed)
        return len(m_indices), int(counts.sum()), w.N, w.K, w.G
    mm = wl.masked_counts(w.G, w.max_m, w.seed)
    return w.G * w.max_m, int(mm.sum()), w.N, w.K, w.G


def algorithmic_bytes(w: wl.Workload):
    """Bytes the GEMM must move at least once: A + B (+ scales) + D, counting
    only useful rows and experts that have any."""
    rows_total, useful, N, K, G = gemm_shape(w)
    KB = K // 128
    NB = -(-N // 128)
    if w.layout == "masked":
        mm = wl.masked_counts(w.G, w.max_m, w.seed)
        experts = int((mm > 0).sum())
    else:
        experts = G
    return useful * K + experts * N * K + useful * KB * 4 + experts * NB * KB * 4 + useful * N * 2


# -------------------------------------------------------- ncu traffic ------
GEMM_SOURCES = ("dg_common.h", "dg_gemm.cu", "dg_ptx.cuh")


def gemm_source_hash() -> str:
    """First 16 hex digits of the SHA-256 of the GEMM kernel's sources with
    comments and blank lines removed (what the compiler sees changes the hash;
    an edited comment does not)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, "moe_grouped_gemm_x128_gb300", "csrc", f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines()]
        h.update("\n".join(ln for ln in lines if ln.strip()).encode())
    return h.hexdigest()[:16]


def measured_traffic(profile: str):
    """DRAM bytes per launch from a committed ncu summary, if that summary was
    taken from the kernel as it is now (its source hash matches), else None."""
    fields = {}
    try:
        with open(os.path.join(ROOT, "profiles", profile)) as fh:
            for line in fh:
                if ":" in line and not line.startswith(("|", "#", " ")):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
    except OSError:
        return None
    if fields.get("source_sha256") != gemm_source_hash() or "dram_bytes_per_launch" not in fields:
        return None
    return int(fields["dram_bytes_per_launch"])


# ------------------------------------------------------------- replicas ----
def max_over_ranks(value: float, device=None) -> float:
    """The largest value over all ranks (the job's time is its slowest
    replica's); a no-op without an initialised process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, units_per_rank_step: float, steps: int, max_ms: float) -> float:
    """Whole-job rate: every replica processes its own units; the job takes
    the slowest replica's time (weak scaling, no data-path collective)."""
    return world * units_per_rank_step * steps / (max_ms * 1e-3)


# ---------------------------------------------------------------- CPU leg --
def cpu_oracle_rate(w: wl.Workload, seconds: float):
    """Time the oracle (quantise + GEMM) over whole rows of the workload,
    repeating the full row range until about `seconds` have passed; returns
    (TFLOP/s, rows computed, elapsed s, threads)."""
    import oracle
    if w.layout != "dense":
        raise SystemExit("the CPU baseline leg covers the dense workloads")
    x, wt = wl.dense_inputs(w.M, w.N, w.K, w.seed, w.outliers)
    qb, sfb = oracle.quant_weight_128x128(wt)
    rows_done, elapsed, chunk, r0 = 0, 0.0, 8, 0
    while elapsed < seconds:
        r1 = min(w.M, r0 + chunk)
        t0 = time.perf_counter()
        qa, sfa = oracle.quant_act_1x128(x[r0:r1])
        oracle.gemm_nt(qa, sfa, qb, sfb)
        elapsed += time.perf_counter() - t0
        rows_done += r1 - r0
        r0 = 0 if r1 >= w.M else r1
        chunk = min(chunk * 2, 64)
    flops = 2.0 * rows_done * w.N * w.K
    return flops / elapsed / 1e12, rows_done, elapsed, oracle.num_threads()


def run_reference(args, w):
    """The oracle as it stands, timed on the host cores: every step quantises
    and multiplies a bounded sample of the workload (up to one row per oracle
    thread, and as many output columns as fit the per-step share of a two
    minute budget); the value is the sampled FLOPs over the sampled time."""
    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    if w.layout != "dense":
        raise SystemExit("the CPU reference arm covers the dense workloads")
    x, wt = wl.dense_inputs(w.M, w.N, w.K, w.seed, w.outliers)
    qb, sfb = oracle.quant_weight_128x128(wt)
    thr = oracle.num_threads()
    rows = min(w.M, thr)
    per_step = 120.0 / (args.steps + args.warmup)
    # calibrate the output-element rate on one 128-column slice
    t0 = time.perf_counter()
    qa, sfa = oracle.quant_act_1x128(x[:rows])
    oracle.gemm_nt(qa, sfa, qb[:128], sfb[:1])
    rate = rows * 128 / max(time.perf_counter() - t0, 1e-6)
    cols = int(max(8, min(w.N, rate * per_step / rows)) // 8 * 8)
    nbs = -(-cols // 128)
    flops = 0.0
    elapsed = 0.0
    for i in range(args.warmup + args.steps):
        r0 = (i * rows) % w.M
        xr = x[r0:r0 + rows]
        t0 = time.perf_counter()
        qa, sfa = oracle.quant_act_1x128(xr)
        oracle.gemm_nt(qa, sfa, np.ascontiguousarray(qb[:cols]), np.ascontiguousarray(sfb[:nbs]))
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            elapsed += dt
            flops += 2.0 * len(xr) * cols * w.K
    value = flops / elapsed / 1e12
    rows_total = gemm_shape(w)[0]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 block sums, fp32 promotion",
        "data": "synthetic", "config": {"workload": describe(w)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle",
                         "sample": f"per step {rows} of {rows_total} rows x {cols} of {w.N} columns "
                                   f"(quantise + GEMM), {elapsed:.1f} s timed"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU leg --
def run_gpu(args, w):
    import torch
    import torch.distributed as dist

    import moe_grouped_gemm_x128_gb300 as dg

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dg.build()
    dg.load()
    if w.layout != "dense":
        raise SystemExit("bench.py times the dense workloads; grouped layouts are covered by the tests")
    M, N, K = w.M, w.N, w.K
    dev = torch.device("cuda", local)

    # inputs: several independent sets so that consecutive steps do not hit L2
    x_host, w_host = wl.dense_inputs(M, N, K, w.seed, w.outliers)
    set_bytes = M * K * 4 + M * K + N * K + M * N * 2
    n_sets = max(2, -(-2 * L2_BYTES // set_bytes))
    xs, qas, sfas, qbs, sfbs, ds = [], [], [], [], [], []
    wt = torch.from_numpy(w_host).to(dev)
    for i in range(n_sets):
        xs.append(torch.from_numpy(x_host).to(dev))
        qb, sfb = dg.dg_quant_weight_128x128(wt)
        qbs.append(qb)
        sfbs.append(sfb)
        qas.append(torch.empty((M, K), dtype=torch.uint8, device=dev))
        sfas.append(torch.zeros((K // 128, dg.round_up(M, 4)), dtype=torch.float32, device=dev))
        ds.append(torch.empty((M, N), dtype=torch.bfloat16, device=dev))
    del wt
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def quant(i):
        j = i % n_sets
        dg.dg_quant_act_1x128(xs[j], qas[j], sfas[j])

    def gemm(i):
        j = i % n_sets
        dg.dg_fp8_gemm_nt(qas[j], sfas[j], qbs[j], sfbs[j], ds[j])

    def step(i):
        quant(i)
        gemm(i)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    # The steps are launched from a CUDA graph (host launch cost would
    # otherwise dominate microsecond kernels): one graph holds `chunk` steps
    # over the rotating input sets and is replayed until `steps` steps have run.
    chunk = min(args.steps, 100)
    reps = -(-args.steps // chunk)
    steps_run = chunk * reps

    def capture(body):
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for i in range(chunk):
                body(i)
        g.replay()
        torch.cuda.synchronize()
        return g

    def timed(graph, n):
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(stream)
        for _ in range(n):
            graph.replay()
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    g_step = capture(step)
    g_gemm = capture(gemm)
    g_quant = capture(quant)
    with ClockSampler(local) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        total_ms = timed(g_step, reps)
        if world > 1:
            dist.barrier()
    # per-kernel durations: the same launches, one kernel kind per graph
    gemm_ms = timed(g_gemm, reps)
    quant_ms = timed(g_quant, reps)
    total_ms = max_over_ranks(total_ms, device=dev)

    # end to end: pinned host activations in, bf16 result out, every step,
    # through the public API with one launch per call.  Independent steps are
    # pipelined over three streams (copy in, compute, copy out); a buffer set
    # is reused only after its previous step's copy out has completed.
    x_pin = torch.from_numpy(x_host).pin_memory()
    d_pins = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(n_sets)]
    ev_cmp = [torch.cuda.Event() for _ in range(n_sets)]
    ev_out = [torch.cuda.Event() for _ in range(n_sets)]
    used = [False] * n_sets

    def e2e_step(i):
        j = i % n_sets
        if used[j]:
            s_in.wait_event(ev_out[j])
        used[j] = True
        with torch.cuda.stream(s_in):
            xs[j].copy_(x_pin, non_blocking=True)
        ev_in[j].record(s_in)
        s_cmp.wait_event(ev_in[j])
        dg.dg_quant_act_1x128(xs[j], qas[j], sfas[j], stream=s_cmp.cuda_stream)
        dg.dg_fp8_gemm_nt(qas[j], sfas[j], qbs[j], sfbs[j], ds[j], stream=s_cmp.cuda_stream)
        ev_cmp[j].record(s_cmp)
        s_out.wait_event(ev_cmp[j])
        with torch.cuda.stream(s_out):
            d_pins[i % 2].copy_(ds[j], non_blocking=True)
        ev_out[j].record(s_out)

    for i in range(2 * n_sets):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = min(args.steps, 500)
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)

    flops_step = 2.0 * M * N * K
    value = job_throughput(world, flops_step, steps_run, total_ms) / 1e12
    e2e_ms = max_over_ranks(e2e_ms, device=dev)
    e2e_value = job_throughput(world, flops_step, e2e_steps, e2e_ms) / 1e12

    hbm, bf16, bf16_sus, src = peaks()
    fp8_peak = bf16 * FP8_PER_BF16
    gemm_s = gemm_ms / steps_run * 1e-3
    ab = algorithmic_bytes(w)
    t_mem = ab / (hbm * 1e9)
    t_cmp = flops_step / (fp8_peak * 1e12)
    if t_mem >= t_cmp:
        roof = {"bound": "hbm", "achieved": ab / gemm_s / 1e9, "peak": hbm, "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": flops_step / gemm_s / 1e12, "peak": fp8_peak, "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = measured_traffic(f"fp8_gemm_{w.name}_M{M}_N{N}_K{K}.md")
    roof["peak_source"] = f"{src} (MEASURED_PEAKS.json; fp8 = bf16 x {FP8_PER_BF16:g})" if src == "measured" \
        else "fallback"
    roof["kernel"] = "fp8_gemm_kernel"
    roof["kernel_us"] = gemm_s * 1e6
    roof["quant_us"] = quant_ms / steps_run * 1e3
    roof["algorithmic_bytes"] = ab

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps_run,
        "warmup": args.warmup, "ms_per_step": total_ms / steps_run, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": describe(w), "l2": f"rotating {n_sets} input sets of {set_bytes / 1e6:.1f} MB "
                                                  f"(> 2x L2) between steps",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": M * K * 4, "d2h_bytes_per_step": M * N * 2},
        "gpu_launches": 2 * steps_run,
        "launch": f"CUDA graph of {chunk} steps replayed {reps} times; kernel times from graphs of the same "
                  f"launches of one kernel",
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, rows, el, thr = cpu_oracle_rate(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": thr, "kind": "oracle",
                                "sample": f"oracle quantise + GEMM over {rows} rows of the {M}-row workload "
                                          f"(row range repeated, {el:.1f} s of CPU time), rate in TFLOP/s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    w = wl.WORKLOADS[args.workload]
    if args.shape:
        M, N, K = (int(v) for v in args.shape.split(","))
        w = wl.Workload(f"shape_{M}x{N}x{K}", "dense", M=M, N=N, K=K, seed=5)
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_gpu(args, w)


if __name__ == "__main__":
    main()
