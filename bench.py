"""Benchmark of the FP8 fine-grained-scaled GEMM hot path on GB300.

One step = the whole path over one batch: 1x128 quantisation of the fp32
activations (dg_quant_act_1x128) followed by the FP8 GEMM with two-level
accumulation and bf16 output; the weights are quantised once, offline, before
timing (dg_quant_weight_128x128).  The headline workload is the largest one
that fits one GPU: the contiguous MoE grouped GEMM (G=8 experts, 32768 routed
tokens, N=4096, K=7168).  Every other workload's GEMM (and quantiser, where
it has one) is timed in the same run and reported under "configs".

Prints ONE JSON line (rank 0).  --impl reference times the CPU oracle on the
host cores instead (a bounded row sample of the same workload).
"""
from __future__ import annotations

import argparse
import hashlib
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
HEADLINE = "contig"
EXTRA = ("tiny", "skinny", "sweep_n7168_k18432", "sweep_n24576_k1536", "sweep_n2112_k7168", "masked")


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="dg", choices=["dg", "reference"])
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--tokens", type=int, default=0,
                    help="contiguous workload: routed tokens (0 = the workload's 32768); a profiling aid")
    ap.add_argument("--shape", default="", help="M,N,K: a dense problem of this shape instead of the workload "
                                                 "(profiling aid; not a bench line)")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--profile-next", default="", choices=["", "bf16", "mx", "requant"],
                    help="run only the BF16, MX or re-quantised-output leg (profiling aid; not a bench line)")
    return ap.parse_args(argv)


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
def with_tokens(w: wl.Workload, tokens: int) -> wl.Workload:
    if not tokens or w.layout != "contiguous":
        return w
    return wl.Workload(f"{w.name}_t{tokens}", w.layout, N=w.N, K=w.K, G=w.G, tokens=tokens, seed=w.seed)


def describe(w: wl.Workload) -> str:
    if w.layout == "dense":
        return (f"dense NT FP8 GEMM M={w.M} N={w.N} K={w.K}" + (" (1% x20 outliers in A)" if w.outliers else "")
                + "; step = 1x128 activation quantisation + GEMM")
    if w.layout == "contiguous":
        return (f"MoE contiguous grouped FP8 GEMM G={w.G} tokens={w.tokens} N={w.N} K={w.K} (expert popularity "
                f"spanning 10x, segments padded to 128 rows); step = 1x128 activation quantisation + GEMM")
    return (f"MoE masked grouped FP8 GEMM G={w.G} max_m={w.max_m} N={w.N} K={w.K}, masked_m ~ U{{0..{w.max_m}}} "
            f"on the device; CUDA-graph captured GEMM")


def gemm_shape(w: wl.Workload):
    """(rows of A, useful rows, N, K, G)."""
    if w.layout == "dense":
        return w.M, w.M, w.N, w.K, 1
    if w.layout == "contiguous":
        counts, m_indices, _ = wl.contiguous_routing(w.G, w.tokens, w.seed)
        return len(m_indices), int(counts.sum()), w.N, w.K, w.G
    mm = wl.masked_counts(w.G, w.max_m, w.seed)
    return w.G * w.max_m, int(mm.sum()), w.N, w.K, w.G


def useful_flops(w: wl.Workload) -> float:
    """2 M N K over the useful rows only (padding rows and masked tails excluded)."""
    _, useful, N, K, _ = gemm_shape(w)
    return 2.0 * useful * N * K


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


def quant_bytes(rows: int, K: int, in_bytes: int = 4) -> int:
    """Bytes the activation quantiser must move: the input once, the codes and
    one fp32 scale per 128 values."""
    return rows * K * in_bytes + rows * K + rows * (K // 128) * 4


def roofline(flops: float, nbytes: float, seconds: float, hbm: float, fp8_peak: float) -> dict:
    """The slower of compute at the FP8 peak and the bytes over HBM decides
    the bound; achieved is the work of that bound over the measured time."""
    t_mem = nbytes / (hbm * 1e9)
    t_cmp = flops / (fp8_peak * 1e12)
    if t_mem >= t_cmp:
        r = {"bound": "hbm", "achieved": nbytes / seconds / 1e9, "peak": hbm, "unit": "GB/s"}
    else:
        r = {"bound": "tensor", "achieved": flops / seconds / 1e12, "peak": fp8_peak, "unit": "TFLOP/s"}
    r["frac"] = r["achieved"] / r["peak"]
    return r


# -------------------------------------------------------- ncu traffic ------
GEMM_SOURCES = ("dg_common.h", "dg_gemm.cu", "dg_gemm_pair.cu", "dg_ptx.cuh", "dg_wait.cuh")


def gemm_source_hash() -> str:
    """First 16 hex digits of the SHA-256 of the GEMM kernel's sources with
    comments and blank lines removed (what the compiler sees changes the hash;
    an edited comment does not)."""
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
def host_inputs(w: wl.Workload):
    """The workload's seeded host inputs: fp32 activations, fp32 weights and
    the MoE metadata (m_indices or masked_m; None for dense)."""
    if w.layout == "dense":
        x, wt = wl.dense_inputs(w.M, w.N, w.K, w.seed, w.outliers)
        return x, wt, None
    if w.layout == "contiguous":
        x, wt, m_indices, _ = wl.contiguous_inputs(w)
        return x, wt, m_indices
    x, wt, masked_m = wl.masked_inputs(w)
    return x, wt, masked_m


def input_fingerprints(x, wt, meta) -> dict:
    """First 16 hex digits of the SHA-256 of each generated input, for the record."""
    f = {"x": hashlib.sha256(np.ascontiguousarray(x).tobytes()).hexdigest()[:16],
         "w": hashlib.sha256(np.ascontiguousarray(wt).tobytes()).hexdigest()[:16]}
    if meta is not None:
        f["meta"] = hashlib.sha256(np.ascontiguousarray(meta).tobytes()).hexdigest()[:16]
    return f


def input_sets(w: wl.Workload, x_bytes: int, min_sets: int = 1):
    """Bytes of one step's activations, codes and output, and how many
    independent copies make the steps' inputs exceed 2x L2."""
    rows, _, N, K, _ = gemm_shape(w)
    set_bytes = x_bytes + rows * K + rows * N * 2
    return set_bytes, max(min_sets, -(-2 * L2_BYTES // set_bytes))


def l2_note(set_bytes: int, n_sets: int) -> str:
    if n_sets > 1:
        return f"rotating {n_sets} input sets of {set_bytes / 1e6:.1f} MB (> 2x L2) between launches"
    return f"inputs of {set_bytes / 1e6:.0f} MB per step (> 2x L2)"


def run_config(w: wl.Workload, x, wt, meta, world: int) -> dict:
    """The `config` object of the JSON line; both arms print the same one."""
    set_bytes, n_sets = input_sets(w, x.nbytes)
    return {"workload": describe(w), "l2": l2_note(set_bytes, n_sets), "inputs_sha256": input_fingerprints(x, wt, meta),
            "parallelism": "replicas" if world > 1 else "single GPU"}


def _contig_sample_setup(w: wl.Workload, inputs=None):
    import oracle
    x, wt, m_indices = inputs if inputs is not None else host_inputs(w)
    qb, sfb = oracle.quant_weight_128x128(wt)
    a_full = np.zeros((len(m_indices), w.K), np.uint8)
    sfa_full = np.zeros((w.K // 128, oracle.round_up(len(m_indices), 4)), np.float32)
    valid = np.flatnonzero(m_indices >= 0)
    return x, qb, sfb, m_indices, a_full, sfa_full, valid


def _oracle_rows(w: wl.Workload, state, rows: np.ndarray):
    """The oracle's quantise + GEMM over the listed rows of the workload
    (contiguous: the listed rows' activations quantised into the full-size
    operand, then the grouped GEMM restricted to those rows)."""
    import oracle
    if w.layout == "dense":
        x, qb, sfb = state
        qa, sfa = oracle.quant_act_1x128(x[rows])
        oracle.gemm_nt(qa, sfa, qb, sfb)
        return
    x, qb, sfb, m_indices, a_full, sfa_full, _ = state
    qa, sfa = oracle.quant_act_1x128(x[rows])
    a_full[rows] = qa
    sfa_full[:, rows] = sfa[:, :len(rows)]
    oracle.grouped_contiguous(a_full, sfa_full, qb, sfb, m_indices, rows=rows)


def _oracle_state(w: wl.Workload, inputs=None):
    import oracle
    if w.layout == "dense":
        x, wt, _ = inputs if inputs is not None else host_inputs(w)
        qb, sfb = oracle.quant_weight_128x128(wt)
        return (x, qb, sfb), np.arange(w.M)
    if w.layout == "contiguous":
        st = _contig_sample_setup(w, inputs)
        return st, st[-1]
    raise SystemExit("the CPU leg covers the dense and contiguous workloads")


def cpu_oracle_rate(w: wl.Workload, seconds: float):
    """Time the oracle (quantise + GEMM) over useful rows of the workload, in
    growing chunks walking through a seeded permutation of them, until about
    `seconds` have passed; returns (TFLOP/s, rows computed, elapsed s, threads)."""
    import oracle
    state, rows_all = _oracle_state(w)
    order = np.random.default_rng(99).permutation(rows_all)
    rows_done, elapsed, chunk, r0 = 0, 0.0, 8, 0
    while elapsed < seconds:
        rows = np.sort(order[r0:r0 + chunk]).astype(np.int32)
        t0 = time.perf_counter()
        _oracle_rows(w, state, rows)
        elapsed += time.perf_counter() - t0
        rows_done += len(rows)
        r0 = 0 if r0 + chunk >= len(order) else r0 + chunk
        chunk = min(chunk * 2, 64)
    flops = 2.0 * rows_done * w.N * w.K
    return flops / elapsed / 1e12, rows_done, elapsed, oracle.num_threads()


def run_reference(args, w):
    """The oracle as it stands, timed on the host cores: every step quantises
    and multiplies a bounded sample of the workload's useful rows (one row
    per oracle thread, walking through a seeded permutation), so that the
    whole run stays within a few minutes; the value is the sampled FLOPs over
    the sampled time."""
    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    inputs = host_inputs(w)
    config = run_config(w, *inputs, args.gpus)
    state, rows_all = _oracle_state(w, inputs)
    del inputs
    thr = oracle.num_threads()
    rows_per_step = min(len(rows_all), thr)
    order = np.random.default_rng(99).permutation(rows_all)
    flops = 0.0
    elapsed = 0.0
    for i in range(args.warmup + args.steps):
        r0 = (i * rows_per_step) % max(len(order) - rows_per_step + 1, 1)
        rows = np.sort(order[r0:r0 + rows_per_step]).astype(np.int32)
        t0 = time.perf_counter()
        _oracle_rows(w, state, rows)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            elapsed += dt
            flops += 2.0 * len(rows) * w.N * w.K
    value = flops / elapsed / 1e12
    rows_total = gemm_shape(w)[0]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 block sums, fp32 promotion",
        "data": "synthetic", "config": config,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle",
                         "sample": f"per step {rows_per_step} of {rows_total} rows x all {w.N} columns "
                                   f"(quantise + GEMM), {elapsed:.1f} s timed"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU leg --
class Case:
    """One workload resident on the device, in `n_sets` independent copies of
    the per-step tensors (activations, codes, scales, output) so that steps
    rotating through them exceed L2; weights are shared."""

    def __init__(self, dg, torch, w: wl.Workload, dev, min_sets: int = 1):
        self.w = w
        self.dg = dg
        self.torch = torch
        rows, useful, N, K, G = gemm_shape(w)
        self.rows, self.useful, self.N, self.K, self.G = rows, useful, N, K, G
        self.flops = useful_flops(w)
        self.bytes = algorithmic_bytes(w)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        x, wt, meta = host_inputs(w)
        self.meta = None if meta is None else t(meta)
        self.x_host = x
        self.input_sha256 = input_fingerprints(x, wt, meta)
        wdev = t(wt)
        self.qb, self.sfb = dg.dg_quant_weight_128x128(wdev)
        del wdev
        self.set_bytes, self.n_sets = input_sets(w, x.nbytes, min_sets)
        self.xs, self.qas, self.sfas, self.ds = [], [], [], []
        xdev = t(x)
        for i in range(self.n_sets):
            self.xs.append(xdev if i == 0 else xdev.clone())
            if w.layout == "masked":
                qa = torch.empty((G, w.max_m, K), dtype=torch.uint8, device=dev)
                sfa = torch.zeros((G, K // 128, dg.round_up(w.max_m, 4)), dtype=torch.float32, device=dev)
                for e in range(G):   # per-expert quantisation (set-up, untimed)
                    dg.dg_quant_act_1x128(self.xs[i][e], qa[e], sfa[e])
                d = torch.empty((G, w.max_m, N), dtype=torch.bfloat16, device=dev)
            else:
                qa = torch.empty((rows, K), dtype=torch.uint8, device=dev)
                sfa = torch.zeros((K // 128, dg.round_up(rows, 4)), dtype=torch.float32, device=dev)
                d = torch.empty((rows, N), dtype=torch.bfloat16, device=dev)
            self.qas.append(qa)
            self.sfas.append(sfa)
            self.ds.append(d)
        torch.cuda.synchronize()

    def plan(self) -> dict:
        w = self.w
        return self.dg.dg_query_plan({"dense": 0, "contiguous": 1, "masked": 2}[w.layout],
                                     w.max_m if w.layout == "masked" else self.rows, self.N, self.K, self.G,
                                     expected_m=w.max_m // 2 if w.layout == "masked" else 0)

    @property
    def has_quant(self) -> bool:
        return self.w.layout != "masked"

    def quant(self, j: int, stream=None):
        j %= self.n_sets
        self.dg.dg_quant_act_1x128(self.xs[j], self.qas[j], self.sfas[j], stream=stream)

    def gemm(self, j: int, stream=None):
        j %= self.n_sets
        dg = self.dg
        if self.w.layout == "dense":
            dg.dg_fp8_gemm_nt(self.qas[j], self.sfas[j], self.qb, self.sfb, self.ds[j], stream=stream)
        elif self.w.layout == "contiguous":
            dg.dg_fp8_grouped_contiguous(self.qas[j], self.sfas[j], self.qb, self.sfb, self.meta, self.ds[j],
                                         stream=stream)
        else:
            dg.dg_fp8_grouped_masked(self.qas[j], self.sfas[j], self.qb, self.sfb, self.meta, self.ds[j],
                                     expected_m=self.w.max_m // 2, stream=stream)

    def step(self, j: int, stream=None):
        if self.has_quant:
            self.quant(j, stream)
        self.gemm(j, stream)

    def l2_note(self) -> str:
        return l2_note(self.set_bytes, self.n_sets)


def gemm_kernel_name(plan: dict) -> str:
    return "fp8_gemm_pair_kernel" if plan["block_m"] == 256 else "fp8_gemm_kernel"


def graph_time_ms(torch, body, launches: int, reps: int) -> float:
    """Average device time of one `body(i)` call: a CUDA graph of `launches`
    calls (rotating i) is captured, replayed once untimed, then `reps` times
    between CUDA events on the replaying stream."""
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        for i in range(launches):
            body(i)
    g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(reps):
        g.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / (launches * reps)


def extra_config(torch, dg, name: str, dev, hbm: float, fp8_peak: float) -> dict:
    """GEMM (and quantiser) device time of one more workload, from CUDA-graph
    replays rotating over input sets larger than 2x L2."""
    w = wl.WORKLOADS[name]
    c = Case(dg, torch, w, dev)
    launches = max(c.n_sets, 8) if c.n_sets > 1 else 8
    for i in range(3):
        c.step(i)
    torch.cuda.synchronize()
    gemm_ms = graph_time_ms(torch, c.gemm, launches, max(1, 200 // launches))
    r = roofline(c.flops, c.bytes, gemm_ms * 1e-3, hbm, fp8_peak)
    plan = c.plan()
    out = {"workload": describe(w), "kernel": gemm_kernel_name(plan), "kernel_us": gemm_ms * 1e3,
           "tflops": c.flops / (gemm_ms * 1e-3) / 1e12, "useful_flop": c.flops, "algorithmic_bytes": c.bytes, **r,
           "traffic": measured_traffic(f"fp8_gemm_{name}.md"), "plan": plan,
           "l2": c.l2_note(), "inputs_sha256": c.input_sha256,
           "timing": f"CUDA graph of {launches} launches, replayed"}
    if w.layout == "masked":
        out["masked_m_sum"] = c.useful
    if c.has_quant:
        q_ms = graph_time_ms(torch, c.quant, launches, max(1, 200 // launches))
        qb = quant_bytes(c.rows, c.K)
        out["quant_us"] = q_ms * 1e3
        out["quant_gbs"] = qb / (q_ms * 1e-3) / 1e9
        out["quant_frac_hbm"] = out["quant_gbs"] / hbm
    del c
    torch.cuda.empty_cache()
    return out


NEXT_SHAPE = (4096, 7168, 7168)   # M, N, K of the BF16 and MX legs


def acc_kernel_name(kind: str, M: int, N: int, dev) -> str:
    """The kernel the library picks for a BF16 or MX problem: the CTA pair
    when there are at least half the SMs' worth of 256 x 256 tiles."""
    import torch
    forced = os.environ.get("DG_FORCE_ACC_PAIR", "")
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    pair = forced == "1" or (forced != "0" and -(-M // 256) * -(-N // 256) >= sms // 2)
    return f"acc_pair_kernel<{kind}>" if pair else f"acc_gemm_kernel<{kind}>"


def next_format_legs(torch, dg, dev, bf16_peak: float, fp8_peak: float, only: str = "") -> dict:
    """The two formats beside per-group-scaled FP8: a BF16 GEMM and an MX GEMM
    (E4M3 with an E8M0 scale per 32 K values) at M=4096, N=7168, K=7168,
    seeded N(0,1) inputs (MX: quantised by dg_quant_mx_1x32), timed as CUDA
    graphs of repeated launches (inputs above L2)."""
    M, N, K = NEXT_SHAPE
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    out = {}
    flops = 2.0 * M * N * K
    a32 = torch.randn((M, K), generator=g, device=dev)
    b32 = torch.randn((N, K), generator=g, device=dev)
    d = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if only in ("", "bf16"):
        a16, b16 = a32.to(torch.bfloat16), b32.to(torch.bfloat16)
        ms = graph_time_ms(torch, lambda i: dg.dg_bf16_gemm_nt(a16, b16, d), 4, 10)
        r = roofline(flops, (M * K + N * K + M * N) * 2, ms * 1e-3, 1e30, bf16_peak)
        out["bf16"] = {"workload": f"BF16 GEMM M={M} N={N} K={K}", "kernel": acc_kernel_name("bf16", M, N, dev),
                       "kernel_us": ms * 1e3, "tflops": flops / (ms * 1e-3) / 1e12, **r,
                       "peak_note": "measured bf16 burst peak"}
        del a16, b16
    if only in ("", "mx"):
        qa, sa = dg.dg_quant_mx_1x32(a32)
        qb, sb = dg.dg_quant_mx_1x32(b32)
        ms = graph_time_ms(torch, lambda i: dg.dg_mx_gemm_nt(qa, sa, qb, sb, d), 4, 10)
        r = roofline(flops, M * K + N * K + (M + N) * K // 32 + M * N * 2, ms * 1e-3, 1e30, fp8_peak)
        out["mx"] = {"workload": f"MX (E4M3, E8M0 per 32) GEMM M={M} N={N} K={K}", "kernel": acc_kernel_name("mx", M, N, dev),
                     "kernel_us": ms * 1e3, "tflops": flops / (ms * 1e-3) / 1e12, **r,
                     "peak_note": "measured bf16 burst peak x 2 (FP8)"}
        del qa, qb
    del a32, b32, d
    if only in ("", "requant"):
        out["requant"] = requant_leg(torch, dg, dev)
    torch.cuda.empty_cache()
    return out


REQUANT_SHAPE = (4096, 7168, 2048)   # M, N, K of the re-quantised-output leg


def requant_leg(torch, dg, dev) -> dict:
    """The FP8 GEMM with its output re-quantised in the epilogue (E4M3 codes +
    1x128 scales, the next GEMM's activation operand) against the two calls it
    replaces (bf16 GEMM, then the quantiser on bf16 D), dense M=4096, N=7168,
    K=2048, seeded N(0,1) inputs, CUDA graphs of repeated launches."""
    M, N, K = REQUANT_SHAPE
    g = torch.Generator(device=dev)
    g.manual_seed(12)
    qa, sa = dg.dg_quant_act_1x128(torch.randn((M, K), generator=g, device=dev))
    qb, sb = dg.dg_quant_weight_128x128(torch.randn((N, K), generator=g, device=dev))
    q = torch.empty((M, N), dtype=torch.uint8, device=dev)
    so = torch.zeros((N // 128, dg.round_up(M, 4)), dtype=torch.float32, device=dev)
    d = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    q2 = torch.empty_like(q)
    so2 = torch.zeros_like(so)
    fused = graph_time_ms(torch, lambda i: dg.dg_fp8_gemm_nt_q(qa, sa, qb, sb, q, so), 4, 10)

    def two_calls(i):
        dg.dg_fp8_gemm_nt(qa, sa, qb, sb, d)
        dg.dg_quant_act_1x128(d, q2, so2)

    pair = graph_time_ms(torch, two_calls, 4, 10)
    gemm_only = graph_time_ms(torch, lambda i: dg.dg_fp8_gemm_nt(qa, sa, qb, sb, d), 4, 10)
    flops = 2.0 * M * N * K
    out_bytes = M * N + (N // 128) * M * 4
    plan = dg.dg_query_plan(dg.DG_LAYOUT_DENSE, M, N, K, 1)
    kernel = ("fp8_gemm_pair_kernel<true>" if plan["block_m"] == 256
              else "fp8_gemm_kernel<128, 5, 64, 1, true>")
    return {"workload": f"dense FP8 GEMM M={M} N={N} K={K}, output re-quantised (E4M3 + 1x128 scales)",
            "kernel": kernel, "fused_us": fused * 1e3,
            "two_calls_us": pair * 1e3, "bf16_gemm_alone_us": gemm_only * 1e3,
            "fused_tflops": flops / (fused * 1e-3) / 1e12, "speedup_over_two_calls": pair / fused,
            "output_bytes": out_bytes}


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
    dev = torch.device("cuda", local)
    hbm, bf16, bf16_sus, src = peaks()
    fp8_peak = bf16 * FP8_PER_BF16

    c = Case(dg, torch, w, dev)
    stream = torch.cuda.current_stream()
    for i in range(args.warmup):
        c.step(i)
    torch.cuda.synchronize()

    # Timed region: `steps` steps launched directly (a step of the headline
    # workload is about a millisecond, so host launch cost is hidden), with a
    # CUDA event before the quantiser, between the two kernels and after the
    # GEMM, all on the launching stream, so that the kernel durations come
    # from the timed region itself.
    steps = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    with ClockSampler(local) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        for i in range(steps):
            ev[i][0].record(stream)
            if c.has_quant:
                c.quant(i)
            ev[i][1].record(stream)
            c.gemm(i)
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    total_ms = ev[0][0].elapsed_time(ev[steps - 1][2])
    quant_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
    gemm_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / steps
    total_ms = max_over_ranks(total_ms, device=dev)

    flops_step = c.flops
    value = job_throughput(world, flops_step, steps, total_ms) / 1e12

    roof = roofline(flops_step, c.bytes, gemm_ms * 1e-3, hbm, fp8_peak)
    prof_name = f"fp8_gemm_{w.name}.md"
    roof["traffic"] = measured_traffic(prof_name)
    roof["peak_source"] = (f"{src} (MEASURED_PEAKS.json: bf16 burst {bf16:g} TFLOP/s x {FP8_PER_BF16:g} for fp8; "
                           f"sustained {bf16_sus:g} x {FP8_PER_BF16:g} = {bf16_sus * FP8_PER_BF16:g}; "
                           f"HBM {hbm:g} GB/s)" if src == "measured" else "fallback")
    roof["kernel"] = gemm_kernel_name(c.plan())
    roof["plan"] = c.plan()
    roof["kernel_us"] = gemm_ms * 1e3
    roof["algorithmic_bytes"] = c.bytes
    roof["useful_flop"] = flops_step
    if c.has_quant:
        qbytes = quant_bytes(c.rows, c.K)
        roof["quant_us"] = quant_ms * 1e3
        roof["quant_gbs"] = qbytes / (quant_ms * 1e-3) / 1e9

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": total_ms / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic (seeded, random init)",
        "config": {"workload": describe(w), "l2": c.l2_note(), "inputs_sha256": c.input_sha256,
                   "parallelism": "replicas" if world > 1 else "single GPU"},   # = run_config()
        "roofline": roof,
        "gpu_launches": (2 if c.has_quant else 1) * steps,
        "launch": "direct launches on one stream with CUDA events around each kernel",
        "clocks": clk.summary(),
    }

    if not args.no_e2e:
        line["e2e"] = e2e(torch, dg, c, args, world, dev)

    if rank == 0 and world == 1 and not args.no_extra:
        others = {}
        for name in EXTRA:
            if name == w.name:
                continue
            others[name] = extra_config(torch, dg, name, dev, hbm, fp8_peak)
        line["configs"] = others
        line["next_formats"] = next_format_legs(torch, dg, dev, bf16, fp8_peak)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, rows, el, thr = cpu_oracle_rate(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": thr, "kind": "oracle",
                                "sample": f"oracle quantise + GEMM over {rows} useful rows of the {c.rows}-row "
                                          f"workload (seeded permutation, chunks of up to 64 rows, "
                                          f"{el:.1f} s of CPU time), rate in TFLOP/s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def e2e(torch, dg, c: Case, args, world: int, dev) -> dict:
    """End to end through the public API: every step copies its fp32
    activations (and the MoE metadata) from pinned host memory to the device,
    runs the quantiser and the GEMM, and copies D back to pinned host memory.
    Independent steps are pipelined over three streams (copy in, compute,
    copy out) with two buffer sets; a set is reused only after its previous
    copy out has completed."""
    nbuf = 2
    x_pin = torch.from_numpy(c.x_host).pin_memory()
    meta_pin = None if c.meta is None else c.meta.cpu().pin_memory()
    d_pins = [torch.empty(c.ds[0].shape, dtype=torch.bfloat16).pin_memory() for _ in range(nbuf)]
    xs = [c.xs[0]] + [torch.empty_like(c.xs[0]) for _ in range(nbuf - 1)]
    metas = None if c.meta is None else [torch.empty_like(c.meta) for _ in range(nbuf)]
    qas = [c.qas[0]] + [torch.empty_like(c.qas[0]) for _ in range(nbuf - 1)]
    sfas = [c.sfas[0]] + [torch.empty_like(c.sfas[0]) for _ in range(nbuf - 1)]
    ds = [c.ds[0]] + [torch.empty_like(c.ds[0]) for _ in range(nbuf - 1)]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]
    ev_cmp = [torch.cuda.Event() for _ in range(nbuf)]
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]
    used = [False] * nbuf
    w = c.w

    def step(i):
        j = i % nbuf
        if used[j]:
            s_in.wait_event(ev_out[j])
        used[j] = True
        with torch.cuda.stream(s_in):
            xs[j].copy_(x_pin, non_blocking=True)
            if metas is not None:
                metas[j].copy_(meta_pin, non_blocking=True)
        ev_in[j].record(s_in)
        s_cmp.wait_event(ev_in[j])
        sc = s_cmp.cuda_stream
        if w.layout == "masked":
            for e in range(c.G):
                dg.dg_quant_act_1x128(xs[j][e], qas[j][e], sfas[j][e], stream=sc)
            dg.dg_fp8_grouped_masked(qas[j], sfas[j], c.qb, c.sfb, metas[j], ds[j], expected_m=w.max_m // 2,
                                     stream=sc)
        else:
            dg.dg_quant_act_1x128(xs[j], qas[j], sfas[j], stream=sc)
            if w.layout == "dense":
                dg.dg_fp8_gemm_nt(qas[j], sfas[j], c.qb, c.sfb, ds[j], stream=sc)
            else:
                dg.dg_fp8_grouped_contiguous(qas[j], sfas[j], c.qb, c.sfb, metas[j], ds[j], stream=sc)
        ev_cmp[j].record(s_cmp)
        s_out.wait_event(ev_cmp[j])
        with torch.cuda.stream(s_out):
            d_pins[j].copy_(ds[j], non_blocking=True)
        ev_out[j].record(s_out)

    for i in range(2 * nbuf):
        step(i)
    torch.cuda.synchronize()
    n = max(args.steps, 4) if c.x_host.nbytes > 64 * 2 ** 20 else min(max(args.steps, 100), 500)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(n):
        step(i)
    e1.record(s_out)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), device=dev)
    h2d = c.x_host.nbytes + (0 if c.meta is None else c.meta.numel() * 4)
    d2h = c.ds[0].numel() * 2

    def copy_ms(dst, src, stream) -> float:
        best = float("inf")
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            with torch.cuda.stream(stream):
                dst.copy_(src, non_blocking=True)
            b.record(stream)
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b))
        return best

    # the host link alone: one copy of the step's input, one of its output
    h2d_ms = copy_ms(xs[0], x_pin, s_in)
    d2h_ms = copy_ms(d_pins[0], ds[0], s_out)
    bound = max(h2d_ms, d2h_ms)
    return {"value": job_throughput(world, c.flops, n, ms) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": n, "ms_per_step": ms / n,
            "link": {"h2d_gbs": c.x_host.nbytes / (h2d_ms * 1e-3) / 1e9, "d2h_gbs": d2h / (d2h_ms * 1e-3) / 1e9,
                     "copy_bound_ms_per_step": bound, "frac_of_copy_bound": bound / (ms / n)},
            "how": "pinned host fp32 activations in, bf16 D out, every step, three streams"}


def profile_next(args):
    import torch

    import moe_grouped_gemm_x128_gb300 as dg
    torch.cuda.set_device(0)
    dg.build()
    dg.load()
    hbm, bf16, _, _ = peaks()
    print(json.dumps(next_format_legs(torch, dg, torch.device("cuda", 0), bf16, bf16 * FP8_PER_BF16,
                                      only=args.profile_next)), flush=True)


def main(argv=None):
    args = parse(argv)
    if args.profile_next:
        profile_next(args)
        return
    w = with_tokens(wl.WORKLOADS[args.workload], args.tokens)
    if args.shape:
        M, N, K = (int(v) for v in args.shape.split(","))
        w = wl.Workload(f"shape_{M}x{N}x{K}", "dense", M=M, N=N, K=K, seed=5)
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_gpu(args, w)


if __name__ == "__main__":
    main()
