"""Benchmark of the FP8 rowwise-scaled grouped GEMM on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gemm|reference]
                    [--workload NAME] [--variant NAME] [--no-sweep] [--no-cpu]

One step = one call of the whole hot path (host checks and planning, the device group
scheduler, the TMA/tcgen05 pipeline and the fused epilogue) on one batch of seeded
synthetic input resident in HBM.  Prints ONE JSON line (rank 0).

Headline workload: the largest single-GPU configuration, llama3-405b-shaped stacked
G=16, N=K=total_M=16384 (inputs 5.1 GB, larger than L2, so no flush is needed).  The
metric is FP8 grouped GEMM TFLOPS (2 * sum_g m_g * N * K per call); the line also carries
us/call, the roofline of the kernel, the end-to-end figure through host buffers (with the
host link's measured copy bandwidth), the CPU oracle baseline, the SM clocks seen, and,
last on the line, one compact row per shape of the sweep (DS-V3 gate_up/down, llama3-70b
total_M in {1, 16, 128, 1024, 8192}, the other layouts) timed by CUDA-graph replay with
rotating input sets sized past twice the L2.

Roofline fractions use the measured peaks: the copy bandwidth, and the FP8 peak = 2 x the
measured bf16 GEMM rate, burst or sustained according to the SM clock seen during each
timed window (burst unless the median clock under load was at or below the clock of the
sustained measurement).  The fraction against the nominal dense FP8 peak (4.5 PFLOP/s) and
HBM bandwidth (8 TB/s) is reported beside it.

--impl reference times the CPU oracle (the plain fp64 C reference) on the same workload,
one bounded row sample per step, on the host cores.

Multi-GPU (torchrun, one rank per GPU): every rank runs the same workload on its own GPU
(independent replicas, no collective on the data path); the time is the max over ranks
and the value is the work of all ranks divided by it ("weak" scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP8 grouped GEMM TFLOPS, µs/call, % of roofline (FP8 peak or HBM) per shape"
UNIT = "TFLOPS"
HEADLINE = "c4_llama405b"
SWEEP = ["c2a_dsv3_gate_up", "c2b_dsv3_down", "c3_llama70b_m1", "c3_llama70b_m16",
         "c3_llama70b_m128", "c3_llama70b_m1024", "c3_llama70b_m8192",
         "n1_batched_llama70b_m512", "n2_offsets_llama70b_m8192", "n3_ragged_n_m1024",
         "n4_ragged_k_wgrad", "n5_groupwise_llama70b_m8192", "n6_groupwise_llama70b_m16",
         "n7_groupwise_batched_llama70b_m512", "n8_groupwise_dynamic_dsv3_m256"]
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0  # nominal dense ratio (4.5 / 2.25 PFLOP/s)
FP8_NOMINAL_TFLOPS = 4500.0  # GB300 dense FP8, nominal
HBM_NOMINAL_GBS = 8000.0     # GB300 HBM3e, nominal
# columns of the compact per-shape rows
PER_SHAPE_COLS = ["workload", "us_per_call", "tflops", "bound", "frac", "frac_nominal",
                  "sm_mhz", "variant"]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# string and character literals (kept), // and /* */ comments (dropped)
_CODE_TOKENS = re.compile(r'"(?:\\.|[^"\\])*"|\'(?:\\.|[^\'\\])*\'|//[^\n]*|/\*.*?\*/', re.S)


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code: comments and whitespace do not count, so a
    committed traffic capture stays valid across documentation edits."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp8_rowwise_scaled_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            text = f.read()
        code = _CODE_TOKENS.sub(lambda m: m.group(0) if m.group(0)[0] in "\"'" else " ", text)
        h.update(name.encode() + " ".join(code.split()).encode())
    return h.hexdigest()[:16]


def dram_traffic(workload: str):
    """Per-launch DRAM bytes from a committed ncu capture, if it was taken on the current
    kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks, power and throttle reasons, every sample stamped
    with the host clock, so that each timed window (the headline's timed steps, every
    sweep shape's replays) gets the clocks seen inside it."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    PERIOD_MS = 25

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None
        self.rows = None

    def __enter__(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()

    def _load(self):
        if self.rows is not None:
            return self.rows
        self.rows = []
        try:
            with open(self.file.name) as f:
                lines = [ln.strip() for ln in f if ln.strip()]
            os.unlink(self.file.name)
        except OSError:
            return self.rows
        for ln in lines:
            self.rows.extend(parse_smi_rows([ln]))
        return self.rows

    def window(self, t0: float | None = None, t1: float | None = None):
        """Clocks of the samples taken in [t0, t1] (host time.time()); the nearest sample
        when none falls inside a window shorter than the sampling period."""
        rows = self._load()
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        sel = rows
        if t0 is not None and t1 is not None:
            sel = [r for r in rows if t0 <= r["t"] <= t1]
            if not sel:
                mid = 0.5 * (t0 + t1)
                sel = [min(rows, key=lambda r: abs(r["t"] - mid))]
        return summarize_clocks(sel)


def parse_smi_rows(lines):
    """Rows of `nvidia-smi --query-gpu=<ClockSampler.Q> --format=csv,noheader,nounits`."""
    import datetime
    out = []
    for ln in lines:
        r = [x.strip() for x in ln.split(",")]
        if len(r) < 10:
            continue
        try:
            t = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            sm, mx, pw = float(r[2]), float(r[3]), float(r[4])
        except ValueError:
            continue
        active = {n for n, v in zip(ClockSampler.REASONS, r[6:10]) if v.lower() == "active"}
        out.append({"t": t, "sm": sm, "max": mx, "power": pw, "reasons": active})
    return out


def summarize_clocks(rows):
    """Median SM clock under load (samples above 30 % of the highest power seen), the
    maximum clock, and every throttle reason that was active."""
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
    pmax = max(r["power"] for r in rows)
    loaded = [r for r in rows if r["power"] > 0.3 * pmax] or rows
    reasons = set()
    for r in rows:
        reasons |= r["reasons"]
    return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
            "sm_max_mhz": max(r["max"] for r in rows), "reasons": sorted(reasons),
            "samples": len(rows), "power_w_max": pmax}


# ---------------------------------------------------------------------------------------
# distributed plumbing (replicas; the barrier and max-over-ranks timing only)
# ---------------------------------------------------------------------------------------
def dist_setup(backend):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group(backend)
    return rank, local, ws


def dist_max(value: float, ws: int, device):
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline field)
# ---------------------------------------------------------------------------------------
def oracle_sample_inputs(wl, rows: int, seed: int):
    """A bounded sample of the workload on the host: `rows` activation rows against one
    group's full [N, K] weights (the work of `rows` output rows of the workload)."""
    import numpy as np
    import torch
    from fp8_rowwise_scaled_gb300.synthetic import quantize_rows
    g = torch.Generator().manual_seed(seed)
    A, sa = quantize_rows(torch.randn((rows, wl.K), generator=g))
    B = torch.empty((1, wl.N, wl.K), dtype=torch.uint8)
    sb = torch.empty((1, wl.N), dtype=torch.float32)
    step = 4096
    for n0 in range(0, wl.N, step):
        q, s = quantize_rows(torch.randn((min(step, wl.N - n0), wl.K), generator=g))
        B[0, n0:n0 + q.shape[0]] = q
        sb[0, n0:n0 + q.shape[0]] = s
    return (A.numpy(), B.numpy(), sa.numpy(), sb.numpy(), np.array([rows], np.int64))


def time_oracle(wl, rows: int, reps: int = 1, warm: int = 0, seed: int = 7):
    import oracle
    orc = oracle.load(0)
    A, B, sa, sb, meta = oracle_sample_inputs(wl, rows, seed)
    threads = len(os.sched_getaffinity(0))
    for _ in range(warm):
        orc.stacked(A, B, sa, sb, meta, threads=threads)
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        orc.stacked(A, B, sa, sb, meta, threads=threads)
        times.append(time.perf_counter() - t0)
    flops = 2.0 * rows * wl.N * wl.K
    return flops, times, threads


# ---------------------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------------------
def run_call(fx, inp, out, wl, stream_ptr):
    if wl.layout == "stacked":
        s = fx.mslkb_f8f8bf16_rowwise_grouped_stacked(
            inp["A"].data_ptr(), inp["B"].data_ptr(), inp["scale_a"].data_ptr(),
            inp["scale_b"].data_ptr(), inp["meta"].data_ptr(), out.data_ptr(), wl.rows, wl.G,
            wl.N, wl.K, stream_ptr)
    elif wl.layout == "offsets":
        s = fx.mslkb_f8f8bf16_rowwise_grouped_offsets(
            inp["A"].data_ptr(), inp["B"].data_ptr(), inp["scale_a"].data_ptr(),
            inp["scale_b"].data_ptr(), inp["meta"].data_ptr(), out.data_ptr(), wl.rows, wl.G,
            wl.N, wl.K, stream_ptr)
    elif wl.layout == "groupwise":
        s = fx.mslkb_f8f8bf16_groupwise_grouped_stacked(
            inp["A"].data_ptr(), inp["B"].data_ptr(), inp["scale_a"].data_ptr(),
            inp["scale_b"].data_ptr(), inp["meta"].data_ptr(), out.data_ptr(), wl.rows, wl.G,
            wl.N, wl.K, stream_ptr)
    elif wl.layout == "groupwise_dynamic":
        s = fx.mslkb_f8f8bf16_groupwise_grouped_dynamic(
            inp["A"].data_ptr(), inp["B"].data_ptr(), inp["scale_a"].data_ptr(),
            inp["scale_b"].data_ptr(), inp["meta"].data_ptr(), out.data_ptr(), wl.G,
            wl.expected_m, wl.N, wl.K, stream_ptr)
    elif wl.layout == "groupwise_batched":
        s = fx.mslkb_f8f8bf16_groupwise_grouped_batched(
            inp["A"].data_ptr(), inp["B"].data_ptr(), inp["scale_a"].data_ptr(),
            inp["scale_b"].data_ptr(), out.data_ptr(), wl.G, wl.expected_m, wl.N, wl.K,
            stream_ptr)
    elif wl.layout == "ragged_n":
        s = fx.mslkb_f8f8bf16_rowwise_grouped_n_offsets(
            inp["A"].data_ptr(), inp["B"].data_ptr(), inp["scale_a"].data_ptr(),
            inp["scale_b"].data_ptr(), inp["meta"].data_ptr(), out.data_ptr(), wl.G, wl.rows,
            wl.N, wl.K, stream_ptr)
    elif wl.layout == "ragged_k":
        s = fx.mslkb_f8f8bf16_rowwise_grouped_k_offsets(
            inp["A"].data_ptr(), inp["B"].data_ptr(), inp["scale_a"].data_ptr(),
            inp["scale_b"].data_ptr(), inp["meta"].data_ptr(), out.data_ptr(), wl.G, wl.rows,
            wl.N, wl.K, stream_ptr)
    elif wl.layout == "batched":
        s = fx.mslkb_f8f8bf16_rowwise_grouped_batched(
            inp["A"].data_ptr(), inp["B"].data_ptr(), inp["scale_a"].data_ptr(),
            inp["scale_b"].data_ptr(), out.data_ptr(), wl.G, wl.expected_m, wl.N, wl.K,
            stream_ptr)
    else:
        s = fx.mslkb_f8f8bf16_rowwise_grouped_dynamic(
            inp["A"].data_ptr(), inp["B"].data_ptr(), inp["scale_a"].data_ptr(),
            inp["scale_b"].data_ptr(), inp["meta"].data_ptr(), out.data_ptr(), wl.G,
            wl.expected_m, wl.N, wl.K, stream_ptr)
    if s != 0:
        raise fx.MslkbError(s, wl.name)


def fp8_peaks(pk):
    """(burst, sustained) FP8 dense peaks in TFLOP/s -- the measured bf16 GEMM rates times
    the nominal fp8/bf16 dense ratio -- and the SM clock (MHz) the sustained figure was
    measured at (None if not recorded)."""
    burst = pk["bf16_tflops"] * FP8_OVER_BF16
    sust = pk.get("bf16_tflops_sustained", pk["bf16_tflops"]) * FP8_OVER_BF16
    f_sust = (pk.get("clocks_under_load") or {}).get("sm_mhz_median")
    return burst, sust, f_sust


def fp8_peak_for_clock(pk, sm_mhz):
    """The FP8 peak that matches the clocks of a timed window: the burst figure, unless the
    window's median SM clock under load was at or below the clock at which the sustained
    (seconds-long, power-capped) figure was measured.  Returns (TFLOP/s, reason)."""
    burst, sust, f_sust = fp8_peaks(pk)
    if sm_mhz is None or f_sust is None:
        return burst, "burst (no clock record to match)"
    if sm_mhz > f_sust:
        return burst, (f"burst: median SM clock {sm_mhz:.0f} MHz above the {f_sust:.0f} MHz "
                       f"of the sustained measurement")
    return sust, (f"sustained: median SM clock {sm_mhz:.0f} MHz at or below the "
                  f"{f_sust:.0f} MHz of the sustained measurement")


def roofline(wl, pk, t_call, sm_mhz):
    """Roofline figures of one call that took t_call seconds in a window whose median SM
    clock was sm_mhz: t_roof = max(F / P_fp8, bytes / BW) with P_fp8 matched to the clock
    and BW the measured copy bandwidth; also the fractions against the burst and the
    sustained peaks, against the sustained figure scaled to the window's clock
    (flops per SM cycle), and against the nominal dense FP8 peak and HBM bandwidth."""
    p_fp8, why = fp8_peak_for_clock(pk, sm_mhz)
    burst, sust, f_sust = fp8_peaks(pk)
    t_fp8 = wl.flops() / (p_fp8 * 1e12)
    t_hbm = wl.bytes() / (pk["hbm_gbs"] * 1e9)
    t_nom = max(wl.flops() / (FP8_NOMINAL_TFLOPS * 1e12), wl.bytes() / (HBM_NOMINAL_GBS * 1e9))
    r = {"bound": "tensor" if t_fp8 >= t_hbm else "hbm",
         "frac": max(t_fp8, t_hbm) / t_call, "p_fp8": p_fp8, "peak_choice": why,
         "frac_of_burst": wl.flops() / (burst * 1e12) / t_call,
         "frac_of_sustained": wl.flops() / (sust * 1e12) / t_call,
         "frac_of_hbm": t_hbm / t_call, "frac_nominal": t_nom / t_call}
    if sm_mhz and f_sust:
        r["frac_at_clock"] = wl.flops() / (sust * 1e12 * sm_mhz / f_sust) / t_call
    return r


def workload_config(wl, ws):
    """The workload-defining part of the `config` object, the same in both arms."""
    return {"workload": wl.name, "layout": wl.layout, "G": wl.G, "N": wl.N, "K": wl.K,
            "total_M": wl.rows, "m_sizes": list(wl.meta), "seed": wl.seed,
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
            "l2": f"inputs larger than L2 ({wl.bytes() / 1e9:.2f} GB per call), no flush"}


def plan_for(fx, wl, sms):
    if wl.layout in ("ragged_n", "ragged_k"):
        return fx.mslkb_plan(2 if wl.layout == "ragged_n" else 3, wl.rows, wl.G, wl.N, wl.K, sms)
    if wl.layout == "groupwise":
        return fx.mslkb_plan(4, wl.rows, wl.G, wl.N, wl.K, sms)
    if wl.block_scaled:
        return fx.mslkb_plan(5, wl.expected_m, wl.G, wl.N, wl.K, sms)
    return fx.mslkb_plan(1 if wl.slabs else 0, wl.expected_m if wl.slabs else wl.rows, wl.G,
                         wl.N, wl.K, sms)


def out_shape(wl):
    """Rows and columns of the output (ragged K: a slab of M rows per group)."""
    return (wl.G * wl.rows if wl.layout == "ragged_k" else wl.rows, wl.N)


def sweep_shape(fx, wl, pk, device):
    """us/call of one shape by CUDA-graph replay (median of 7 timed replays of ~25 ms),
    rotating input sets so that the data touched by one replay cycle exceeds twice the L2.
    Returns the time and the host-clock window of the timed replays (for their clocks)."""
    import torch
    from fp8_rowwise_scaled_gb300.synthetic import make_inputs
    ws_bytes = max(1, wl.bytes())
    n_sets = max(1, min(16, math.ceil(2 * L2_BYTES / ws_bytes)))
    base = make_inputs(wl, device)
    sets = [base] + [{k: v.clone() for k, v in base.items()} for _ in range(n_sets - 1)]
    outs = [torch.empty(out_shape(wl), dtype=torch.bfloat16, device=device) for _ in sets]
    stream = torch.cuda.Stream(device=device)
    sp = stream.cuda_stream
    # the inputs were written by kernels on the current stream; the calls run on `stream`
    stream.wait_stream(torch.cuda.current_stream(device))
    fx.device_status(sp)  # start clean: the word is read and cleared
    with torch.cuda.stream(stream):
        t_end = time.perf_counter() + 0.5  # clock ramp
        while time.perf_counter() < t_end:
            for i in range(n_sets):
                run_call(fx, sets[i], outs[i], wl, sp)
            stream.synchronize()
    # calls per replay: ~25 ms of work and at least 16 calls, a multiple of the set count
    t_fp8 = wl.flops() / (fp8_peaks(pk)[0] * 1e12)
    t_est = max(t_fp8, wl.bytes() / (pk["hbm_gbs"] * 1e9)) * 1.5 + 3e-6
    reps = max(16 // n_sets + 1, min(1600, int(2.5e-2 / t_est) // n_sets)) * n_sets
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for r in range(reps):
            i = r % n_sets
            run_call(fx, sets[i], outs[i], wl, sp)
    times = []
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        graph.replay()  # untimed
        stream.synchronize()
        t0 = time.time()
        for _ in range(7):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3 / reps)  # us per call
        t1 = time.time()
    us = statistics.median(times)
    status = fx.device_status(sp)
    plan = plan_for(fx, wl, torch.cuda.get_device_properties(device).multi_processor_count)
    del graph, sets, outs, base
    torch.cuda.empty_cache()
    return {"wl": wl, "us": us, "window": (t0, t1), "variant": fx.variant_name(plan.variant),
            "status": status}


def compact_row(name, us, tflops, bound, frac, frac_nominal, sm_mhz, variant):
    """One PER_SHAPE_COLS row, short enough that all rows fit the last 1500 characters of
    the output line: whole TFLOPS and MHz, 0.1 us, and the variant name without its
    "stacked_" prefix and "_tma" suffix (the layout is the workload's; TMA unless "cpasync")."""
    if variant.startswith("stacked_"):
        variant = variant[len("stacked_"):]
    if variant.endswith("_tma"):
        variant = variant[:-len("_tma")]
    return [name, round(us, 1), int(round(tflops)), bound, round(frac, 3),
            round(frac_nominal, 3), None if sm_mhz is None else int(round(sm_mhz)), variant]


def shape_row(res, pk, clk):
    """Compact per-shape row (PER_SHAPE_COLS) with the clocks of the shape's own window."""
    if "error" in res:
        return [res["workload"], None, None, None, None, None, None, res["error"][:80]]
    wl, us = res["wl"], res["us"]
    sm = clk.window(*res["window"])["sm_mhz"]
    r = roofline(wl, pk, us * 1e-6, sm)
    return compact_row(wl.name, us, wl.flops() / (us * 1e-6) / 1e12, r["bound"], r["frac"],
                       r["frac_nominal"], sm, res["variant"])


def link_bandwidth(device, nbytes=1 << 30, reps=3):
    """Pinned host <-> device copy bandwidth in GB/s: host to device, device to host, and
    both directions at once (best of `reps`, CUDA events on the copying streams)."""
    import torch
    host = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    host2 = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    dev = torch.empty(nbytes, dtype=torch.uint8, device=device)
    dev2 = torch.empty(nbytes, dtype=torch.uint8, device=device)
    s1 = torch.cuda.Stream(device=device)
    s2 = torch.cuda.Stream(device=device)

    def best(fn):
        ts = []
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            ts.append(time.perf_counter() - t0)
        return min(ts)

    def h2d():
        with torch.cuda.stream(s1):
            dev.copy_(host, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            host2.copy_(dev2, non_blocking=True)

    def both():
        h2d()
        d2h()

    r = {"h2d_gbs": round(nbytes / best(h2d) / 1e9, 1),
         "d2h_gbs": round(nbytes / best(d2h) / 1e9, 1),
         "both_gbs": round(2 * nbytes / best(both) / 1e9, 1)}
    del host, host2, dev, dev2
    return r


def gpu_arm(args):
    import torch
    rank, local, ws = dist_setup("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import fp8_rowwise_scaled_gb300 as fx
    from fp8_rowwise_scaled_gb300 import build as fxbuild
    from fp8_rowwise_scaled_gb300.synthetic import make_inputs, workloads
    fxbuild.build()
    fx.lib()
    if args.chunk is not None:
        fx.mslkb_set_accumulation_chunk(args.chunk)
    if args.variant is not None:
        fx.mslkb_force_variant(fx.variant_index(args.variant))
    pk, pk_kind = peaks()
    wl = workloads()[args.workload]
    inp = make_inputs(wl, device)
    out = torch.empty(out_shape(wl), dtype=torch.bfloat16, device=device)
    stream = torch.cuda.Stream(device=device)
    sp = stream.cuda_stream
    stream.wait_stream(torch.cuda.current_stream(device))  # inputs written on the current stream
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    plan = plan_for(fx, wl, sms)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    # one clock sampler over the whole arm; each timed window reads its own samples
    clk = ClockSampler(local).__enter__()
    try:
        with torch.cuda.stream(stream):
            # clock ramp (0.5 s), then the untimed warm-up steps
            t_end = time.perf_counter() + 0.5
            while time.perf_counter() < t_end:
                run_call(fx, inp, out, wl, sp)
                stream.synchronize()
            e0.record(stream)
            for _ in range(args.warmup):
                run_call(fx, inp, out, wl, sp)
            e1.record(stream)
            e1.synchronize()
            t_call = e0.elapsed_time(e1) / 1e3 / max(1, args.warmup)
            steps = (args.steps if args.steps is not None
                     else max(20, math.ceil(1.5 / max(t_call, 1e-6))))
            stream.synchronize()
            dist_barrier(ws)
            torch.cuda.synchronize()
            w0 = time.time()
            e0.record(stream)
            for _ in range(steps):
                run_call(fx, inp, out, wl, sp)
            e1.record(stream)
            e1.synchronize()
            w1 = time.time()
            torch.cuda.synchronize()
            dist_barrier(ws)
        t_total = e0.elapsed_time(e1) / 1e3
        t_max = dist_max(t_total, ws, device)
        ms_per_step = t_max / steps * 1e3
        value = ws * wl.flops() * steps / t_max / 1e12
        status = fx.device_status(stream)
        e2e = e2e_leg(fx, wl, inp, out, stream, sp, steps, ws, device)
        link = link_bandwidth(device)
        t_link = max(e2e["h2d_bytes_per_step"] / (link["h2d_gbs"] * 1e9),
                     e2e["d2h_bytes_per_step"] / (link["d2h_gbs"] * 1e9),
                     (e2e["h2d_bytes_per_step"] + e2e["d2h_bytes_per_step"])
                     / (link["both_gbs"] * 1e9))
        e2e["host_link"] = link
        e2e["frac_of_link"] = round(t_link / (e2e["ms_per_step"] * 1e-3), 4)
        if args.variant is not None:
            fx.mslkb_force_variant(-1)  # the sweep runs the planner's choices
        sweep = []
        if args.sweep and rank == 0:
            for name in SWEEP:
                try:
                    sweep.append(sweep_shape(fx, workloads()[name], pk, device))
                except Exception as e:  # noqa: BLE001 - report and continue
                    sweep.append({"workload": name, "error": repr(e)})
    finally:
        clk.__exit__(None, None, None)
    clocks = clk.window(w0, w1)

    # roofline of the one kernel launched per step (per-launch time = per-step time),
    # against the peak that matches the timed region's clocks
    t_launch = t_total / steps
    rf = roofline(wl, pk, t_launch, clocks["sm_mhz"])
    burst, sust, f_sust = fp8_peaks(pk)
    if rf["bound"] == "tensor":
        roof = {"bound": "tensor", "achieved": round(wl.flops() / t_launch / 1e12, 2),
                "peak": round(rf["p_fp8"], 1), "unit": "TFLOP/s",
                "peak_source": f"{pk_kind}: bf16 GEMM {pk['bf16_tflops']} TFLOP/s burst / "
                               f"{pk.get('bf16_tflops_sustained')} sustained (at "
                               f"{f_sust} MHz) x {FP8_OVER_BF16:g}, the nominal fp8/bf16 "
                               f"dense ratio"}
    else:
        roof = {"bound": "hbm", "achieved": round(wl.bytes() / t_launch / 1e9, 1),
                "peak": pk["hbm_gbs"], "unit": "GB/s",
                "peak_source": f"{pk_kind} copy bandwidth"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["traffic"] = dram_traffic(wl.name)
    roof["peak_choice"] = rf["peak_choice"]
    roof["sm_mhz"] = clocks["sm_mhz"]
    for k in ("frac_of_burst", "frac_of_sustained", "frac_at_clock", "frac_nominal"):
        if k in rf:
            roof[k] = round(rf[k], 4)
    roof["algorithmic"] = {"flops": wl.flops(), "bytes": wl.bytes()}
    roof["kernel"] = fx.variant_name(plan.variant)

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 x e4m3 -> fp32 accumulate -> bf16", "data": "synthetic",
        "config": {**workload_config(wl, ws),
                   "us_per_call": round(ms_per_step * 1e3, 2),
                   "variant": fx.variant_name(plan.variant), "grid": plan.grid,
                   "accumulation_chunk_kblocks": fx.mslkb_accumulation_chunk()},
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": steps,
        "clocks": clocks,
        "device_status": status,
    }
    if args.cpu and rank == 0 and ws == 1:
        rows = args.cpu_rows
        flops, times, threads = time_oracle(wl, rows)
        result["cpu_baseline"] = {
            "value": round(flops / times[0] / 1e12, 6), "unit": UNIT, "cores": threads,
            "kind": "oracle", "seconds": round(times[0], 2),
            "sample": f"{rows} output rows x N={wl.N} x K={wl.K} of {wl.name} (one group's "
                      f"weights), plain fp64 C oracle, OpenMP over rows"}
    if sweep:
        # compact rows, last on the line: each shape's roofline fraction against the peak
        # that matches the clocks of its own timed replays
        rows = [shape_row(r, pk, clk) for r in sweep]
        rows.append(compact_row(wl.name, ms_per_step * 1e3, value / ws, rf["bound"], rf["frac"],
                                rf["frac_nominal"], clocks["sm_mhz"],
                                fx.variant_name(plan.variant)))
        # the device status word after each shape's calls: 0 everywhere, else the
        # shapes whose calls set a bit (MSLKB_DEV_*)
        flagged = {r["wl"].name: r["status"] for r in sweep if r.get("status")}
        result["sweep_device_status"] = flagged or 0
        result["per_shape_cols"] = PER_SHAPE_COLS
        result["per_shape"] = rows
    if rank == 0:
        print(json.dumps(result, separators=(",", ":")), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def e2e_leg(fx, wl, inp, out, stream, sp, steps, ws, device):
    """End to end through the C ABI with host buffers: every step copies its inputs in from
    pinned host memory, makes the call, and copies its result out.  Two device buffer sets
    let step j + 1's inputs cross the host link while step j computes and its result comes
    back (host-to-device copies, calls and device-to-host copies on three streams, ordered
    by events so that no buffer is overwritten before the step that reads it is done)."""
    import torch
    host = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in inp.items()}
    for k in inp:
        host[k].copy_(inp[k])
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    dev = [{k: torch.empty_like(v) for k, v in inp.items()} for _ in range(2)]
    outs = [out, torch.empty_like(out)]
    s_in = torch.cuda.Stream(device=device)
    s_out = torch.cuda.Stream(device=device)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_k = [torch.cuda.Event() for _ in range(2)]
    ev_o = [torch.cuda.Event() for _ in range(2)]
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2e_steps = max(3, min(steps, 10))
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = host_out.numel() * host_out.element_size()

    def run(n):
        for j in range(n):
            b = j % 2
            if j >= 2:
                s_in.wait_event(ev_k[b])    # the call of step j - 2 has read dev[b]
            with torch.cuda.stream(s_in):
                for k in dev[b]:
                    dev[b][k].copy_(host[k], non_blocking=True)
            ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if j >= 2:
                stream.wait_event(ev_o[b])  # step j - 2's result has left outs[b]
            with torch.cuda.stream(stream):
                run_call(fx, dev[b], outs[b], wl, sp)
            ev_k[b].record(stream)
            s_out.wait_event(ev_k[b])
            with torch.cuda.stream(s_out):
                host_out.copy_(outs[b], non_blocking=True)
            ev_o[b].record(s_out)

    run(2)  # untimed round
    torch.cuda.synchronize()
    dist_barrier(ws)
    e0.record(s_in)
    run(e2e_steps)
    e1.record(s_out)  # after the last result's copy, which follows every earlier step
    e1.synchronize()
    torch.cuda.synchronize()
    dist_barrier(ws)
    t_e2e = dist_max(e0.elapsed_time(e1) / 1e3, ws, device)
    del host, dev, outs, host_out
    torch.cuda.empty_cache()
    return {"value": round(ws * wl.flops() * e2e_steps / t_e2e / 1e12, 3), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(t_e2e / e2e_steps * 1e3, 3), "steps": e2e_steps}


def reference_arm(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from fp8_rowwise_scaled_gb300.synthetic import workloads
    wl = workloads()[args.workload]
    import oracle
    oracle.build()
    steps = args.steps if args.steps is not None else 5
    cores = len(os.sched_getaffinity(0))
    # size each step's row sample so the whole run stays near two minutes: probe one
    # row per core, then scale (at least one row per core, at most --cpu-rows)
    _, probe, _ = time_oracle(wl, cores)
    budget = 120.0 / (steps + args.warmup)
    rows = cores * max(1, int(budget / max(probe[0], 1e-3)))
    rows = max(1, min(rows, args.cpu_rows))
    flops, times, threads = time_oracle(wl, rows, reps=steps, warm=args.warmup)
    total = sum(times)
    value = flops * steps / total / 1e12
    result = {
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": ws, "steps": steps,
        "warmup": args.warmup, "ms_per_step": round(total / steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 (exact e4m3 products, correctly rounded bf16)", "data": "synthetic",
        "impl": "reference",
        "config": workload_config(wl, ws),
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": threads,
                         "kind": "oracle",
                         "sample": f"per step {rows} output rows x N={wl.N} x K={wl.K} of "
                                   f"{wl.name} (one group's weights)"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(result), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: enough for >= 1.5 s of kernel time)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gemm", "reference"], default="gemm")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--chunk", type=int, default=None,
                    help="tensor-core accumulation chunk in K blocks (default: library's)")
    ap.add_argument("--variant", default=None,
                    help="run the headline workload on this kernel variant instead of the "
                         "planner's choice (for profiling; the per-shape sweep keeps the planner's)")
    ap.add_argument("--no-sweep", dest="sweep", action="store_false")
    ap.add_argument("--no-cpu", dest="cpu", action="store_false")
    ap.add_argument("--cpu-rows", type=int, default=256,
                    help="output rows of the CPU oracle sample")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
