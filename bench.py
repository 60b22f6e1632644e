#!/usr/bin/env python3
"""Throughput of the W4A16 linear layer on GB300: one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl cuda|reference] [--config NAME]

A step is one pass of the hot path over one batch of a workload: one w4a16_gemm call (validation,
runtime dispatch, weight streaming, dequantisation, multiply-accumulate, split-K reduction and the
bias/cast epilogue) for every (M, K, N) case of the workload. Weight packing is a model-load step and
is not part of a step.

Headline workload "decode" (M <= 8): the cases of decode_2112 (the non-128-aligned layers of the
PR #43731 report's motivation: M in {1, 2, 4, 5, 8} x (K, N) in {(1152, 4224), (2112, 1152)}, G = 32,
bf16, symmetric uint4b8) followed by those of decode_4b (the 4B-class layers of the PR #40977 report's
motivation: M in {1, 4, 8} x (K, N) in {(2560, 3840), (2560, 19456), (9728, 2560)}, G = 128, fp16,
asymmetric zero points, bias). Metric: GB/s over the algorithmic bytes
K*N/2 + 2(K/G)N [+ (K/G)N/2] + 2MK + 2MN [+ 2N] per call, and its fraction of the measured HBM copy
bandwidth. The same line carries a "workloads" object with every measurement workload timed the same
way: decode_2112, decode_4b, mid_m (M 17-64), prefill (TFLOP/s, 2MNK per call, against the measured
dense bf16 rate) and a sample of the full M sweep (every M on one 27B-class layer), each with both
roofline fractions and a per-case table.

Timing: W eager warm-up steps through the C ABI, then exactly K steps replayed from CUDA graphs (the
library's calls are capture-safe), bracketed by CUDA events on the launching stream, with a barrier
and a device synchronise on both sides; every call reads its own replica of the weights, and each
replica pool is larger than twice the L2 cache, so weights stream from HBM. Under torchrun each rank
runs the same workload on its own GPU (replicas, weak scaling) and the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import re
import statistics
import subprocess
import sys
import tempfile
import time

HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)

# The CPU baseline uses every host core; fix the BLAS thread count before numpy loads.
_CPU_THREADS = os.cpu_count() or 1
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CPU_THREADS))

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "decode GB/s (frac of HBM peak) at M=1–8; prefill TFLOP/s at M≥1024"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# a timed region shorter than this is compared with the burst tensor rate, a longer one with the
# sustained rate (the measured copy bandwidth has one figure)
SUSTAINED_AFTER_S = 1.0

WORKLOADS = {
    "decode": "decode M<=8: decode_2112 cases then decode_4b cases (19 calls per step)",
    "decode_pp": "the decode workload with the weights in the library's prepacked layout (w4a16_prepack)",
    "decode_2112": "decode, non-Marlin-aligned: M in {1,2,4,5,8} x (K,N) in {(1152,4224),(2112,1152)}, "
                   "G=32, bf16, symmetric uint4b8, scales U[0.005,0.02], A~N(0,1)",
    "decode_4b": "decode 4B-class: M in {1,4,8} x (K,N) in {(2560,3840),(2560,19456),(9728,2560)}, G=128, "
                 "fp16, asymmetric qzeros, fp16 bias N(0,0.1)",
    "prefill": "prefill: M in {512,1024,4096} x (K,N) in {(5120,34816),(17408,5120)}, G=64, bf16, "
               "asymmetric qzeros, scales U[0.002,0.01]",
    "mid_m": "mid M: M in {17,24,32,64} x (K,N) in {(5120,7168),(17408,5120)}, G=128, bf16, symmetric "
             "uint4b8, scales U[0.005,0.02], A~N(0,1)",
    "sweep": "full M sweep, sampled: every M of 1..8192 (powers of 2, 5, 6, 24) on (K,N)=(5120,7168), cycling "
             "fp16/bf16, G in {128, K} and symmetric/asymmetric across the M values",
    "tiny": "tiny: M=4, K=256, N=512, G=128, fp16, symmetric",
}
# the workloads the default run reports beside the headline
SIDE_WORKLOADS = ["decode_2112", "decode_4b", "decode_pp", "mid_m", "prefill", "sweep"]


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ------------------------------------------------------------------------------------------------
# workload bookkeeping (shared by both arms)
# ------------------------------------------------------------------------------------------------
def sweep_sample():
    """One case per M of the full sweep on (5120, 7168), cycling through its dtype / group-size /
    zero-point variants so that every variant appears (seeds: the case index)."""
    c = synth.CONFIGS["sweep"]
    K, N = 5120, 7168
    variants = [(dt, g, asym) for dt in c["dtypes"] for g in c["Gs"] for asym in c["asym"]]
    out = []
    for i, M in enumerate(c["Ms"]):
        dt, g, asym = variants[i % len(variants)]
        G = K if g == "K" else g
        out.append((M, K, N, G, dt, asym, c["bias"], c["scale"][0], c["scale"][1], 5000 + i))
    return out


def cases_of(name):
    if name in ("decode", "decode_pp"):
        return list(synth.config_cases("decode_2112")) + list(synth.config_cases("decode_4b"))
    if name == "sweep":
        return sweep_sample()
    return list(synth.config_cases(name))


def algo_bytes(M, K, N, G, asym, bias):
    b = K * N // 2 + 2 * (K // G) * N + 2 * M * K + 2 * M * N
    if asym:
        b += (K // G) * N // 2
    if bias:
        b += 2 * N
    return b


def narrow_bytes(M, K, N, G):
    """The narrower roofline sum: packed weights + scales + activations."""
    return K * N // 2 + 2 * (K // G) * N + 2 * M * K


def algo_flops(M, K, N):
    return 2 * M * N * K


def unit_of(name):
    return ("TFLOP/s", "tensor") if name == "prefill" else ("GB/s", "hbm")


def units_per_case(name, args):
    M, K, N, G, dt, asym, bias = args[:7]
    return algo_flops(M, K, N) if name == "prefill" else algo_bytes(M, K, N, G, asym, bias)


def scale_units(name, x):
    return x / 1e12 if name == "prefill" else x / 1e9


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of the ranks' values (each rank passes its own); x itself on one rank."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(name: str, units_per_step: float, steps: int, world: int, elapsed_ms: float) -> float:
    """Aggregate throughput: the units every rank processed (weak scaling: the same workload per
    rank) over the slowest rank's time."""
    return scale_units(name, units_per_step * steps * world) / (elapsed_ms / 1e3)


def load_peaks():
    path = os.path.join(HERE, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def tensor_peak(peaks, timed_s):
    """Dense bf16 rate (fp16 runs at the same rate): burst for a short timed region, sustained for a
    long one."""
    key = "bf16_tflops_sustained" if timed_s >= SUSTAINED_AFTER_S else "bf16_tflops"
    return float(peaks.get(key, FALLBACK_PEAKS[key])), key


def roofline_time_s(M, K, N, G, asym, bias, hbm_gbs, tflops):
    return max(algo_bytes(M, K, N, G, asym, bias) / (hbm_gbs * 1e9), algo_flops(M, K, N) / (tflops * 1e12))


def profile_traffic(kernel_tag, workload):
    """DRAM bytes per launch recorded by an ncu capture under profiles/, if the kernel source is unchanged."""
    path = os.path.join(HERE, "profiles", f"{kernel_tag}_{workload}.md")
    try:
        txt = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    h = re.search(r"source_sha256:\s*([0-9a-f]+)", txt)
    if not m or not h:
        return None
    src = os.path.join(HERE, "w4a16_int4_weight_group_gb300", "csrc", f"{kernel_tag}.cu")
    try:
        cur = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    return float(m.group(1)) if cur == h.group(1) else None


def dominant_kernel(name):
    return "gemm_prefill" if name in ("prefill", "sweep") else "gemm_decode"


def workload_config(name, per_graph=None):
    """The config object of a line; both arms print the same one for the same workload."""
    cases = cases_of(name)
    return {"workload": f"{name}: {WORKLOADS.get(name, name)}", "calls_per_step": len(cases),
            "l2": "every call reads its own weight replica; each replica pool exceeds twice the L2 cache",
            "timing": f"CUDA graphs of up to {per_graph or 100} steps, events on the launching stream"}


def cpu_description():
    model = platform.processor() or ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if not model:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
            m = re.search(r"Model name:\s*(.+)", out)
            model = m.group(1).strip() if m else platform.machine()
        except (OSError, subprocess.SubprocessError):
            model = platform.machine()
    return {"cpu_model": model, "machine": platform.machine(), "omp_num_threads": os.environ.get("OMP_NUM_THREADS")}


# ------------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.15)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for nm, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        loaded = [s for s in sm if s >= 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------------------------
# the CUDA arm
# ------------------------------------------------------------------------------------------------
class Workload:
    """Device state of one workload: weight replica pools (prepared layers), activation and output
    buffers (one per dtype, mirrored by pinned host buffers) and the call list of one step."""

    def __init__(self, name, cases, dev, w4, l2):
        import torch
        self.name, self.cases, self.dev = name, cases, dev
        tdt = {"f16": torch.float16, "bf16": torch.bfloat16}
        self.tdt = tdt

        def to_t(bits, dt):
            return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(tdt[dt])

        # one weight set per (K, N, G, dtype, asym, bias) shape, replicated so that each pool exceeds 2 x L2
        self.pools = {}
        for (M, K, N, G, dt, asym, bias, lo, hi, seed) in cases:
            key = (K, N, G, dt, asym, bias)
            if key in self.pools:
                continue
            c = synth.make_case(0, K, N, G, dt, asym=asym, bias=bias, seed=seed, scale_lo=lo, scale_hi=hi)
            wbytes = K * N // 2 + 2 * (K // G) * N + ((K // G) * N // 2 if asym else 0)
            reps = int(max(2, min(512, -(-2 * l2 // max(1, wbytes)) + 1)))
            b_q = torch.from_numpy(c.b_q).to(dev)
            sc = to_t(c.scales, dt).to(dev)
            qz = torch.from_numpy(c.qzeros).to(dev) if c.qzeros is not None else None
            bi = to_t(c.bias, dt).to(dev) if c.bias is not None else None
            b_qs = [b_q] + [b_q.clone() for _ in range(reps - 1)]
            scs = [sc] + [sc.clone() for _ in range(reps - 1)]
            qzs = None if qz is None else [qz] + [qz.clone() for _ in range(reps - 1)]
            # one prepared layer per weight replica (the public API a model would hold per layer)
            pp = name.endswith("_pp")
            layers = [w4.W4A16Linear(b_qs[r], scs[r], None if qzs is None else qzs[r], G, 8, bi, prepacked=pp)
                      for r in range(reps)]
            if pp:  # the prepacked layers keep their own copies; the canonical replicas are not needed
                b_qs = None
            self.pools[key] = {"layers": layers, "reps": reps, "keep": (b_qs, scs, qzs, bi)}
        # activations and outputs of all the calls of a step: one device byte buffer each (16-byte
        # aligned slices, viewed in each call's dtype), mirrored by pinned host buffers; the end-to-end
        # leg moves a step's inputs with one host-to-device copy and its results with one
        # device-to-host copy
        def padded(elems):
            return ((2 * elems + 15) // 16) * 16
        a_bytes = sum(padded(M * K) for (M, K, *_r) in cases)
        o_bytes = sum(padded(M * N) for (M, K, N, *_r) in cases)
        self.a_dev = torch.empty(a_bytes, dtype=torch.uint8, device=dev)
        self.o_dev = torch.empty(o_bytes, dtype=torch.uint8, device=dev)
        self.a_pin = torch.empty(a_bytes, dtype=torch.uint8).pin_memory()
        self.o_pin = torch.empty(o_bytes, dtype=torch.uint8).pin_memory()
        self.calls = []
        ao = oo = 0
        for (M, K, N, G, dt, asym, bias, lo, hi, seed) in cases:
            key = (K, N, G, dt, asym, bias)
            a_host = to_t(synth.activations(M, K, dt, seed=1000 + seed), dt)
            self.a_pin[ao:ao + 2 * M * K].view(tdt[dt]).copy_(a_host.reshape(-1))
            a = self.a_dev[ao:ao + 2 * M * K].view(tdt[dt]).view(M, K)
            a.copy_(a_host)
            out = self.o_dev[oo:oo + 2 * M * N].view(tdt[dt]).view(M, N)
            self.calls.append({"key": key, "a": a, "out": out, "case": (M, K, N, G, dt, asym, bias)})
            ao += padded(M * K)
            oo += padded(M * N)
        self.counters = {key: 0 for key in self.pools}

    def call(self, c):
        pool = self.pools[c["key"]]
        r = self.counters[c["key"]] % pool["reps"]
        self.counters[c["key"]] += 1
        pool["layers"][r](c["a"], out=c["out"])

    def step(self, use_host=False):
        if use_host:
            self.a_dev.copy_(self.a_pin, non_blocking=True)
        for c in self.calls:
            self.call(c)
        if use_host:
            self.o_pin.copy_(self.o_dev, non_blocking=True)

    def io_bytes(self):
        return self.a_dev.numel(), self.o_dev.numel()


def _graph_time(fn_per_step, steps, per_graph, stream, dev, barrier=None, world=1):
    """Capture fn_per_step into CUDA graphs of per_graph steps and time exactly `steps` steps of
    replay (events on `stream`, barrier and synchronise on both sides). Returns milliseconds."""
    import torch
    per_graph = max(1, min(steps, per_graph))
    n_full, rem = divmod(steps, per_graph)
    graphs = []
    for size in [per_graph] * min(n_full, 1) + ([rem] if rem else []):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for _ in range(size):
                    fn_per_step()
        graphs.append(g)
    full_graph = graphs[0] if n_full else None
    rem_graph = graphs[-1] if rem else None
    with torch.cuda.stream(stream):  # first replay uploads the graphs
        for g in graphs:
            g.replay()
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if barrier:
        barrier()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(n_full):
            full_graph.replay()
        if rem_graph is not None:
            rem_graph.replay()
        end.record(stream)
    torch.cuda.synchronize(dev)
    if barrier:
        barrier()
    ms = max_over_ranks(start.elapsed_time(end), world, dev)
    del graphs
    return ms


def _per_case_table(wl, stream, dev, peaks, calls_per_case):
    """Each case of the workload alone: a graph of back-to-back calls on rotating replicas."""
    rows = []
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    for c in wl.calls:
        M, K, N, G, dt, asym, bias = c["case"]
        ms = _graph_time(lambda c=c: wl.call(c), calls_per_case, calls_per_case, stream, dev)
        us = ms * 1e3 / calls_per_case
        gbs = algo_bytes(M, K, N, G, asym, bias) / us / 1e3
        tfs = algo_flops(M, K, N) / us / 1e6
        roof_us = roofline_time_s(M, K, N, G, asym, bias, hbm, burst) * 1e6
        rows.append({"M": M, "K": K, "N": N, "G": G, "dtype": dt, "zp": "asym" if asym else "sym", "us": round(us, 3),
                     "GB/s": round(gbs, 1), "TFLOP/s": round(tfs, 2), "frac_hbm": round(gbs / hbm, 4),
                     "frac_tensor": round(tfs / burst, 4), "frac_roofline": round(roof_us / us, 4),
                     "GB/s_narrow": round(narrow_bytes(M, K, N, G) / us / 1e3, 1)})
    return rows


def measure_workload(name, wl, args, stream, dev, peaks, world, barrier, per_case):
    """Warm-up, then exactly args.steps steps from CUDA graphs; the aggregate and both fractions."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            wl.step()
    torch.cuda.synchronize(dev)
    ms = _graph_time(wl.step, args.steps, args.graph_steps, stream, dev, barrier, world)
    cases = [c["case"] for c in wl.calls]
    bytes_step = sum(algo_bytes(M, K, N, G, asym, bias) for (M, K, N, G, dt, asym, bias) in cases)
    narrow_step = sum(narrow_bytes(M, K, N, G) for (M, K, N, G, *_r) in cases)
    flops_step = sum(algo_flops(M, K, N) for (M, K, N, *_r) in cases)
    timed_s = ms / 1e3
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    tpk, tkey = tensor_peak(peaks, timed_s)
    t_step = timed_s / args.steps
    gbs = bytes_step * world / t_step / 1e9
    tfs = flops_step * world / t_step / 1e12
    roof_step = sum(roofline_time_s(M, K, N, G, asym, bias, hbm, tpk) for (M, K, N, G, dt, asym, bias) in cases)
    unit, bound = unit_of(name)
    value = tfs if unit == "TFLOP/s" else gbs
    peak = tpk if bound == "tensor" else hbm
    entry = {"value": round(value, 3), "unit": unit, "ms_per_step": round(ms / args.steps, 6), "steps": args.steps,
             "calls_per_step": len(cases),
             "roofline": {"bound": bound, "achieved": round(value, 3), "peak": peak, "unit": unit,
                          "frac": round(value / peak, 4),
                          "traffic": profile_traffic(dominant_kernel(name), name),
                          "peak_source": "hbm_gbs" if bound == "hbm" else tkey, "kernel": dominant_kernel(name),
                          "frac_hbm": round(gbs / hbm, 4), "frac_tensor": round(tfs / tpk, 4),
                          "frac_roofline_time": round(roof_step / t_step, 4),
                          "GB/s": round(gbs, 1), "GB/s_narrow": round(narrow_step * world / t_step / 1e9, 1),
                          "TFLOP/s": round(tfs, 2)}}
    if per_case:
        entry["cases"] = _per_case_table(wl, stream, dev, peaks, max(8, min(args.steps, args.case_calls)))
    return entry, ms


def run_cuda(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    import w4a16_int4_weight_group_gb300 as w4
    from w4a16_int4_weight_group_gb300 import build as w4build
    w4build.build()
    w4.lib()

    def barrier():
        if world > 1:
            dist.barrier()

    name = args.config
    cases = cases_of(name)
    if args.case is not None:
        cases = [cases[args.case]]  # one case of the workload (for profiler captures)
    unit, bound = unit_of(name)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream(dev)

    wl = Workload(name, cases, dev, w4, l2)
    clocks = ClockSampler(local_rank)
    clocks.start()
    launches_before = w4.w4a16_debug_launch_count()
    head, elapsed_ms = measure_workload(name, wl, args, stream, dev, peaks, world, barrier, per_case=False)
    launches = w4.w4a16_debug_launch_count() - launches_before
    clk = clocks.stop()
    # library launches inside one timed step: the graphs replay what was captured (warm-up steps and
    # the capture itself count as launches of the host calls; the replays do not call the host)
    launches_per_step = len(wl.calls)
    value = head["value"]

    # ---- end to end through the public API with host buffers (eager, copies inside) ----
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            wl.step(use_host=True)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    units_step = sum(units_per_case(name, c["case"]) for c in wl.calls)
    e2e_value = whole_job_value(name, units_step, e2e_steps, world, e2e_ms)
    h2d, d2h = wl.io_bytes()

    # ---- every other measurement workload, timed the same way, with a per-case table ----
    side = {}
    if args.case is None and not args.no_side and world == 1:
        del wl
        torch.cuda.empty_cache()
        for other in SIDE_WORKLOADS:
            if other == name:
                continue
            owl = Workload(other, cases_of(other), dev, w4, l2)
            entry, _ = measure_workload(other, owl, args, stream, dev, peaks, world, None, per_case=True)
            entry["config"] = workload_config(other, args.graph_steps)["workload"]
            side[other] = entry
            del owl
            torch.cuda.empty_cache()

    if rank != 0:
        return None
    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "/".join(sorted({c[4] for c in cases})),
        "data": "synthetic", "config": workload_config(name, args.graph_steps),
        "roofline": dict(head["roofline"], peak_source=f"{peak_src} ({head['roofline']['peak_source']})"),
        "e2e": {"value": round(e2e_value, 3), "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps},
        "gpu_launches": int(launches_per_step * args.steps),
        "gpu_launches_host_calls": int(launches),
        "clocks": clk,
    }
    if side:
        line["workloads"] = side
    if args.case is not None:
        line["config"]["case"] = args.case
    if not args.no_cpu_baseline and world == 1 and args.case is None:
        line["cpu_baseline"] = cpu_baseline(name, cases, budget_s=args.cpu_seconds)
    return line


# ------------------------------------------------------------------------------------------------
# the CPU oracle (baseline leg and the reference arm)
# ------------------------------------------------------------------------------------------------
def _oracle_case(args):
    M, K, N, G, dt, asym, bias, lo, hi, seed = args
    return synth.make_case(M, K, N, G, dt, asym=asym, bias=bias, seed=seed, scale_lo=lo, scale_hi=hi)


def cpu_baseline(name, cases, budget_s=10.0, per_step_s=None):
    """Time the oracle, as it stands, on column blocks of the workload's cases for about budget_s."""
    import oracle
    made = [_oracle_case(c) for c in cases]
    done_units, t_total, n_calls, cols_total, cols_full = 0.0, 0.0, 0, 0, 0
    i = 0
    deadline = time.perf_counter() + budget_s
    while time.perf_counter() < deadline or n_calls == 0:
        c = made[i % len(made)]
        args = cases[i % len(cases)]
        ncols = c.N if per_step_s is None else max(8, min(c.N, 256))
        cols = np.arange(ncols)
        t0 = time.perf_counter()
        oracle.gemm_ref(c.a, c.b_q, c.scales, c.qzeros, c.G, c.zp_bias, c.bias, c.dtype, cols=cols)
        t_total += time.perf_counter() - t0
        done_units += units_per_case(name, args) * ncols / c.N
        cols_total += ncols
        cols_full += c.N
        n_calls += 1
        i += 1
    unit, _ = unit_of(name)
    return dict({"value": round(scale_units(name, done_units) / t_total, 6), "unit": unit, "cores": _CPU_THREADS,
                 "kind": "oracle",
                 "sample": f"{n_calls} oracle calls cycling over the {len(cases)} cases of '{name}' "
                           f"({cols_total} of {cols_full} output columns; units scaled by the columns computed), "
                           f"{t_total:.1f} s of CPU time, numpy fp64 with {_CPU_THREADS} BLAS threads"},
                **cpu_description())


def run_reference(args, rank, world):
    if rank != 0:
        return None
    name = args.config
    cases = cases_of(name)
    import oracle
    made = [_oracle_case(c) for c in cases]
    budget = max(0.02, min(2.0, args.ref_seconds / max(1, args.steps + args.warmup)))

    # calibrate: oracle throughput in output columns per second on the first case
    c0 = made[0]
    t0 = time.perf_counter()
    oracle.gemm_ref(c0.a, c0.b_q, c0.scales, c0.qzeros, c0.G, c0.zp_bias, c0.bias, c0.dtype, cols=np.arange(min(64, c0.N)))
    cols_per_s = min(64, c0.N) / max(1e-6, time.perf_counter() - t0)

    def step(i):
        c = made[i % len(made)]
        ncols = int(max(8, min(c.N, (budget * cols_per_s) // 8 * 8)))
        t = time.perf_counter()
        oracle.gemm_ref(c.a, c.b_q, c.scales, c.qzeros, c.G, c.zp_bias, c.bias, c.dtype, cols=np.arange(ncols))
        return time.perf_counter() - t, units_per_case(name, cases[i % len(cases)]) * ncols / c.N, ncols

    for i in range(args.warmup):
        step(i)
    tot_t, tot_u, tot_cols = 0.0, 0.0, 0
    for i in range(args.steps):
        dt, u, nc = step(i)
        tot_t += dt
        tot_u += u
        tot_cols += nc
    unit, _ = unit_of(name)
    value = scale_units(name, tot_u) / tot_t
    sample = (f"each step: the oracle over one case of '{name}' (cycling), restricted to its first output "
              f"columns ({tot_cols} columns over {args.steps} steps); units scaled by the columns computed")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * tot_t / max(1, args.steps), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "/".join(sorted({c[4] for c in cases})),
            "data": "synthetic", "config": workload_config(name, getattr(args, "graph_steps", None)),
            "cpu_baseline": dict({"value": round(value, 6), "unit": unit, "cores": _CPU_THREADS, "kind": "oracle",
                                  "sample": sample}, **cpu_description()),
            "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    ap.add_argument("--config", choices=sorted(WORKLOADS), default="decode")
    ap.add_argument("--graph-steps", type=int, default=100, help="steps captured per CUDA graph")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--case-calls", type=int, default=50, help="calls per case in the per-case tables")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU baseline budget")
    ap.add_argument("--ref-seconds", type=float, default=120.0, help="reference-arm budget for all steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-side", action="store_true", help="time the named workload only")
    ap.add_argument("--case", type=int, default=None, help="run only this case of the workload (profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        log(f"note: --gpus {args.gpus} but WORLD_SIZE={world}; using WORLD_SIZE")

    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        line = run_cuda(args, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
