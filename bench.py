#!/usr/bin/env python3
"""Throughput of the W4A16 linear layer on GB300: one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl cuda|reference] [--config NAME]

A step is one pass of the hot path over one batch of the workload: one w4a16_gemm call (validation,
runtime dispatch, weight streaming, dequantisation, multiply-accumulate, split-K reduction and the
bias/cast epilogue) for every (M, K, N) case of the workload. Weight packing is a model-load step and
is not part of a step.

Default workload "decode_2112" (the non-128-aligned decode layers of the PR #43731 report's
motivation): M in {1, 2, 4, 5, 8} x (K, N) in {(1152, 4224), (2112, 1152)}, G = 32, bf16,
symmetric uint4b8, scales U[0.005, 0.02], A ~ N(0, 1). Metric: decode GB/s over the algorithmic bytes
K*N/2 + 2(K/G)N [+ (K/G)N/2] + 2MK + 2MN [+ 2N] per call. "prefill" reports TFLOP/s (2MNK per call);
"mid_m" (17 <= M <= 64, served by the prefill kernel split over clusters) reports GB/s like decode.

Timing: W eager warm-up steps through the C ABI, then exactly K steps replayed from CUDA graphs (the
library's calls are capture-safe), bracketed by CUDA events on the launching stream, with a barrier
and a device synchronise on both sides; every call reads its own replica of the weights, and the
replica pool is larger than twice the L2 cache, so weights stream from HBM. Under torchrun each rank
runs the same workload on its own GPU (replicas, weak scaling) and the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
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

WORKLOADS = {
    "decode_2112": "decode, non-Marlin-aligned: M in {1,2,4,5,8} x (K,N) in {(1152,4224),(2112,1152)}, "
                   "G=32, bf16, symmetric uint4b8, scales U[0.005,0.02], A~N(0,1)",
    "decode_4b": "decode 4B-class: M in {1,4,8} x (K,N) in {(2560,3840),(2560,19456),(9728,2560)}, G=128, "
                 "fp16, asymmetric qzeros, fp16 bias N(0,0.1)",
    "prefill": "prefill: M in {512,1024,4096} x (K,N) in {(5120,34816),(17408,5120)}, G=64, bf16, "
               "asymmetric qzeros, scales U[0.002,0.01]",
    "mid_m": "mid M: M in {17,24,32,64} x (K,N) in {(5120,7168),(17408,5120)}, G=128, bf16, symmetric "
             "uint4b8, scales U[0.005,0.02], A~N(0,1)",
    "tiny": "tiny: M=4, K=256, N=512, G=128, fp16, symmetric",
}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ------------------------------------------------------------------------------------------------
# workload bookkeeping (shared by both arms)
# ------------------------------------------------------------------------------------------------
def cases_of(name):
    return list(synth.config_cases(name))


def algo_bytes(M, K, N, G, asym, bias):
    b = K * N // 2 + 2 * (K // G) * N + 2 * M * K + 2 * M * N
    if asym:
        b += (K // G) * N // 2
    if bias:
        b += 2 * N
    return b


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


def profile_traffic(kernel_tag, workload):
    """dram bytes per launch recorded by an ncu capture under profiles/, if the kernel source is unchanged."""
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
def run_cuda(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    import w4a16_int4_weight_group_gb300 as w4
    from w4a16_int4_weight_group_gb300 import build as w4build
    w4build.build()
    w4.lib()

    name = args.config
    cases = cases_of(name)
    if args.case is not None:
        cases = [cases[args.case]]  # one case of the workload (for profiler captures)
    unit, bound = unit_of(name)
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}

    def to_t(bits, dt):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(tdt[dt])

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    # one weight set per (K, N, G, dtype, asym) shape, replicated so that each pool exceeds 2 x L2
    shapes = {}
    for (M, K, N, G, dt, asym, bias, lo, hi, seed) in cases:
        key = (K, N, G, dt, asym, bias)
        if key not in shapes:
            c = synth.make_case(0, K, N, G, dt, asym=asym, bias=bias, seed=seed, scale_lo=lo, scale_hi=hi)
            shapes[key] = c
    pools = {}
    for key, c in shapes.items():
        K, N, G, dt, asym, bias = key
        wbytes = K * N // 2 + 2 * (K // G) * N + ((K // G) * N // 2 if asym else 0)
        reps = int(max(2, min(512, -(-2 * l2 // max(1, wbytes)) + 1)))
        b_q = torch.from_numpy(c.b_q).to(dev)
        sc = to_t(c.scales, dt).to(dev)
        qz = torch.from_numpy(c.qzeros).to(dev) if c.qzeros is not None else None
        bi = to_t(c.bias, dt).to(dev) if c.bias is not None else None
        pools[key] = {"b_q": [b_q] + [b_q.clone() for _ in range(reps - 1)],
                      "scales": [sc] + [sc.clone() for _ in range(reps - 1)],
                      "qzeros": None if qz is None else [qz] + [qz.clone() for _ in range(reps - 1)],
                      "bias": bi, "reps": reps, "G": G}
        pool = pools[key]
        # one prepared layer per weight replica (the public API a model would hold per layer)
        pool["layers"] = [w4.W4A16Linear(pool["b_q"][r], pool["scales"][r],
                                         None if qz is None else pool["qzeros"][r], G, 8, bi)
                          for r in range(reps)]
    # Activations and outputs of all the calls of a step live in one device buffer each (16-byte
    # aligned slices), mirrored by one pinned host buffer each: the end-to-end leg moves a step's
    # inputs with one host-to-device copy and its results with one device-to-host copy.
    a_elems = [((M * K + 7) // 8) * 8 for (M, K, *_r) in cases]
    o_elems = [((M * N + 7) // 8) * 8 for (M, K, N, *_r) in cases]
    edt = tdt[cases[0][4]]
    a_dev = torch.empty(sum(a_elems), dtype=edt, device=dev)
    o_dev = torch.empty(sum(o_elems), dtype=edt, device=dev)
    a_pin = torch.empty(sum(a_elems), dtype=edt).pin_memory()
    o_pin = torch.empty(sum(o_elems), dtype=edt).pin_memory()
    calls = []
    ao = oo = 0
    for i, (M, K, N, G, dt, asym, bias, lo, hi, seed) in enumerate(cases):
        key = (K, N, G, dt, asym, bias)
        a_host = to_t(synth.activations(M, K, dt, seed=1000 + seed), dt)
        a_pin[ao:ao + M * K].copy_(a_host.reshape(-1))
        a = a_dev[ao:ao + M * K].view(M, K)
        a.copy_(a_host)
        out = o_dev[oo:oo + M * N].view(M, N)
        calls.append({"key": key, "a": a, "out": out, "units": units_per_case(name, (M, K, N, G, dt, asym, bias)),
                      "M": M, "K": K, "N": N})
        ao += a_elems[i]
        oo += o_elems[i]
    counters = {key: 0 for key in pools}
    stream = torch.cuda.Stream(dev)

    def one_step(use_host=False):
        if use_host:
            a_dev.copy_(a_pin, non_blocking=True)
        for c in calls:
            pool = pools[c["key"]]
            r = counters[c["key"]] % pool["reps"]
            counters[c["key"]] += 1
            pool["layers"][r](c["a"], out=c["out"])
        if use_host:
            o_pin.copy_(o_dev, non_blocking=True)

    def barrier():
        if world > 1:
            dist.barrier()

    # ---- warm-up: eager calls through the C ABI ----
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            one_step()
    torch.cuda.synchronize(dev)

    # ---- capture: one graph holds `per_graph` steps with their own weight replicas ----
    per_graph = max(1, min(args.steps, args.graph_steps))
    n_full, rem = divmod(args.steps, per_graph)
    graphs = []
    launches_before = w4.w4a16_debug_launch_count()
    for size in [per_graph] * min(n_full, 1) + ([rem] if rem else []):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for _ in range(size):
                    one_step()
        graphs.append((size, g))
    launches_captured = w4.w4a16_debug_launch_count() - launches_before
    full_graph = graphs[0][1] if n_full else None
    rem_graph = graphs[-1][1] if rem else None
    launches_per_step = launches_captured / max(1, (per_graph if n_full else 0) + rem)
    # replay once untimed so every graph's first upload is done
    with torch.cuda.stream(stream):
        for _, g in graphs:
            g.replay()
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(local_rank)
    clocks.start()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
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
    barrier()
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(start.elapsed_time(end), world, dev)
    units_per_step = sum(c["units"] for c in calls)
    value = whole_job_value(name, units_per_step, args.steps, world, elapsed_ms)
    launches = int(round(launches_per_step * args.steps))

    # ---- end to end through the public API with host buffers (eager, copies inside) ----
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            one_step(use_host=True)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e_value = whole_job_value(name, units_per_step, e2e_steps, world, e2e_ms)
    h2d = a_dev.numel() * a_dev.element_size()
    d2h = o_dev.numel() * o_dev.element_size()

    if rank != 0:
        return None

    peaks, peak_src = load_peaks()
    if bound == "hbm":
        peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    else:
        # a kernel timed inside a long run of back-to-back steps: the sustained bf16 figure
        peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])))
    dominant = "gemm_prefill" if name in ("prefill", "mid_m") else "gemm_decode"
    achieved = value  # every launch in the timed region is the dominant kernel (see gpu_launches)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(elapsed_ms / args.steps, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": cases[0][4], "data": "synthetic",
        "config": {"workload": f"{name}: {WORKLOADS.get(name, name)}", "calls_per_step": len(calls),
                   "l2": f"every call reads its own weight replica; replica pools > 2x L2 ({l2 >> 20} MiB)",
                   "timing": f"CUDA graphs of {per_graph} steps, events on the launching stream"},
        "roofline": {"bound": bound, "achieved": round(achieved, 3), "peak": peak, "unit": unit,
                     "frac": round(achieved / peak, 4), "traffic": profile_traffic(dominant, name),
                     "peak_source": f"{peak_src} ({'hbm_gbs' if bound == 'hbm' else 'bf16_tflops_sustained'})",
                     "kernel": dominant},
        "e2e": {"value": round(e2e_value, 3), "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps},
        "gpu_launches": launches,
        "clocks": clk,
    }
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
    return {"value": round(scale_units(name, done_units) / t_total, 6), "unit": unit, "cores": _CPU_THREADS,
            "kind": "oracle",
            "sample": f"{n_calls} oracle calls cycling over the {len(cases)} cases of '{name}' "
                      f"({cols_total} of {cols_full} output columns; units scaled by the columns computed), "
                      f"{t_total:.1f} s of CPU time, numpy fp64 with {_CPU_THREADS} BLAS threads"}


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
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cases[0][4],
            "data": "synthetic", "config": {"workload": f"{name}: {WORKLOADS.get(name, name)}"},
            "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": _CPU_THREADS, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    ap.add_argument("--config", choices=sorted(WORKLOADS), default="decode_2112")
    ap.add_argument("--graph-steps", type=int, default=100, help="steps captured per CUDA graph")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU baseline budget")
    ap.add_argument("--ref-seconds", type=float, default=120.0, help="reference-arm budget for all steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
