"""Throughput of the tiled dense matrix multiply on GB300.

One step = the two products the headline metric is quoted on, each one call of
the C entry point on inputs already resident in HBM:
  * 8192 x 8192 x 8192, bf16 inputs, fp32 accumulate and output (tgemm_bf16);
  * 4096 x 4096 x 4096, fp32 (tgemm_f32, FFMA).
``value`` = their flops (2mnk each) / their summed device time, in TFLOP/s.
Each launch is bracketed by CUDA events on the stream it runs on.  L2 hygiene:
inputs larger than L2 -- every shape keeps R copies of its inputs (R copies
>= 384 MiB, about 3x the 129 MB L2) and each launch reads the next copy, so no
launch finds its operands in L2.  (A write-flush between launches was not used:
it leaves ~129 MB of dirty lines that are written back during the next kernel,
which penalises memory-bound kernels for work they did not do.)

The same JSON line carries, for information, the other measured shapes
(4096^3 on the TF32 tensor-core path, 16 x 8192 x 8192 bf16, the
4097 x 3001 x 1023 edge-tile case, 1024 x 1024 x 8192 on tensor-core split-K
pieces, the pages' kernels), a roofline object for the kernel
taking most of the step's time, the end-to-end number through the C ABI from
pinned host buffers (every step copies its inputs in and its results out; the
copies run on their own streams beside the products, and the same step with
nothing overlapped is reported with it), the CPU oracle timed on a bounded sample of the same
workload, and the SM clocks sampled while timing.  After the timed region each
shape is also launched back to back between a single event pair
(``ms_back_to_back``): the per-launch event pairs add a microsecond or two,
which shows on the 16 x 8192 x 8192 case (~28 us); ``ms`` and the roofline
keep the per-launch figure.

``--impl reference`` times the CPU oracle instead (a bounded sample of the
same workload per step) and prints the same metric for it.

Per shape, ``ms`` is the median of the per-launch event timings (the mean is
reported beside it).  The FP32 FMA peak is derived at run time from the SM
count the device reports and the highest SM clock nvidia-smi reported while
timing; tensor-core fractions are given against the measured peaks of
MEASURED_PEAKS.json (``frac``) and against the nominal dense peaks
(``frac_of_nominal``).  DRAM traffic per call comes from the ncu table
profiles/dram_traffic.csv and is reported as null once the kernel sources it
was captured on have changed.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tgemm|reference]
                       [--shard rows|replicas]
Under torchrun (N > 1) the step's two products are split by rows across the
ranks by default (``--shard rows``: rank r computes its row block of each C
from the same rows of A and all of B, one independent call per product on its
own GPU, no collective on the data path; strong scaling, ``value`` = the full
products' flops / the slowest rank's step time).  ``--shard replicas`` runs
the whole step on every rank instead (weak scaling).  Rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOPS (2mnk/s) at 4096³ fp32 & 8192³ bf16; % of GB300 roofline"
UNIT = "TFLOP/s"
FP32_LANES_PER_SM = 128          # FP32 FMA lanes per SM (sm_100 family)
NOMINAL_BF16, NOMINAL_TF32 = 2250.0, 1100.0   # dense tensor peaks, TFLOP/s
CSRC = os.path.join(ROOT, "dense_tiled_matrix_gb300", "csrc")
TRAFFIC_TABLE = os.path.join(ROOT, "profiles", "dram_traffic.csv")

# name -> (workload, entry, dtype)
PARTS = {
    "bf16_8192": ("bf16_8192", "bf16", "bf16"),
    "f32_4096": ("n4096", "f32", "f32"),
}
EXTRAS = {
    "tf32_4096": ("n4096", "tf32", "f32"),
    "skinny_bf16": ("skinny", "bf16", "bf16"),
    "irregular_f32": ("irregular", "f32", "f32"),
    "irregular_tf32": ("irregular", "tf32", "f32"),
    "irregular_bf16": ("irregular", "bf16", "bf16"),
    # fewer tensor-core tiles than SMs: split-K pieces and their reduce
    "long_k_tf32": ("long_k", "tf32", "f32"),
    "long_k_bf16": ("long_k", "bf16", "bf16"),
    # the pages' own experiment (naive -> tiled -> libtgemm) at 1024^3 and 4096^3
    "f32_1024": ("int1024", "f32", "f32"),
    "pages_naive_1024": ("int1024", "pages_naive", "f32"),
    "pages_tiled16_1024": ("int1024", "pages_tiled16", "f32"),
    "pages_tiled32_1024": ("int1024", "pages_tiled32", "f32"),
    "pages_naive_4096": ("n4096", "pages_naive", "f32"),
    "pages_tiled16_4096": ("n4096", "pages_tiled16", "f32"),
    "pages_tiled32_4096": ("n4096", "pages_tiled32", "f32"),
}
SLOW_EXTRAS = {"pages_naive_4096", "pages_tiled16_4096", "pages_tiled32_4096"}
SLOW_EXTRA_ITERS = 4   # timed launches of the pages' kernels at 4096^3 (tens of ms each)
KERNEL_NAMES = {"f32": "ffma_f32_ws_kernel (912 tiles, then 448 split pieces) + ffma_f32_reduce_kernel (one tgemm_f32 call)", "tf32": "transpose_tma_kernel + umma_kernel<1, 1, 1, 224, 0, 0, 4>", "bf16": "umma_kernel<0, 0, 1, 256, 0, 0, 4>"}


def source_digest(files):
    """First 16 hex digits of the sha256 of the named csrc files, concatenated in order."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_table(path=TRAFFIC_TABLE):
    """part -> {"bytes": int or None, "source": str, "stale": bool} from the ncu traffic table.
    An entry whose kernel sources have changed since the capture gives bytes None."""
    out = {}
    try:
        with open(path, newline="") as fh:
            rows = [line for line in fh if not line.startswith("#")]
    except OSError:
        return out
    for row in csv.DictReader(rows):
        files = row["sources"].split()
        try:
            current = source_digest(files)
        except OSError:
            current = None
        stale = current != row["sha256_16"]
        out[row["part"]] = {"bytes": None if stale else int(row["bytes_per_call"]),
                            "source": f"{row['summary']} ({row['kernels']})", "stale": stale}
    return out


def plan_of(entry, m, n, k, sm_count):
    """The tiles libtgemm picks for a shape (tgemm_plan / tgemm_plan_f32: host
    arithmetic), or None for the pages' comparator kernels."""
    from dense_tiled_matrix_gb300 import tgemm
    if entry == "f32":
        return tgemm.tgemm_plan_f32(m, n, k, sm_count)
    if entry in ("tf32", "bf16"):
        return tgemm.tgemm_plan(entry, m, n, k, sm_count)
    return None


def fp32_peak(sm_count, sm_max_mhz):
    """(TFLOP/s, derivation) of the FP32 FMA peak: SMs x lanes x 2 flop x max SM clock."""
    tf = sm_count * FP32_LANES_PER_SM * 2 * sm_max_mhz * 1e6 / 1e12
    return tf, f"{sm_count} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 flop x {sm_max_mhz:.0f} MHz = {tf:.2f} TFLOP/s"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def roofline_for(entry, case, seconds, peaks, peaks_src, fp32=None):
    """Roofline object of one launch: skinny bf16 is HBM-bound, the rest compute-bound.
    ``fp32`` = (peak TFLOP/s, derivation) of the FP32 FMA pipes (fp32_peak)."""
    flops = 2.0 * case.m * case.n * case.k
    es = 2 if entry == "bf16" else 4
    bytes_ = es * (case.m * case.k + case.k * case.n) + 4 * case.m * case.n
    if entry == "bf16" and case.m <= 64:
        achieved = bytes_ / seconds / 1e9
        peak = float(peaks["hbm_gbs"])
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": None,
                "peak_source": f"hbm_gbs of {peaks_src}", "algorithmic_bytes": int(bytes_)}
    achieved = flops / seconds / 1e12
    nominal = None
    if entry == "f32" or entry.startswith("pages"):
        peak, src = fp32 if fp32 is not None else fp32_peak(152, 2070.0)
        bound = "alu"
    elif entry == "bf16":
        peak, src = float(peaks["bf16_tflops"]), f"bf16_tflops (burst, cuBLAS) of {peaks_src}"
        bound, nominal = "tensor", NOMINAL_BF16
    else:
        peak = float(peaks["bf16_tflops"]) * NOMINAL_TF32 / NOMINAL_BF16
        src = f"bf16_tflops (burst, cuBLAS) of {peaks_src} x 1.1/2.25 (nominal tf32/bf16)"
        bound, nominal = "tensor", NOMINAL_TF32
    out = {"bound": bound, "achieved": round(achieved, 2), "peak": round(peak, 2), "unit": "TFLOP/s",
           "frac": round(achieved / peak, 4), "traffic": None, "peak_source": src,
           "algorithmic_flops": int(flops)}
    if nominal is not None:
        out["nominal_peak"] = nominal
        out["frac_of_nominal"] = round(achieved / nominal, 4)
    return out


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while timing."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.device_index = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix=f"tgemm_clocks_{os.getpid()}_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.device_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
            # wait (up to 5 s) for the first sample so the timed region is covered
            t0 = time.time()
            while time.time() - t0 < 5.0 and os.path.getsize(self.path) == 0:
                time.sleep(0.05)
        except OSError:
            self.proc = None
            if getattr(self, "fh", None) is not None:
                self.fh.close()
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        try:
            os.unlink(self.path)   # the log is only read here
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "window": "warm-up, timed steps and extra shapes (nvidia-smi every 100 ms)",
                "power_w_max": max(power) if power else None}


def step_config(world, shard_rows):
    """The ``config`` object of the JSON line (the same for both arms)."""
    if shard_rows:
        parallelism = f"rows x{world} (each rank its row block of every product; no collective)"
    else:
        parallelism = f"replicas x{world}"
    return {"workload": "gemm 8192x8192x8192 bf16->fp32 (tcgen05) + 4096x4096x4096 fp32 (FFMA)",
            "l2": "inputs larger than L2: each launch reads the next of R input copies (>= 384 MiB per shape)",
            "parallelism": parallelism}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "tgemm" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value, world):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_sample(cases, target_s, max_rows=None):
    """Times the oracle on the first r rows of each case, growing r until one
    pass takes about target_s seconds.  Returns (flops, seconds, rows, cores)."""
    import oracle
    cores = oracle.available_cores()
    limit = min(c.m for c in cases) if max_rows is None else min(max_rows, min(c.m for c in cases))
    r = min(max(1, cores // 2), limit)
    while True:
        t0 = time.perf_counter()
        flops = 0
        for c in cases:
            oracle.gemm(c.A[:r], c.B)
            flops += 2 * r * c.n * c.k
        dt = time.perf_counter() - t0
        if dt >= 0.5 * target_s or r >= limit:
            return flops, dt, r, cores
        grow = int(r * min(8.0, 0.8 * target_s / max(dt, 1e-3)))
        r = min(limit, max(r + 1, grow))


def bench_reference(args, world, rank):
    """The CPU oracle as it stands, on a bounded sample of the step's workload:
    each step runs it on the first r rows of both products, r sized so the
    whole run (warm-up + timed steps) takes about --ref-seconds."""
    import oracle
    from dense_tiled_matrix_gb300 import inputs
    if rank != 0:
        return
    cases = [inputs.make(PARTS[p][0]) for p in PARTS]
    per_step_target = max(0.05, args.ref_seconds / (args.warmup + args.steps))
    flops, dt, rows, cores = cpu_sample(cases, target_s=per_step_target)
    per_step = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        for c in cases:
            oracle.gemm(c.A[:rows], c.B)
        if i >= args.warmup:
            per_step.append(time.perf_counter() - t0)
    total = sum(per_step)
    value = flops * len(per_step) / total / 1e12
    sample = (f"first {rows} rows of each of 8192x8192x8192 bf16 and 4096x4096x4096 fp32 per step "
              f"(fp64 oracle, {cores} threads)")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total / len(per_step) * 1e3, "higher_is_better": True,
            "scaling": "strong" if world > 1 and args.shard == "rows" else "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded SplitMix64)",
            "impl": "reference",
            "config": step_config(world, world > 1 and args.shard == "rows"),
            "reference_sample": {"rows_per_part": rows, "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def bench_tgemm(args, world, rank, local):
    import torch

    from dense_tiled_matrix_gb300 import inputs, pages, sharding, tgemm

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    tgemm.load()
    peaks, peaks_src = load_peaks()
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    stream = torch.cuda.current_stream(dev)
    rotate_bytes = 384 * 2 ** 20
    # Row sharding (N > 1, default): this rank's rows of every product of the step.
    shard_rows = world > 1 and args.shard == "rows"

    def to_dev(arr):
        import numpy as np
        if arr.dtype == np.uint16:
            return torch.from_numpy(arr.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(arr).to(dev)

    case_cache = {}

    def case_of(name):
        if name not in case_cache:
            case_cache[name] = inputs.make(name)
        return case_cache[name]

    class Shape:
        def __init__(self, m, n, k):
            self.m, self.n, self.k = m, n, k

    def prepare(spec, shard):
        wl, entry, _ = spec
        c = case_of(wl)
        cc = inputs.convert(c, "bf16" if entry == "bf16" else "f32")
        A_host = cc.A
        if shard:
            r0, r1 = sharding.rows(c.m, world, rank)
            A_host = A_host[r0:r1]
        A0, B0 = to_dev(A_host), to_dev(cc.B)
        per_copy = A0.numel() * A0.element_size() + B0.numel() * B0.element_size()
        R = max(1, -(-rotate_bytes // per_copy))
        copies = [(A0, B0)] + [(A0.clone(), B0.clone()) for _ in range(R - 1)]
        C = torch.empty((A0.shape[0], c.n), dtype=torch.float32, device=dev)
        fn = {"f32": tgemm.tgemm_f32, "tf32": tgemm.tgemm_tf32, "bf16": tgemm.tgemm_bf16,
              "pages_naive": lambda A, B, C, st: pages.tgemm_pages_naive_f32(A, B, C, st),
              "pages_tiled16": lambda A, B, C, st: pages.tgemm_pages_tiled_f32(A, B, C, 16, st),
              "pages_tiled32": lambda A, B, C, st: pages.tgemm_pages_tiled_f32(A, B, C, 32, st)}[entry]
        return Shape(A0.shape[0], c.n, c.k), copies, C, fn

    def timed(runs, iters, start=0, iters_of=None):
        """Per-launch device times (s) of `iters` launches of each of `runs`; launch i reads copy i mod R."""
        times = {name: [] for name in runs}
        # each shape in its own back-to-back run, so no launch inherits another
        # shape's dirty output lines in L2
        for name, (c, copies, C, fn) in runs.items():
            n_it = (iters_of or {}).get(name, iters)
            for it in range(start, start + n_it):
                A, B = copies[it % len(copies)]
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn(A, B, C, stream)
                e1.record(stream)
                times[name].append((e0, e1))
        torch.cuda.synchronize(dev)
        return {n: [a.elapsed_time(b) / 1e3 for a, b in v] for n, v in times.items()}

    def back_to_back(runs, iters):
        """Mean device time (s) of `iters` launches issued back to back between one event pair
        (no events in between; copies rotated as above).  Reported beside the per-launch figure:
        an event pair around every launch adds its own ~1-2 us, which matters for short kernels."""
        out = {}
        for name, (c, copies, C, fn) in runs.items():
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for it in range(iters):
                A, B = copies[it % len(copies)]
                fn(A, B, C, stream)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            out[name] = e0.elapsed_time(e1) / 1e3 / iters
        return out

    only = set(args.only.split(",")) if args.only else None
    if only and not only <= set(PARTS) | set(EXTRAS):
        raise SystemExit(f"--only: unknown parts {sorted(only - set(PARTS) - set(EXTRAS))}")
    runs = {name: prepare(spec, shard_rows) for name, spec in PARTS.items() if not only or name in only}
    extras = {} if args.no_extras or rank != 0 else {name: prepare(spec, False) for name, spec in EXTRAS.items()
                                                     if not only or name in only}

    with ClockSampler(local) as clocks:
        timed(runs, args.warmup)
        barrier(world)
        torch.cuda.synchronize(dev)
        launches0 = tgemm.tgemm_kernel_launches()
        t_wall0 = time.perf_counter()
        per = timed(runs, args.steps, start=args.warmup)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall0
        launches = tgemm.tgemm_kernel_launches() - launches0
        barrier(world)
        slow = {n: args.warmup + SLOW_EXTRA_ITERS for n in extras if n in SLOW_EXTRAS}
        extra_times = timed(extras, args.warmup + args.steps, iters_of=slow) if extras else {}
        # after the timed region: the same launches back to back (not the pages' slow kernels)
        b2b = back_to_back(runs, args.steps)
        b2b.update(back_to_back({n: r for n, r in extras.items() if n not in slow}, args.steps))
    clock_summary = clocks.summary()
    step_s = max(sum(sum(v) for v in per.values()) / args.steps, 1e-12)
    step_s = max_over_ranks(step_s, world)
    if shard_rows:
        # the full products' flops: the ranks' row blocks together cover every row once
        flops_step = sum(2.0 * case_of(PARTS[n][0]).m * runs[n][0].n * runs[n][0].k for n in runs)
        value = flops_step / step_s / 1e12
    else:
        flops_step = sum(2.0 * runs[n][0].m * runs[n][0].n * runs[n][0].k for n in runs)
        value = world * flops_step / step_s / 1e12

    # FP32 peak from the device's SM count and the highest SM clock seen while timing
    max_mhz = clock_summary.get("sm_max_mhz") or float(peaks.get("sm_max_mhz", 2070.0))
    fp32 = fp32_peak(sm_count, float(max_mhz))
    traffic = traffic_table()

    parts = {}
    for name, ts in list(per.items()) + [(n, v[args.warmup:]) for n, v in extra_times.items()]:
        c = (runs.get(name) or extras.get(name))[0]
        entry = (PARTS.get(name) or EXTRAS.get(name))[1]
        med = statistics.median(ts)
        roof_part = roofline_for(entry, c, med, peaks, peaks_src, fp32)
        if name in traffic:
            roof_part["traffic"] = traffic[name]["bytes"]
            roof_part["traffic_source"] = traffic[name]["source"] + (" -- stale: kernel changed since the capture"
                                                                     if traffic[name]["stale"] else "")
        parts[name] = {"m": c.m, "n": c.n, "k": c.k, "entry": f"tgemm_{entry}", "launches_timed": len(ts),
                       "ms": round(med * 1e3, 4), "ms_mean": round(sum(ts) / len(ts) * 1e3, 4),
                       "tflops": round(2.0 * c.m * c.n * c.k / med / 1e12, 2),
                       "roofline": roof_part}
        plan = plan_of(entry, c.m, c.n, c.k, sm_count)
        if plan is not None:
            parts[name]["plan"] = plan
        if name in b2b:
            # informational: `ms`, `tflops` and the roofline use the per-launch event pairs
            parts[name]["ms_back_to_back"] = round(b2b[name] * 1e3, 4)
            parts[name]["roofline_frac_back_to_back"] = round(roof_part["frac"] * med / b2b[name], 4)
    if runs:
        dominant = max(runs, key=lambda n: sum(per[n]))
        roof = dict(parts[dominant]["roofline"])
        roof["kernel"] = KERNEL_NAMES[PARTS[dominant][1]]
        roof["workload"] = dominant
    else:
        roof = None   # --only without a part of the step: no step, no step roofline

    # The lecture's transpose case study (naive -> coalesced shared tile ->
    # padded tile) next to libtgemm's transpose, at the lecture's 1024 x 1024
    # and at 16384 x 16384 (HBM-bound); GB/s counts the bytes read and written.
    transposes = {}
    if extras and not only:
        gen = torch.Generator(device=dev)
        gen.manual_seed(1006)
        kernels = {"tgemm_transpose_f32": lambda a, b: tgemm.tgemm_transpose_f32(a, b, stream),
                   "pages_naive": lambda a, b: pages.tgemm_pages_transpose_f32(a, b, "naive", stream),
                   "pages_coalesced": lambda a, b: pages.tgemm_pages_transpose_f32(a, b, "coalesced", stream),
                   "pages_padded": lambda a, b: pages.tgemm_pages_transpose_f32(a, b, "padded", stream)}
        for rows, cols in [(1024, 1024), (16384, 16384)]:
            nbytes = rows * cols * 4
            R = max(1, -(-rotate_bytes // nbytes))
            srcs = [torch.empty((rows, cols), device=dev).normal_(generator=gen) for _ in range(R)]
            dst = torch.empty((cols, rows), device=dev)
            for name, fn in kernels.items():
                ev = []
                for it in range(args.warmup + 10):
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    fn(srcs[it % R], dst)
                    e1.record(stream)
                    ev.append((e0, e1))
                torch.cuda.synchronize(dev)
                ts = [a.elapsed_time(b) / 1e3 for a, b in ev[args.warmup:]]
                med = statistics.median(ts)
                gbs = 2 * nbytes / med / 1e9
                transposes[f"{name}_{rows}x{cols}"] = {
                    "us": round(med * 1e6, 2), "GB_s": round(gbs, 1),
                    "frac_of_hbm": round(gbs / float(peaks["hbm_gbs"]), 4)}
            del srcs, dst

    # Read-stream ceilings (libtgemm_probes): 128 MiB -- the skinny product's B --
    # read once through TMA bulk copies and once with 128-bit loads, four
    # rotated buffers (512 MiB, about 4x L2); the skinny kernel's bandwidth is
    # reported as a fraction of each beside its fraction of the copy peak.
    read_streams = {}
    if extras and not only:
        from dense_tiled_matrix_gb300 import probes
        nbytes = 128 * 2 ** 20
        bufs = [torch.randint(-2 ** 31, 2 ** 31 - 1, (nbytes // 4,), dtype=torch.int32, device=dev)
                for _ in range(4)]
        total = torch.zeros(1, dtype=torch.int64, device=dev)
        for how in ("tma", "ldg"):
            ev = []
            for it in range(args.warmup + 20):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                probes.read_stream(bufs[it % 4], how, total, stream)
                e1.record(stream)
                ev.append((e0, e1))
            torch.cuda.synchronize(dev)
            med = statistics.median(a.elapsed_time(b) / 1e3 for a, b in ev[args.warmup:])
            gbs = nbytes / med / 1e9
            read_streams[how] = {"us": round(med * 1e6, 2), "GB_s": round(gbs, 1),
                                 "frac_of_hbm": round(gbs / float(peaks["hbm_gbs"]), 4)}
        del bufs
        if "skinny_bf16" in parts:
            sk = parts["skinny_bf16"]["roofline"]["achieved"]
            for how in read_streams:
                read_streams[how]["skinny_frac"] = round(sk / read_streams[how]["GB_s"], 4)

    # Paired-FMA ceiling (libtgemm_probes): the FFMA product's 8 x 8 register-tile
    # update with register operands only, one CTA per SM of 8 warps (the product
    # kernel's consumer warps) and of 16; the fp32 products are reported as a
    # fraction of it beside their fraction of the derived FP32 peak.
    alu_ceiling = {}
    if extras and not only:
        from dense_tiled_matrix_gb300 import probes
        ab = torch.tensor([2.0 ** -(i % 4) for i in range(8)] + [2.0 ** (j % 3 - 1) for j in range(8)],
                          dtype=torch.float32, device=dev)
        out = torch.zeros(1, dtype=torch.float64, device=dev)
        iters = 16384
        for warps in (8, 16):
            ev = []
            for it in range(args.warmup + 10):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                probes.ffma2(warps, iters, ab, out, stream)
                e1.record(stream)
                ev.append((e0, e1))
            torch.cuda.synchronize(dev)
            med = statistics.median(a.elapsed_time(b) / 1e3 for a, b in ev[args.warmup:])
            flops = 128.0 * sm_count * 32 * warps * iters
            tf = flops / med / 1e12
            alu_ceiling[f"ffma2_{warps}_warps"] = {"us": round(med * 1e6, 2), "tflops": round(tf, 2),
                                                   "frac_of_fp32_peak": round(tf / fp32[0], 4)}
        best = max(v["tflops"] for v in alu_ceiling.values())
        for name in ("f32_4096", "irregular_f32", "f32_1024"):
            if name in parts:
                alu_ceiling[f"{name}_frac"] = round(parts[name]["tflops"] / best, 4)

    # End to end through the C ABI: pinned host inputs -> device, product, result -> host,
    # every step.  The copies run as a pipeline beside the products: inputs go in on
    # two copy streams (each matrix in two halves of rows), the products run on the
    # compute stream as each part's inputs land, results come back on two more streams
    # as each product finishes, and two sets of device buffers alternate between steps
    # so that step i + 1's inputs can land while step i computes and reads back (each
    # set is reused only after the products and the read-back that used it two steps
    # before are done).  Measured on GB300: one copy stream per direction reaches the
    # link's rate in that direction (210 GB/s in, 192 out), but copies in both
    # directions at once moved 202 / 248 / 279 GB/s with 1 / 2 / 4 streams.
    e2e = None
    if not args.no_e2e and runs:
        host = {}
        h2d = d2h = 0
        for name, (c, copies, C, fn) in runs.items():
            A, B = copies[0]
            hA = torch.empty(A.shape, dtype=A.dtype, pin_memory=True)
            hB = torch.empty(B.shape, dtype=B.dtype, pin_memory=True)
            hA.copy_(A)
            hB.copy_(B)
            hC = torch.empty(C.shape, dtype=C.dtype, pin_memory=True)
            sets = [(torch.empty_like(A), torch.empty_like(B), torch.empty_like(C)) for _ in range(2)]
            host[name] = (hA, hB, hC, sets, runs[name][3])
            h2d += hA.numel() * hA.element_size() + hB.numel() * hB.element_size()
            d2h += hC.numel() * hC.element_size()
        s_ins = [torch.cuda.Stream(dev) for _ in range(2)]
        s_outs = [torch.cuda.Stream(dev) for _ in range(2)]
        freed = [None, None]   # per buffer set: the events after which it may be overwritten

        def halves(t):
            h = (t.shape[0] + 1) // 2
            return (t[:h], t[h:])

        def e2e_step(i):
            b = i % 2
            landed, done = {}, {}
            for s_in in s_ins:
                for ev in freed[b] or ():
                    s_in.wait_event(ev)
            for name, (hA, hB, hC, sets, fn) in host.items():
                dA, dB, _ = sets[b]
                landed[name] = []
                for j, s_in in enumerate(s_ins):
                    with torch.cuda.stream(s_in):
                        halves(dA)[j].copy_(halves(hA)[j], non_blocking=True)
                        halves(dB)[j].copy_(halves(hB)[j], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(s_in)
                    landed[name].append(ev)
            for ev in freed[b] or ():
                stream.wait_event(ev)
            for name, (hA, hB, hC, sets, fn) in host.items():
                dA, dB, dC = sets[b]
                for ev in landed[name]:
                    stream.wait_event(ev)
                fn(dA, dB, dC, stream)
                done[name] = torch.cuda.Event()
                done[name].record(stream)
            freed[b] = []
            for j, s_out in enumerate(s_outs):
                for name, (hA, hB, hC, sets, fn) in host.items():
                    s_out.wait_event(done[name])
                    with torch.cuda.stream(s_out):
                        halves(hC)[j].copy_(halves(sets[b][2])[j], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(s_out)
                freed[b].append(ev)

        for i in range(args.warmup):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        barrier(world)
        freed[0] = freed[1] = None
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for s_in in s_ins:
            s_in.wait_event(e0)
        for i in range(args.steps):
            e2e_step(i)
        for ev in freed[(args.steps - 1) % 2]:
            stream.wait_event(ev)
        if args.steps > 1:
            for ev in freed[args.steps % 2]:
                stream.wait_event(ev)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3 / args.steps, world)

        # The same step with nothing overlapped (copies, products and read-back one
        # after another on one stream), for comparison.
        def serial_step():
            for hA, hB, hC, sets, fn in host.values():
                dA, dB, dC = sets[0]
                dA.copy_(hA, non_blocking=True)
                dB.copy_(hB, non_blocking=True)
                fn(dA, dB, dC, stream)
                hC.copy_(dC, non_blocking=True)

        serial_step()
        torch.cuda.synchronize(dev)
        barrier(world)
        e0.record(stream)
        for _ in range(args.steps):
            serial_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        serial_s = max_over_ranks(e0.elapsed_time(e1) / 1e3 / args.steps, world)
        scale = 1 if shard_rows else world
        e2e = {"value": round(scale * flops_step / e2e_s / 1e12, 3), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(e2e_s * 1e3, 3),
               "how": "input copies (two streams), products and read-back (two streams) pipelined, two buffer sets",
               "serial": {"value": round(scale * flops_step / serial_s / 1e12, 3),
                          "ms_per_step": round(serial_s * 1e3, 3),
                          "how": "the same copies and products one after another on one stream"}}

    status = tgemm.tgemm_get_device_status(stream)
    if status != tgemm.TGEMM_OK:
        raise RuntimeError(f"device status after the bench: {tgemm.tgemm_status_string(status)}")

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and not only:
        flops, dt, rows, cores = cpu_sample([case_of(PARTS[p][0]) for p in PARTS], target_s=args.cpu_seconds)
        cpu = {"value": flops / dt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"first {rows} rows of each of the step's two products (fp64 oracle), {dt:.1f} s"}

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 4), "higher_is_better": True,
                "scaling": "strong" if shard_rows else "weak", "vs_baseline": None, "dtype": "bf16+f32",
                "data": "synthetic (seeded SplitMix64; bf16 N(0,1)/sqrt(k), fp32 N(0,1))",
                "config": step_config(world, shard_rows),
                "roofline": roof, "parts": parts, "transposes": transposes, "read_streams": read_streams, "alu_ceiling": alu_ceiling,
                "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": int(launches), "clocks": clock_summary,
                "fp32_peak": {"tflops": round(fp32[0], 2), "derivation": fp32[1]},
                "wall_s_timed_region": round(t_wall, 3), "impl": "tgemm"}
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["tgemm", "reference"], default="tgemm")
    ap.add_argument("--shard", choices=["rows", "replicas"], default="rows",
                    help="N > 1: split each product's rows across the ranks (strong scaling, default) "
                         "or run the whole step on every rank (weak scaling)")
    ap.add_argument("--no-extras", action="store_true", help="skip the informational extra shapes")
    ap.add_argument("--only", default="", help="profiling aid: time only these comma-separated parts "
                                                "(names of `parts` in the JSON line); no CPU baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffer) measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip timing the CPU oracle")
    ap.add_argument("--cpu-seconds", type=float, default=20.0, help="target length of the CPU-oracle sample")
    ap.add_argument("--ref-seconds", type=float, default=90.0,
                    help="--impl reference: target length of the whole oracle run (warm-up + steps)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        bench_reference(args, world, rank)
    else:
        bench_tgemm(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
