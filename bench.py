#!/usr/bin/env python
"""Benchmark of the low-bit GEMM library on GB300.

Workload (one step): the 8-bit GEMM shape sweep -- M, N, K each in
{64, 128, ..., 16384}, 729 shapes, operands uniform in [-127, 127] -- run once
per shape through lbgemm_run with the kernel the selection table picked.
Before the timed steps the sweep itself runs, for 8-, 4- and 1-bit operands
(tune.py): every shape is timed under all nine tile x stage variants and the
shape-route kernels that can run it (lbgemm_candidates), and the table
stores the labelled variant and the dispatch's pick, each only once it has
won again head to head against the default variant.  L2 is flushed before
every GEMM, outside the timed intervals; the step time is the sum of the
per-GEMM CUDA-event times.

value = sum over the 729 shapes of 2*M*N*K / step time, in TOPS (integer
operations, 2 per multiply-add).  The same line reports, per bit width, the
selected-vs-default speedups on an independent interleaved re-time with its
measured noise floor; the other configurations and the linear layer; the
roofline of the dominant kernel; an end-to-end number through the
host-buffer entry point; and the CPU oracle on a row sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

SIZES = [64, 128, 256, 512, 1024, 2048, 4096, 8192, 16384]
SWEEP = [(m, n, k) for m in SIZES for n in SIZES for k in SIZES]
# Balanced ninth of the sweep: every (M, N) pair once, each K value nine times.
E2E_SHAPES = [(SIZES[i], SIZES[j], SIZES[(-(i + j)) % 9]) for i in range(9) for j in range(9)]
MAXD = SIZES[-1]
E2E_PASSES = 5
METRIC = "int8 GEMM TOPS over the 729-shape sweep (selected variant)"
BITS = (8, 4, 1)
SEED_OF = {8: 2, 4: 3, 1: 4}  # workload numbers of the 8-, 4- and 1-bit configurations
ROUTE_TABLE = 0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--sweep-reps", type=int, default=10,
                   help="runs per candidate and shape in the selection sweep (median)")
    p.add_argument("--retime-reps", type=int, default=20,
                   help="runs per arm and shape in the head-to-head checks and the re-time")
    p.add_argument("--offgrid", type=int, default=100,
                   help="random shapes per bit width off the grid for the fallback check")
    p.add_argument("--shapes", type=int, default=0, help="debug: use only the first N shapes")
    p.add_argument("--no-cpu", action="store_true", help="debug: skip the CPU oracle sample")
    p.add_argument("--dump", default="", help="write per-shape sweep data (JSON) to this path")
    p.add_argument("--table", default="",
                   help="profiling: load this selection table instead of running the sweep "
                        "(no selection re-time in the line)")
    return p.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def ops_of(shapes):
    return float(sum(2 * m * n * k for m, n, k in shapes))


ROUTE_NAMES = {0: "table", 1: "popcount", 2: "skinny_dp4a", 3: "warp_mma", 4: "small_dp4a",
               5: "in_kernel_conversion", 6: "none", 7: "stream_mma"}


def route_name(route, param):
    """Name of a (route, param) kernel: the route, with the tile width of the
    in-kernel conversion kernel and the variant of the popcount kernel."""
    if route == 5:
        return f"{ROUTE_NAMES[route]}_{param}"
    if route == 1:
        return f"{ROUTE_NAMES[route]}_v{param}"
    return ROUTE_NAMES[route]


def route_histogram(L, shapes, times_ms=None, routes=None):
    """Shapes (and, given per-shape times, milliseconds) per kernel: of the
    given (route, param) list, else of the 8-bit shape rules (lbgemm_route)."""
    out = {}
    for i, (m, n, k) in enumerate(shapes):
        if routes is not None:
            name = route_name(*routes[i])
        else:
            route, tile = L.lbgemm_route(8, m, n, k)
            name = route_name(route, tile)
        e = out.setdefault(name, {"shapes": 0, "ms": 0.0})
        e["shapes"] += 1
        if times_ms is not None:
            e["ms"] += float(times_ms[i])
    if times_ms is None:
        for e in out.values():
            del e["ms"]
    return dict(sorted(out.items()))


def geomean(x) -> float:
    return float(np.exp(np.mean(np.log(np.asarray(x, dtype=np.float64)))))


def shape_roofline_ms(bits, shapes, peaks):
    """Per-shape roofline time (ms): the slower of the tensor pipe (sustained
    bf16 peak for 8-bit operands encoded as fp16; twice that, the fp8 rate,
    for 4- and 1-bit operands encoded as e4m3) and the HBM bytes of the
    operation (A and B read once in their own format, int32 C written once)."""
    rate = peaks["bf16_tflops_sustained"] * 1e12 * (1 if bits == 8 else 2)
    per_elem = {8: 1.0, 4: 0.5, 1: 0.125}[bits]
    return np.array([max(2.0 * m * n * k / rate,
                         (per_elem * (m * k + n * k) + 4.0 * m * n) / (peaks["hbm_gbs"] * 1e9))
                     for m, n, k in shapes]) * 1e3


def selection_summary(bits, shapes, recs, disp, T, sweep_seconds, peaks, reps):
    """Selected-vs-default figures of one bit width from the re-time T
    [shape, arm]: arms default, label, dispatch, default again."""
    d, t, s, d2 = T[:, 0], T[:, 1], T[:, 2], T[:, 3]
    ops = ops_of(shapes)
    noise = np.abs(d2 / d - 1.0)
    noise_p95 = float(np.percentile(noise, 95))
    speed, dspeed = d / t, d / s
    labels = [r["label"] for r in recs]
    picks = [tuple(r["pick"]) for r in recs]
    dv = 7
    t_roof = shape_roofline_ms(bits, shapes, peaks)
    summ = {
        "shapes": len(shapes),
        "what": f"{bits}-bit: labelled vs default (variant 7) tile x stage variant, both on the "
                "tensor-core kernel; dispatch_* = the kernel lbgemm_run runs (the table's pick "
                "among the nine variants and the shape-route kernels) vs variant 7",
        "retime": f"median of {reps} interleaved runs per arm and shape, L2 flushed before each",
        "label_ne_default": int(sum(v != dv for v in labels)),
        "pick_ne_default": int(sum(p != (ROUTE_TABLE, dv) for p in picks)),
        "noise_floor_p95": noise_p95,
        "noise_floor_max": float(noise.max()),
        "noise_floor_what": "|t2 / t1 - 1| between two interleaved re-times of the default "
                            "variant (the identical kernel)",
        "speedup_geomean": geomean(speed),
        "speedup_max": float(speed.max()),
        "speedup_min": float(speed.min()),
        "speedup_min_shape": list(shapes[int(np.argmin(speed))]),
        "shapes_slower_beyond_noise": int((speed < 1.0 - noise_p95).sum()),
        "shapes_slower_by_2pct": int((speed < 0.98).sum()),
        "dispatch_speedup_geomean": geomean(dspeed),
        "dispatch_speedup_max": float(dspeed.max()),
        "dispatch_speedup_min": float(dspeed.min()),
        "dispatch_speedup_min_shape": list(shapes[int(np.argmin(dspeed))]),
        "dispatch_slower_beyond_noise": int((dspeed < 1.0 - noise_p95).sum()),
        "dispatch_slower_by_2pct": int((dspeed < 0.98).sum()),
        "sweep_tops_default": ops / (d.sum() / 1e3) / 1e12,
        "sweep_tops_label": ops / (t.sum() / 1e3) / 1e12,
        "sweep_tops_dispatch": ops / (s.sum() / 1e3) / 1e12,
        "sweep_seconds": round(sweep_seconds, 1),
        "variant_histogram": [int(sum(v == i for v in labels)) for i in range(9)],
        "routes": route_histogram(None, shapes, s, disp),
    }
    roof = {"frac": float(t_roof.sum() / s.sum()),
            "roofline_tops": ops / (t_roof.sum() / 1e3) / 1e12,
            "definition": "sum over shapes of max(2MNK / tensor peak, operand and C bytes / HBM) "
                          "divided by the sum of the dispatch's re-timed medians; tensor peak = "
                          "sustained bf16 (8-bit, fp16 encoding) or twice it (4- and 1-bit, e4m3)"}
    if bits == 8:
        roof["frac_hbm_8tbs"] = float(np.sum([
            max(2.0 * m * n * k / (peaks["bf16_tflops_sustained"] * 1e12),
                (m * k + n * k + 4.0 * m * n) / 8.0e12) for m, n, k in shapes]) * 1e3 / s.sum())
    return summ, roof


def mlp_on_grid(L, bits, shapes, recs, sm):
    """The shipped selector network of this bit width judged on this run's own
    nine tensor-core medians of the grid shapes (None if none is shipped)."""
    path = os.path.join(ROOT, "bit_tensor_gemm_gb300", "data", f"mlp_gb300_s{bits}.txt")
    if not os.path.exists(path):
        return None
    L.lbgemm_mlp_load(path)  # (the library loads it by default too; grid shapes hit the table)
    T = np.array([r["ms"][:9] for r in recs])
    pred = np.array([L.lbgemm_mlp_predict(bits, m, n, k, sm) for (m, n, k) in shapes])
    best = T.argmin(axis=1)
    idx = np.arange(len(T))
    t_pred = T[idx, pred[:, 0]]
    t_top2 = np.minimum(T[idx, pred[:, 0]], T[idx, pred[:, 1]])
    srt = np.sort(T, axis=1)
    return {
        "network": "log2 M, log2 N, log2 K, SM count -> 3 x 128 ReLU -> 9 variants",
        "file": os.path.relpath(path, ROOT),
        "trained_on": f"bit_tensor_gemm_gb300/data/sweep_gb300_s{bits}.csv (random shapes; "
                      "the grid is held out)",
        "top1_accuracy": float(np.mean(pred[:, 0] == best)),
        "top2_accuracy": float(np.mean((pred[:, 0] == best) | (pred[:, 1] == best))),
        "top2_near_best": float(np.mean(t_top2 <= T.min(axis=1) * 1.02)),
        "within_2pct_of_best": float(np.mean(t_pred <= T.min(axis=1) * 1.02)),
        "best_two_within_2pct": float(np.mean(srt[:, 1] <= srt[:, 0] * 1.02)),
        "time_pred_over_best": float(t_pred.sum() / T.min(axis=1).sum()),
        "speedup_over_default": float(T[:, 7].sum() / t_pred.sum()),
    }


def max_over_ranks(x: float, device=None) -> float:
    """The largest x over all ranks (replicas time the same workload; the
    whole job takes as long as its slowest rank).  Identity without a
    process group."""
    import torch  # noqa: PLC0415
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(ops_per_step: float, steps: int, world: int, max_total_ms: float) -> float:
    """Whole-job throughput in TOPS: every rank runs the full workload (weak
    scaling), so the job does world x steps x ops in the slowest rank's time."""
    return ops_per_step * steps * world / (max_total_ms / 1e3) / 1e12


# ---- clocks during the timed region ------------------------------------------------

class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for i, nm in enumerate(self.REASONS):
                if len(r) > 5 + i and r[5 + i].strip() == "Active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---- the CPU oracle on a row sample (reference arm and cpu_baseline) --------------------

def oracle_sample(shapes, rows, A, B, threads):
    """Time the oracle on the first `rows` rows of C for every shape: (ops, seconds)."""
    import oracle  # noqa: PLC0415 -- the CPU baseline leg may run the oracle
    ops = 0.0
    t0 = time.perf_counter()
    for m, n, k in shapes:
        r = min(rows, m)
        oracle.gemm(8, A[: r * k].reshape(r, k), B[: n * k].reshape(n, k), k, threads=threads)
        ops += 2.0 * r * n * k
    return ops, time.perf_counter() - t0


def host_operands(seed):
    from bit_tensor_gemm_gb300 import synth  # noqa: PLC0415
    g = synth.rng(seed)
    A = synth.s8(g, MAXD, MAXD).reshape(-1)
    B = synth.s8(g, MAXD, MAXD).reshape(-1)
    return A, B


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle  # noqa: PLC0415
    from bit_tensor_gemm_gb300 import synth  # noqa: PLC0415
    shapes = SWEEP[: args.shapes] if args.shapes else SWEEP
    A, B = host_operands(synth.config_seed(2))
    threads = oracle.default_threads()
    rows = threads  # the oracle threads over rows of C: one row per thread
    for _ in range(args.warmup):
        oracle_sample(shapes, rows, A, B, threads)
    times, ops = [], 0.0
    for _ in range(args.steps):
        ops, dt = oracle_sample(shapes, rows, A, B, threads)
        times.append(dt)
    total = sum(times)
    value = ops * args.steps / total / 1e12
    sample = (f"first {rows} rows of C for each of the {len(shapes)} sweep shapes "
              f"({ops / 2:.3g} MACs per step)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "s8",
        "data": "synthetic",
        "config": {"workload": "int8_sweep_729", "shapes": len(shapes)},
        "cpu_baseline": {"value": value, "unit": "TOPS", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


# ---- our arm ---------------------------------------------------------------------------------

def source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_tensor_gemm_gb300", "csrc")
    for name in ("tc_gemm.cuh", "tc_pair.cuh", "ptx.cuh", "tc_params.h"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


TRAFFIC_FILE = os.path.join("profiles", "tc_traffic_int8_sweep.md")
TRAFFIC_SOURCE = (f"{TRAFFIC_FILE}: ncu dram__bytes_read.sum + dram__bytes_write.sum of single "
                  "launches of representative sweep shapes; each sweep shape takes the ratio "
                  "of DRAM bytes to the kernel's own operand and C bytes (fp16 A and B, int32 C) "
                  "of its nearest representative (sum of |log2| differences of M, N, K)")


def kernel_bytes(m, n, k):
    """Bytes the tensor-core GEMM kernel must move for one launch: fp16 A and
    B (the re-encoded operands) read once, int32 C written once."""
    return 2.0 * (m + n) * k + 4.0 * m * n


def profiled_traffic(shapes):
    """Per-launch DRAM bytes of the dominant kernel averaged over the sweep's
    launches, estimated from the committed single-launch ncu captures (when
    they were taken from the kernel source as it is now); else None."""
    import math  # noqa: PLC0415
    path = os.path.join(ROOT, TRAFFIC_FILE)
    if not os.path.exists(path):
        return None
    reps, src = [], None
    with open(path) as f:
        for line in f:
            w = line.split()
            if len(w) == 2 and w[0] == "source_sha256_16":
                src = w[1]
            elif len(w) == 6 and w[0] == "capture":
                m, n, k, dram = int(w[1]), int(w[2]), int(w[3]), float(w[5])
                reps.append((m, n, k, dram / kernel_bytes(m, n, k)))
    if src != source_hash() or not reps:
        return None
    total = 0.0
    for m, n, k in shapes:
        r = min(reps, key=lambda e: abs(math.log2(m / e[0])) + abs(math.log2(n / e[1])) +
                abs(math.log2(k / e[2])))
        total += r[3] * kernel_bytes(m, n, k)
    return total / len(shapes)


def run_ours(args):
    import torch  # noqa: PLC0415

    from bit_tensor_gemm_gb300 import build as bld  # noqa: PLC0415
    from bit_tensor_gemm_gb300 import lbgemm as L  # noqa: PLC0415
    from bit_tensor_gemm_gb300 import synth  # noqa: PLC0415
    from bit_tensor_gemm_gb300 import tune  # noqa: PLC0415

    rank, world, local = dist_env()
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    bld.build()
    L.load()
    peaks, peak_kind = load_peaks()
    shapes = SWEEP[: args.shapes] if args.shapes else SWEEP

    A_h, B_h = host_operands(synth.config_seed(2))
    A = torch.from_numpy(A_h).to(dev)
    B = torch.from_numpy(B_h).to(dev)
    C = torch.empty(MAXD * MAXD, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    dev_ops = {8: (A, B)}

    def operands_of(bits):
        """Device operands of a bit width's sweep (seeded; kept for the re-time)."""
        if bits not in dev_ops:
            dev_ops[bits] = tune.device_operands(bits, shapes, dev,
                                                 synth.config_seed(SEED_OF[bits]), with_c=False)
        return dev_ops[bits]

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()

    sm = torch.cuda.get_device_properties(dev).multi_processor_count

    # -- the sweep, per bit width: every candidate kernel per shape; the table
    #    keeps the label and the dispatch pick (tune.py) ---------------------------------------
    L.lbgemm_table_clear()
    recs, sweep_s, mlp_eval = {}, {}, {}
    if args.table:
        L.lbgemm_table_load(args.table)
    for bits in ([] if args.table else BITS):
        Ab, Bb = operands_of(bits)
        t0 = time.perf_counter()
        recs[bits] = tune.sweep(L, bits, shapes, Ab, Bb, C, sm, reps=args.sweep_reps,
                                confirm_reps=args.retime_reps)
        sweep_s[bits] = time.perf_counter() - t0
        mlp_eval[bits] = mlp_on_grid(L, bits, shapes, recs[bits], sm)
        del Ab, Bb

    def timed_pass(run_one, shp_list=shapes):
        """One pass: flush L2, event, GEMM, event, per shape.  Returns per-shape ms."""
        evs = []
        for shp in shp_list:
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run_one(*shp)
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    def sel(m, n, k):
        L.lbgemm_run(8, m, n, k, A, B, C)

    for _ in range(args.warmup):
        timed_pass(sel)
    barrier()
    clocks = Clocks(local)
    clocks.start()
    launches0 = L.lbgemm_launch_count()
    t_wall0 = time.perf_counter()
    step_ms = []
    torch.cuda.nvtx.range_push("timed")  # lets a profiler list the timed launches alone
    for _ in range(args.steps):
        step_ms.append(sum(timed_pass(sel)))
    barrier()
    torch.cuda.nvtx.range_pop()
    wall_s = time.perf_counter() - t_wall0
    launches = L.lbgemm_launch_count() - launches0
    clk = clocks.stop()
    L.lbgemm_device_status()
    total_ms = max_over_ranks(sum(step_ms), dev)
    ops_step = ops_of(shapes)
    value = job_value(ops_step, args.steps, world, total_ms)

    # -- selected vs default, on an independent re-time, interleaved --------------------------
    # The pages' comparison: the chosen tile x stage variant against the
    # default one, both forced on the tensor-core kernel.  Also the library's
    # full dispatch (which adds the shape rules) against the same default.
    # The pages' comparison: the labelled tile x stage variant against the
    # default one, both forced on the tensor-core kernel; and the library's
    # dispatch (the kernel lbgemm_run runs: the table's pick) against the same
    # default.  A second run of the default measures the noise floor: two
    # timings of the identical kernel.
    dv = (ROUTE_TABLE, L.lbgemm_default_variant())
    selection_by_bits, rooflines = {}, {}
    s_ms = None
    for bits in ([] if args.table else BITS):
        Ab, Bb = operands_of(bits)
        label = [(ROUTE_TABLE, r["label"]) for r in recs[bits]]
        disp = [tuple(L.lbgemm_dispatch_for(sm, bits, *sh)) for sh in shapes]
        T = tune.retime(L, bits, shapes, [[dv] * len(shapes), label, disp, [dv] * len(shapes)],
                        Ab, Bb, C, reps=args.retime_reps)
        summ, roof = selection_summary(bits, shapes, recs[bits], disp, T, sweep_s[bits], peaks,
                                       args.retime_reps)
        summ["mlp_selector"] = mlp_eval[bits]
        summ["sweep_roofline_frac"] = roof["frac"]
        if args.offgrid:
            # shapes the table does not hold: the kernel lbgemm_run picks there
            # (the shape rules, the network's variant) against every candidate
            shp = tune.random_shapes(args.offgrid, 2027 + bits)
            Ao, Bo, Co = tune.device_operands(bits, shp, dev, synth.config_seed(SEED_OF[bits]))
            summ["offgrid"] = tune.offgrid_check(L, bits, shp, Ao, Bo, Co, sm, reps=10)
            summ["offgrid"]["what"] = ("random shapes without a table entry (log-uniform in "
                                       "64-16384, at most 2^37 MACs): time of the kernel "
                                       "lbgemm_run picks over the fastest candidate, and of "
                                       "the default variant 7")
            del Ao, Bo, Co
        selection_by_bits[bits], rooflines[bits] = summ, roof
        if bits == 8:
            s_ms = T[:, 2]
        del Ab, Bb
    if args.table:
        selection = {"table": args.table, "note": "loaded, not measured in this run"}
        sweep_roofline = None
    else:
        selection = dict(selection_by_bits[8])
        selection["by_bits"] = {str(b): selection_by_bits[b] for b in BITS if b != 8}
        sweep_roofline = rooflines[8]

    # -- roofline of the dominant kernel: the variant-table tensor-core GEMM, on the
    #    shapes whose dispatch runs it (with the variant it runs), alone on encoded
    #    operands -------------------------------------------------------------------------
    encA = torch.empty(L.lbgemm_encoded_size(8, MAXD, MAXD), dtype=torch.uint8, device=dev)
    encB = torch.empty(L.lbgemm_encoded_size(8, MAXD, MAXD), dtype=torch.uint8, device=dev)
    tc_shapes = [(sh, prm) for sh in shapes
                 for rt, prm in [L.lbgemm_dispatch_for(sm, 8, *sh)] if rt == ROUTE_TABLE]
    enc_ms = []
    torch.cuda.nvtx.range_push("roofline")  # lets a profiler capture these launches alone
    for (m, n, k), v in tc_shapes:
        L.lbgemm_encode(8, m, k, A, encA)
        L.lbgemm_encode(8, n, k, B, encB)
        L.lbgemm_run_encoded(8, m, n, k, encA, encB, C, v)  # warm-up
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        L.lbgemm_run_encoded(8, m, n, k, encA, encB, C, v)
        e1.record(stream)
        e1.synchronize()
        enc_ms.append(e0.elapsed_time(e1))
    torch.cuda.nvtx.range_pop()
    tc_ops = ops_of([sh for sh, _ in tc_shapes])
    kernel_tflops = tc_ops / (sum(enc_ms) / 1e3) / 1e12
    # each launch is timed alone (L2 flushed, synchronised): the burst peak
    peak_tc = peaks["bf16_tflops"]
    alg_bytes = sum(m * k + n * k + 4.0 * m * n for (m, n, k), _ in tc_shapes) / len(tc_shapes)
    traffic = profiled_traffic([sh for sh, _ in tc_shapes])
    roofline = {"bound": "tensor", "achieved": kernel_tflops, "peak": peak_tc, "unit": "TFLOP/s",
                "frac": kernel_tflops / peak_tc, "traffic": traffic,
                "kernel": "tensor-core GEMM: tc_gemm_kernel (small and medium tiles) and "
                          "tc_pair_kernel (large tile, CTA pairs); int8 encoded as fp16, "
                          "tcgen05 kind::f16",
                "per": f"launch average over the {len(tc_shapes)} sweep shapes whose dispatch "
                       "runs this kernel (the variant it runs), each launch timed alone with CUDA "
                       "events after a warm-up call, L2 flushed before it",
                "peak_source": f"{peak_kind} bf16 dense, burst (launches timed alone)",
                "frac_of_sustained": kernel_tflops / peaks["bf16_tflops_sustained"],
                "algorithmic_bytes_per_launch": alg_bytes,
                "traffic_over_algorithmic": traffic / alg_bytes if traffic else None,
                "traffic_source": TRAFFIC_SOURCE if traffic else "no capture of the current "
                                                                 "kernel source"}
    del encA, encB

    # -- the other bit widths and the linear layer ------------------------------------------------
    def median_ms(fn, reps):
        ts = []
        for _ in range(reps):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        return float(np.median(ts))

    per_config = {}
    t = median_ms(lambda: L.lbgemm_run(8, 256, 256, 256, A, B, C), 20)
    per_config["int8_256x256x256"] = {"us": t * 1e3, "tops": 2 * 256 ** 3 / t / 1e9}
    for (m, n, k) in [(8192, 8192, 8192), (16384, 16384, 16384)]:
        t = median_ms(lambda: L.lbgemm_run(8, m, n, k, A, B, C), 3)
        per_config[f"int8_{m}x{n}x{k}"] = {"us": t * 1e3, "tops": 2 * m * n * k / t / 1e9}
    g4 = synth.rng(synth.config_seed(3))
    A4 = torch.from_numpy(synth.s4(g4, 8192, 8192)).to(dev)
    B4 = torch.from_numpy(synth.s4(g4, 8192, 8192)).to(dev)
    t = median_ms(lambda: L.lbgemm_run(4, 8192, 8192, 8192, A4, B4, C), 5)
    tops4 = 2 * 8192 ** 3 / t / 1e9
    per_config["int4_8192x8192x8192"] = {
        "us": t * 1e3, "tops": tops4,
        "frac_of_fp8_sustained": tops4 / (2 * peaks["bf16_tflops_sustained"])}
    del A4, B4
    g1 = synth.rng(synth.config_seed(4))
    A1 = torch.from_numpy(synth.b1(g1, 8192, 65536).view(np.int32)).to(dev)
    B1 = torch.from_numpy(synth.b1(g1, 8192, 65536).view(np.int32)).to(dev)
    ops1 = 2 * 8192 * 8192 * 65536
    t = median_ms(lambda: L.lbgemm_run(1, 8192, 8192, 65536, A1, B1, C), 3)
    clk_popc = Clocks(local)
    clk_popc.start()
    tp = median_ms(lambda: L.lbgemm_run_popc(8192, 8192, 65536, A1, B1, C), 3)
    popc_clk = clk_popc.stop()
    # ALU peak of the popcount route: 16 popcounts per clock per SM (the SM's
    # integer pipe), the device's SM count, the SM clock sampled while it ran
    popc_mhz = popc_clk.get("sm_mhz") or peaks.get("sm_max_mhz", 2070.0)
    popc_peak = sm * 16 * popc_mhz * 1e6 * 64 / 1e12
    per_config["b1_8192x8192x65536"] = {
        "us": t * 1e3, "tops": ops1 / t / 1e9, "route": "tensor cores (+-1 as e4m3)",
        "frac_of_fp8_sustained": ops1 / t / 1e9 / (2 * peaks["bf16_tflops_sustained"]),
        "popc_us": tp * 1e3, "popc_tops": ops1 / tp / 1e9,
        "popc_frac_of_alu_peak": ops1 / tp / 1e9 / popc_peak, "popc_alu_peak_tops": popc_peak,
        "popc_alu_peak_from": f"{sm} SMs x 16 popc/clk x {popc_mhz:.0f} MHz (median SM clock "
                              "sampled during the popcount runs) x 64 ops per 32-bit word"}
    del A1, B1
    # The linear layer (11008 x 4096 weights).  "us": one call alone, L2
    # flushed before it (median of 20); "b2b_us": calls back to back, each on
    # the next of six weight copies (270 MB, twice the L2), the way the layers
    # of a model follow one another; "default_us": the tensor-core default
    # variant 7 forced (the pages' section 4 compares the selected kernel with
    # a default template on a linear layer).
    NL, KL, COPIES = 11008, 4096, 6
    gw = synth.rng(synth.config_seed(5) + 7)
    W_copies = [torch.from_numpy(synth.s8(gw, NL, KL)).to(dev) for _ in range(COPIES)]
    sw_dev = torch.from_numpy((gw.random(NL, dtype=np.float32) + 0.5) / 127).to(dev)

    def b2b_us(call, n=60):
        for i in range(COPIES):
            call(W_copies[i])
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            call(W_copies[i % COPIES])
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / n * 1e3

    def linear_entry(M, byts, t, tb, td, route):
        return {"us": t * 1e3, "b2b_us": tb, "default_us": td * 1e3,
                "speedup_vs_default": td / t, "route": route,
                "tops": 2 * M * NL * KL / t / 1e9, "gbs": byts / t / 1e6,
                "frac_of_hbm": byts / t / 1e6 / peaks["hbm_gbs"],
                "frac_of_hbm_b2b": byts / tb / 1e3 / peaks["hbm_gbs"]}

    for M in (1, 16, 128, 2048):
        X, sx, W, sw = synth.linear_operands(M, NL, KL, synth.config_seed(5) + M)
        dX, dW = torch.from_numpy(X).to(dev), torch.from_numpy(W).to(dev)
        dsx, dsw = torch.from_numpy(sx).to(dev), torch.from_numpy(sw).to(dev)
        Y = torch.empty((M, NL), dtype=torch.bfloat16, device=dev)
        t = median_ms(lambda: L.lbgemm_linear(M, NL, KL, dX, dsx, dW, dsw, Y), 20)
        td = median_ms(lambda: L.lbgemm_linear_variant(M, NL, KL, dX, dsx, dW, dsw, Y,
                                                       L.lbgemm_default_variant()), 20)
        tb = b2b_us(lambda w: L.lbgemm_linear(M, NL, KL, dX, dsx, w, sw_dev, Y))
        byts = NL * KL + M * KL + 4 * (M + NL) + 2 * M * NL
        per_config[f"linear_M{M}_N11008_K4096"] = linear_entry(
            M, byts, t, tb, td, route_name(*L.lbgemm_route(8, M, NL, KL, linear=True)))
    # the linear layer on bf16 activations: per-token quantisation in front
    for M in (1, 16, 128, 2048):
        gq = np.random.default_rng(synth.config_seed(5) + 100 + M)
        Xf = torch.from_numpy(gq.standard_normal((M, KL), dtype=np.float32)).to(
            dev).to(torch.bfloat16)
        _, _, W, sw = synth.linear_operands(M, NL, KL, synth.config_seed(5) + M)
        dW, dsw = torch.from_numpy(W).to(dev), torch.from_numpy(sw).to(dev)
        Y = torch.empty((M, NL), dtype=torch.bfloat16, device=dev)
        t = median_ms(lambda: L.lbgemm_linear_quant(M, NL, KL, Xf, dW, dsw, Y), 20)
        tb = b2b_us(lambda w: L.lbgemm_linear_quant(M, NL, KL, Xf, w, sw_dev, Y))
        byts = NL * KL + 2 * M * KL + 4 * NL + 2 * M * NL
        per_config[f"linear_quant_M{M}_N11008_K4096"] = {
            "us": t * 1e3, "b2b_us": tb, "tops": 2 * M * NL * KL / t / 1e9, "gbs": byts / t / 1e6,
            "frac_of_hbm": byts / t / 1e6 / peaks["hbm_gbs"],
            "frac_of_hbm_b2b": byts / tb / 1e3 / peaks["hbm_gbs"]}
    del W_copies
    L.lbgemm_device_status()

    # -- end to end through the host-buffer entry point, on the balanced 81-shape ninth ----------
    A_pin = torch.from_numpy(A_h).pin_memory()
    B_pin = torch.from_numpy(B_h).pin_memory()
    C_pin = torch.empty(MAXD * MAXD, dtype=torch.int32).pin_memory()
    e2e_shapes = [s for s in E2E_SHAPES if s in set(shapes)] or shapes[:1]
    # one untimed pass first: the staging buffer grows to its final size and
    # the host pages and copy paths are warm, as for the timed steps' warm-up
    for (m, n, k) in e2e_shapes:
        L.lbgemm_run_host(8, m, n, k, A_pin, B_pin, C_pin, -1, stream)
    # E2E_PASSES timed passes, each call timed on the host clock; the median
    # pass is the value (a single pass once read 2.4x slower than its
    # neighbours on the same box), every pass is reported
    h2d = sum(m * k + n * k for m, n, k in e2e_shapes)
    d2h = sum(4 * m * n for m, n, k in e2e_shapes)
    e2e_ops = ops_of(e2e_shapes)
    pass_s = []
    for _ in range(E2E_PASSES):
        e2e_s = 0.0
        for (m, n, k) in e2e_shapes:
            t0 = time.perf_counter()
            L.lbgemm_run_host(8, m, n, k, A_pin, B_pin, C_pin, -1, stream)
            e2e_s += time.perf_counter() - t0
        pass_s.append(e2e_s)
    e2e_s = float(np.median(pass_s))
    dev_same = np.median(np.array([timed_pass(sel, e2e_shapes) for _ in range(2)]), axis=0)
    e2e = {"value": e2e_ops * world / e2e_s / 1e12, "unit": "TOPS",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "passes_tops": [round(e2e_ops * world / t / 1e12, 1) for t in pass_s],
           "shapes": f"{len(e2e_shapes)} of the sweep: every (M, N) pair once, each K nine times",
           "device_value_same_shapes": e2e_ops / (dev_same.sum() / 1e3) / 1e12,
           "entry": "lbgemm_run_host: pinned host buffers, copies and a sync inside the call; "
                    "one untimed pass over the shapes, then the median of "
                    f"{E2E_PASSES} timed passes"}
    del A_pin, B_pin, C_pin

    # -- the CPU oracle on a row sample -------------------------------------------------------------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle  # noqa: PLC0415
        threads = oracle.default_threads()
        _, dt1 = oracle_sample(shapes, threads, A_h, B_h, threads)
        rows = int(threads * max(1, min(8, round(15.0 / max(dt1, 1e-3)))))
        opsr, dtr = oracle_sample(shapes, rows, A_h, B_h, threads)
        cpu = {"value": opsr / dtr / 1e12, "unit": "TOPS", "cores": threads, "kind": "oracle",
               "sample": f"first {rows} rows of C for each of the {len(shapes)} sweep shapes "
                         f"({opsr / 2:.3g} MACs in {dtr:.1f} s)"}

    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_ms / args.steps, "wall_ms_per_step": wall_s * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "s8",
            "data": "synthetic",
            "config": {"workload": "int8_sweep_729", "shapes": len(shapes),
                       "sizes": "M, N, K each in {64, 128, ..., 16384}",
                       "values": f"uniform [-127, 127], seed {synth.config_seed(2)}",
                       "l2": "flushed (256 MB write) before every GEMM, outside the timed events",
                       "timing": "sum of per-GEMM CUDA-event times on the launching stream",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "clocks": clk, "gpu_launches": launches, "e2e": e2e, "roofline": roofline,
            "cpu_baseline": cpu, "selection": selection,
            "sweep_roofline": sweep_roofline,
            "per_config": per_config,
        }), flush=True)
        if args.dump:
            with open(args.dump, "w") as f:
                json.dump({"shapes": shapes, "sm_count": sm,
                           "records": {str(b): r for b, r in recs.items()},
                           "dispatch_ms_8bit": None if s_ms is None else s_ms.tolist(),
                           "kernel_only_ms": enc_ms}, f)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
