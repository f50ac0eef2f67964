#!/usr/bin/env python
"""Benchmark of the low-bit GEMM library on GB300.

Workload (one step): the 8-bit GEMM shape sweep -- M, N, K each in
{64, 128, ..., 16384}, 729 shapes, operands uniform in [-127, 127] -- run once
per shape through lbgemm_run with the variant the selection table picked.
Before the timed steps the sweep itself runs: every shape is timed under all
nine tile x stage variants (lbgemm_time_variants) and the table stores
lbgemm_choose's pick, once a pick other than the default has won again head
to head against it.  L2 is flushed before every GEMM, outside the timed
intervals; the step time is the sum of the per-GEMM CUDA-event times.

value = sum over the 729 shapes of 2*M*N*K / step time, in TOPS (integer
operations, 2 per multiply-add).  The same line reports the selected-vs-
default speedups, the other bit widths and the linear layer, the roofline of
the dominant kernel, an end-to-end number through the host-buffer entry
point, and the CPU oracle on a row sample.

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
METRIC = "int8 GEMM TOPS over the 729-shape sweep (selected variant)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--sweep-reps", type=int, default=5)
    p.add_argument("--shapes", type=int, default=0, help="debug: use only the first N shapes")
    p.add_argument("--no-cpu", action="store_true", help="debug: skip the CPU oracle sample")
    p.add_argument("--dump", default="", help="write per-shape sweep data (JSON) to this path")
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
               5: "in_kernel_conversion", 6: "none"}


def route_histogram(L, shapes, times_ms=None):
    """Shapes (and, given per-shape times, milliseconds) per kernel of the
    library's 8-bit default dispatch (lbgemm_route)."""
    out = {}
    for i, (m, n, k) in enumerate(shapes):
        route, tile = L.lbgemm_route(8, m, n, k)
        name = ROUTE_NAMES[route] + (f"_{tile}" if tile else "")
        e = out.setdefault(name, {"shapes": 0, "ms": 0.0})
        e["shapes"] += 1
        if times_ms is not None:
            e["ms"] += float(times_ms[i])
    if times_ms is None:
        for e in out.values():
            del e["ms"]
    return dict(sorted(out.items()))


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


def profiled_traffic():
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu summary,
    when it was taken from the kernel source as it is now; else None."""
    path = os.path.join(ROOT, "profiles", "tc_gemm_int8_sweep.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("source_sha256_16") != source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def run_ours(args):
    import torch  # noqa: PLC0415

    from bit_tensor_gemm_gb300 import build as bld  # noqa: PLC0415
    from bit_tensor_gemm_gb300 import lbgemm as L  # noqa: PLC0415
    from bit_tensor_gemm_gb300 import synth  # noqa: PLC0415

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

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()

    def beats_default(m, n, k, v, keep, reps=5):
        """Variant v against the default, interleaved, L2 flushed before each
        run: is v's median faster by more than `keep` (relative)?"""
        dv = L.lbgemm_default_variant()
        pairs = []
        for _ in range(reps):
            for var in (v, dv):
                flush.zero_()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                L.lbgemm_run_variant(8, m, n, k, A, B, C, var)
                e1.record(stream)
                pairs.append((var, e0, e1))
        torch.cuda.synchronize()
        tv = np.median([a.elapsed_time(b) for var, a, b in pairs if var == v])
        td = np.median([a.elapsed_time(b) for var, a, b in pairs if var == dv])
        return tv < td * (1.0 - keep)

    # -- the sweep: nine variants per shape; the table keeps lbgemm_choose's pick ------------
    t_sweep0 = time.perf_counter()
    L.lbgemm_table_clear()
    sweep_times = []
    for (m, n, k) in shapes:
        t = L.lbgemm_time_variants(8, m, n, k, A, B, C, warmup=1, reps=args.sweep_reps,
                                   flush_l2=True)
        sweep_times.append(t)
        # keep the default unless another variant is faster by more than 2 %
        # and by more than 2 us, the resolution of the event timings
        keep = max(0.02, 0.002 / max(min(t), 1e-6))
        v = L.lbgemm_choose(t, L.lbgemm_default_variant(), keep)
        # a pick other than the default must win again head to head, in fresh
        # interleaved timings, or the default stays: one noisy sweep sample
        # must not make a shape slower than the default tile
        if v != L.lbgemm_default_variant() and not beats_default(m, n, k, v, keep):
            v = L.lbgemm_default_variant()
        L.lbgemm_table_set(8, m, n, k, v)
    sweep_s = time.perf_counter() - t_sweep0

    # -- the learned selector (trained offline on a separate random-shape GB300
    #    sweep) judged on this run's own timings of the 729 grid shapes --------------------
    mlp_eval = None
    mlp_path = os.path.join(ROOT, "bit_tensor_gemm_gb300", "data", "mlp_gb300_s8.txt")
    if os.path.exists(mlp_path):
        L.lbgemm_mlp_load(mlp_path)
        sm = torch.cuda.get_device_properties(dev).multi_processor_count
        T = np.array(sweep_times)
        pred = np.array([L.lbgemm_mlp_predict(8, m, n, k, sm) for (m, n, k) in shapes])
        best = T.argmin(axis=1)
        t_pred = T[np.arange(len(T)), pred[:, 0]]
        mlp_eval = {
            "network": "log2 M, log2 N, log2 K, SM count -> 3 x 128 ReLU -> 9 variants",
            "trained_on": "bit_tensor_gemm_gb300/data/sweep_gb300_s8.csv (3000 random shapes)",
            "top1_accuracy": float(np.mean(pred[:, 0] == best)),
            "top2_accuracy": float(np.mean((pred[:, 0] == best) | (pred[:, 1] == best))),
            "within_2pct_of_best": float(np.mean(t_pred <= T.min(axis=1) * 1.02)),
            "time_pred_over_best": float(t_pred.sum() / T.min(axis=1).sum()),
            "speedup_over_default": float(T[:, 7].sum() / t_pred.sum()),
        }
        L.lbgemm_mlp_clear()  # the timed steps use the measured table

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

    def dflt(m, n, k):
        L.lbgemm_run_variant(8, m, n, k, A, B, C, L.lbgemm_default_variant())

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
    chosen = [L.lbgemm_select(8, *s) for s in shapes]
    chosen_of = dict(zip(shapes, chosen))

    def sel_tc(m, n, k):
        L.lbgemm_run_variant(8, m, n, k, A, B, C, chosen_of[(m, n, k)])

    d_runs, t_runs, s_runs = [], [], []
    for _ in range(3):
        d_runs.append(timed_pass(dflt))
        t_runs.append(timed_pass(sel_tc))
        s_runs.append(timed_pass(sel))
    d_ms = np.median(np.array(d_runs), axis=0)
    t_ms = np.median(np.array(t_runs), axis=0)
    s_ms = np.median(np.array(s_runs), axis=0)
    # a shape whose chosen variant is the default runs the identical kernel:
    # its ratio is 1 by definition, not the noise between two timings
    same = np.array([c == L.lbgemm_default_variant() for c in chosen])
    speed = np.where(same, 1.0, d_ms / t_ms)
    dspeed = d_ms / s_ms
    # Per-shape roofline: the slower of the tensor pipe and the HBM bytes of
    # the operation (int8 A and B read once, int32 C written once).
    t_roof = np.array([max(2.0 * m * n * k / (peaks["bf16_tflops_sustained"] * 1e12),
                           (m * k + n * k + 4.0 * m * n) / (peaks["hbm_gbs"] * 1e9))
                       for m, n, k in shapes])
    t_roof8 = np.array([max(2.0 * m * n * k / (peaks["bf16_tflops_sustained"] * 1e12),
                            (m * k + n * k + 4.0 * m * n) / 8.0e12) for m, n, k in shapes])
    sweep_roofline = {
        "frac": float(t_roof.sum() / (s_ms.sum() / 1e3)),
        "frac_hbm_8tbs": float(t_roof8.sum() / (s_ms.sum() / 1e3)),
        "roofline_tops": ops_step / t_roof.sum() / 1e12,
        "definition": "sum over shapes of max(2MNK / sustained bf16 peak, (MK+NK+4MN) bytes / "
                      "HBM) divided by the sum of measured times (selected variants)"}
    worst = int(np.argmin(speed))
    selection = {
        "shapes": len(shapes),
        "selected_ne_default": int(sum(v != L.lbgemm_default_variant() for v in chosen)),
        "what": "chosen vs default (variant 7) tile x stage variant, both on the tensor-core "
                "kernel; dispatch_* adds the shape rules (lbgemm_run vs variant 7)",
        "speedup_geomean": float(np.exp(np.mean(np.log(speed)))),
        "speedup_max": float(speed.max()),
        "speedup_min": float(speed.min()),
        "speedup_min_shape": list(shapes[worst]),
        "shapes_slower_than_default_by_2pct": int((speed < 0.98).sum()),
        "dispatch_speedup_geomean": float(np.exp(np.mean(np.log(dspeed)))),
        "dispatch_speedup_max": float(dspeed.max()),
        "dispatch_speedup_min": float(dspeed.min()),
        "sweep_tops_default": ops_step / (d_ms.sum() / 1e3) / 1e12,
        "sweep_tops_chosen_variant": ops_step / (t_ms.sum() / 1e3) / 1e12,
        "sweep_tops_dispatch": ops_step / (s_ms.sum() / 1e3) / 1e12,
        "sweep_seconds": round(sweep_s, 1),
        "variant_histogram": [int(sum(v == i for v in chosen)) for i in range(9)],
        "routes": route_histogram(L, shapes, s_ms),
    }

    # -- roofline of the dominant kernel: the tensor-core GEMM alone on encoded operands ------
    encA = torch.empty(L.lbgemm_encoded_size(8, MAXD, MAXD), dtype=torch.uint8, device=dev)
    encB = torch.empty(L.lbgemm_encoded_size(8, MAXD, MAXD), dtype=torch.uint8, device=dev)
    enc_ms = []
    torch.cuda.nvtx.range_push("roofline")  # lets a profiler capture these launches alone
    for (m, n, k) in shapes:
        L.lbgemm_encode(8, m, k, A, encA)
        L.lbgemm_encode(8, n, k, B, encB)
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        L.lbgemm_run_encoded(8, m, n, k, encA, encB, C)
        e1.record(stream)
        e1.synchronize()
        enc_ms.append(e0.elapsed_time(e1))
    torch.cuda.nvtx.range_pop()
    kernel_tflops = ops_step / (sum(enc_ms) / 1e3) / 1e12
    peak_tc = peaks["bf16_tflops_sustained"]
    roofline = {"bound": "tensor", "achieved": kernel_tflops, "peak": peak_tc, "unit": "TFLOP/s",
                "frac": kernel_tflops / peak_tc, "traffic": profiled_traffic(),
                "kernel": "tensor-core GEMM: tc_gemm_kernel (small and medium tiles) and "
                          "tc_pair_kernel (large tile, CTA pairs); int8 encoded as fp16, "
                          "tcgen05 kind::f16",
                "per": "launch average over the sweep's 729 launches (selected variants)",
                "peak_source": f"{peak_kind} bf16 dense, sustained",
                "frac_of_burst": kernel_tflops / peaks["bf16_tflops"]}
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
    tp = median_ms(lambda: L.lbgemm_run_popc(8192, 8192, 65536, A1, B1, C), 3)
    popc_peak = 152 * 16 * peaks.get("sm_max_mhz", 2070.0) * 1e6 * 64 / 1e12
    per_config["b1_8192x8192x65536"] = {
        "us": t * 1e3, "tops": ops1 / t / 1e9, "route": "tensor cores (+-1 as e4m3)",
        "frac_of_fp8_sustained": ops1 / t / 1e9 / (2 * peaks["bf16_tflops_sustained"]),
        "popc_us": tp * 1e3, "popc_tops": ops1 / tp / 1e9,
        "popc_frac_of_alu_peak": ops1 / tp / 1e9 / popc_peak, "popc_alu_peak_tops": popc_peak}
    del A1, B1
    for M in (1, 16, 128, 2048):
        X, sx, W, sw = synth.linear_operands(M, 11008, 4096, synth.config_seed(5) + M)
        dX, dW = torch.from_numpy(X).to(dev), torch.from_numpy(W).to(dev)
        dsx, dsw = torch.from_numpy(sx).to(dev), torch.from_numpy(sw).to(dev)
        Y = torch.empty((M, 11008), dtype=torch.bfloat16, device=dev)
        t = median_ms(lambda: L.lbgemm_linear(M, 11008, 4096, dX, dsx, dW, dsw, Y), 20)
        byts = 11008 * 4096 + M * 4096 + 4 * (M + 11008) + 2 * M * 11008
        per_config[f"linear_M{M}_N11008_K4096"] = {
            "us": t * 1e3, "tops": 2 * M * 11008 * 4096 / t / 1e9, "gbs": byts / t / 1e6,
            "frac_of_hbm": byts / t / 1e6 / peaks["hbm_gbs"]}
    # the linear layer on bf16 activations: per-token quantisation in front
    for M in (1, 16, 128, 2048):
        gq = np.random.default_rng(synth.config_seed(5) + 100 + M)
        Xf = torch.from_numpy(gq.standard_normal((M, 4096), dtype=np.float32)).to(
            dev).to(torch.bfloat16)
        _, _, W, sw = synth.linear_operands(M, 11008, 4096, synth.config_seed(5) + M)
        dW, dsw = torch.from_numpy(W).to(dev), torch.from_numpy(sw).to(dev)
        Y = torch.empty((M, 11008), dtype=torch.bfloat16, device=dev)
        t = median_ms(lambda: L.lbgemm_linear_quant(M, 11008, 4096, Xf, dW, dsw, Y), 20)
        byts = 11008 * 4096 + 2 * M * 4096 + 4 * 11008 + 2 * M * 11008
        per_config[f"linear_quant_M{M}_N11008_K4096"] = {
            "us": t * 1e3, "tops": 2 * M * 11008 * 4096 / t / 1e9, "gbs": byts / t / 1e6,
            "frac_of_hbm": byts / t / 1e6 / peaks["hbm_gbs"]}
    L.lbgemm_device_status()

    # -- end to end through the host-buffer entry point, on the balanced 81-shape ninth ----------
    A_pin = torch.from_numpy(A_h).pin_memory()
    B_pin = torch.from_numpy(B_h).pin_memory()
    C_pin = torch.empty(MAXD * MAXD, dtype=torch.int32).pin_memory()
    e2e_shapes = [s for s in E2E_SHAPES if s in set(shapes)] or shapes[:1]
    L.lbgemm_run_host(8, 256, 256, 256, A_pin, B_pin, C_pin, -1, stream)
    e2e_s, h2d, d2h = 0.0, 0, 0
    for (m, n, k) in e2e_shapes:
        t0 = time.perf_counter()
        L.lbgemm_run_host(8, m, n, k, A_pin, B_pin, C_pin, -1, stream)
        e2e_s += time.perf_counter() - t0
        h2d += m * k + n * k
        d2h += 4 * m * n
    dev_same = np.median(np.array([timed_pass(sel, e2e_shapes) for _ in range(2)]), axis=0)
    e2e_ops = ops_of(e2e_shapes)
    e2e = {"value": e2e_ops * world / e2e_s / 1e12, "unit": "TOPS",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "shapes": f"{len(e2e_shapes)} of the sweep: every (M, N) pair once, each K nine times",
           "device_value_same_shapes": e2e_ops / (dev_same.sum() / 1e3) / 1e12,
           "entry": "lbgemm_run_host: pinned host buffers, copies and a sync inside the call"}
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
            "cpu_baseline": cpu, "selection": selection, "mlp_selector": mlp_eval,
            "sweep_roofline": sweep_roofline,
            "per_config": per_config,
        }), flush=True)
        if args.dump:
            with open(args.dump, "w") as f:
                json.dump({"shapes": shapes, "variant_times_ms": sweep_times, "chosen": chosen,
                           "selected_ms": s_ms.tolist(), "default_ms": d_ms.tolist(),
                           "chosen_variant_ms": t_ms.tolist(),
                           "kernel_only_ms": enc_ms, "roofline_ms": (t_roof * 1e3).tolist(),
                           "sm_count": None}, f)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
