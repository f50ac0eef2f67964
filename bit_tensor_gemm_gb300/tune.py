"""Per-shape kernel selection on this GPU, and the table it writes.

Method: "Leveraging Large-Scale Data for Efficient Low-Bit CUTLASS GEMM
Optimization via Neural Networks" (press summary page).  Section 2: every
(M, N, K) sample is timed under all nine tile x stage templates and labelled
with the fastest; the intro and section 3: the selection happens per (M, N,
K, SM count) at run time; section 4: the selected template is compared with a
default one.  Here the timed candidates are the nine tensor-core variants
plus the library's shape-route kernels that can run the shape
(lbgemm_candidates), so the default dispatch itself is chosen by measurement.

For each shape:
  1. every candidate runs `reps` times, interleaved, L2 flushed before each
     run, and keeps its median (lbgemm_time_candidates);
  2. the label is lbgemm_choose over the nine tensor-core medians (the
     fastest variant, the default kept when within `keep`);
  3. the dispatch pick is the fastest candidate, unless the default variant
     is within `keep` of it (lbgemm_choose_candidate);
  4. a label or pick other than the default must win again against the
     default head to head, in `confirm_reps` fresh interleaved runs, by more
     than `keep`, or the default takes its place;
where keep = max(2 %, 1 us / fastest median) -- event timings resolve about
a microsecond.  The entry (label, route, param) goes into the library's
table (lbgemm_table_set_choice_for).

    python -m bit_tensor_gemm_gb300.tune --bits 8 4 1 --reps 20 \
        --out bit_tensor_gemm_gb300/data/lbgemm_table_gb300.txt

writes the table file that the library loads by default, and one CSV of the
nine tensor-core medians per bit width (the selector network's grid data).

    python -m bit_tensor_gemm_gb300.tune --bits 8 4 1 --offgrid 300 --out unused

judges the loaded table's fallback on random shapes it does not hold.
"""
from __future__ import annotations

import argparse
import os
import sys
import time

import numpy as np

SIZES = [64, 128, 256, 512, 1024, 2048, 4096, 8192, 16384]
GRID = [(m, n, k) for m in SIZES for n in SIZES for k in SIZES]
DEFAULT = 7
ROUTE_TABLE = 0
KEEP_REL = 0.02
KEEP_ABS_MS = 0.001


def keep_margin(t_fast_ms: float) -> float:
    """Relative margin a candidate must beat the default by."""
    return max(KEEP_REL, KEEP_ABS_MS / max(t_fast_ms, 1e-6))


def row_bytes(bits: int, k: int) -> int:
    return k if bits == 8 else k // 2 if bits == 4 else k // 8


def device_operands(bits: int, shapes, dev, seed: int, with_c: bool = True):
    """Seeded operands large enough for every shape (rows of the largest K),
    and (with_c) C for the largest M x N.  Uniform codes as in the synthetic
    workloads."""
    import torch  # noqa: PLC0415  (device memory only)

    from . import synth  # noqa: PLC0415
    g = synth.rng(seed)
    ra = max(m * row_bytes(bits, k) for m, n, k in shapes)
    rb = max(n * row_bytes(bits, k) for m, n, k in shapes)
    if bits == 8:
        a, b = synth.s8(g, 1, ra), synth.s8(g, 1, rb)
    elif bits == 4:  # ra bytes = 2 ra nibbles
        a, b = synth.s4(g, 1, 2 * ra), synth.s4(g, 1, 2 * rb)
    else:  # ra bytes = 8 ra bits (K is a multiple of 32, so ra of 4)
        a, b = synth.b1(g, 1, 8 * ra), synth.b1(g, 1, 8 * rb)
    A = torch.from_numpy(np.ascontiguousarray(a).reshape(-1).view(np.int8)).to(dev)
    B = torch.from_numpy(np.ascontiguousarray(b).reshape(-1).view(np.int8)).to(dev)
    if not with_c:
        return A, B
    C = torch.empty(max(m * n for m, n, k in shapes), dtype=torch.int32, device=dev)
    return A, B, C


def select_shape(L, bits, m, n, k, A, B, C, reps=10, confirm_reps=20):
    """Steps 1-4 for one shape.  Returns a record with the candidates, their
    medians, the label and the pick."""
    cands = L.lbgemm_candidates(bits, m, n, k)
    t = L.lbgemm_time_candidates(bits, m, n, k, A, B, C, cands, warmup=1, reps=reps,
                                 flush_l2=True)
    keep = keep_margin(min(t))
    label = L.lbgemm_choose(t[:9], DEFAULT, keep)
    best = L.lbgemm_choose_candidate(t, DEFAULT, keep)
    if label < 0 or best < 0:
        raise RuntimeError(f"{bits}-bit {m}x{n}x{k}: unusable timings {t}")
    pick = tuple(cands[best])
    confirmed = {}

    def wins(c):
        if c == (ROUTE_TABLE, DEFAULT):
            return True
        if c not in confirmed:
            h = L.lbgemm_time_candidates(bits, m, n, k, A, B, C, [c, (ROUTE_TABLE, DEFAULT)],
                                         warmup=1, reps=confirm_reps, flush_l2=True)
            confirmed[c] = (L.lbgemm_choose_candidate(h, 1, keep_margin(min(h))) == 0, h)
        return confirmed[c][0]

    if not wins((ROUTE_TABLE, label)):
        label = DEFAULT
    if not wins(tuple(pick)):
        pick = (ROUTE_TABLE, DEFAULT)
    return {"shape": (m, n, k), "candidates": [list(c) for c in cands], "ms": list(map(float, t)),
            "label": int(label), "pick": [int(pick[0]), int(pick[1])],
            "confirm": {f"{c[0]}:{c[1]}": [bool(v[0])] + [float(x) for x in v[1]]
                        for c, v in confirmed.items()}}


def sweep(L, bits, shapes, A, B, C, sm_count, reps=10, confirm_reps=20, log=None):
    """Select every shape and store the entries in the library's table."""
    recs = []
    t0 = time.perf_counter()
    for i, (m, n, k) in enumerate(shapes):
        r = select_shape(L, bits, m, n, k, A, B, C, reps, confirm_reps)
        L.lbgemm_table_set_choice_for(sm_count, bits, m, n, k, r["label"], *r["pick"])
        recs.append(r)
        if log and i % 100 == 99:
            print(f"{bits}-bit: {i + 1}/{len(shapes)} shapes, {time.perf_counter() - t0:.0f} s",
                  file=log, flush=True)
    return recs


def retime(L, bits, shapes, arms, A, B, C, reps=20):
    """Interleaved re-time of several candidates per shape: arms is a list of
    per-shape (route, param) lists; returns an array [shape, arm] of medians."""
    out = np.zeros((len(shapes), len(arms)))
    for i, (m, n, k) in enumerate(shapes):
        cands = [arm[i] for arm in arms]
        out[i] = L.lbgemm_time_candidates(bits, m, n, k, A, B, C, cands, warmup=1, reps=reps,
                                          flush_l2=True)
    return out


def random_shapes(count, seed, max_work=2.0 ** 37):
    """Log-uniform shapes in [64, 16384] per dimension, multiples of 16 (32
    along K), at most max_work MACs: shapes the grid table does not hold."""
    g = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        m, n, k = (int(round(2 ** g.uniform(6, 14))) for _ in range(3))
        m, n, k = max(16, m // 16 * 16), max(16, n // 16 * 16), max(32, k // 32 * 32)
        if float(m) * n * k <= max_work and (m, n, k) not in GRID:
            out.append((m, n, k))
    return out


def offgrid_check(L, bits, shapes, A, B, C, sm_count, reps=10):
    """How the dispatch does on shapes without a table entry: every candidate
    timed per shape; the time of the kernel lbgemm_run picks (the shape rules,
    with the selector network's variant on the tensor-core route) against the
    fastest candidate and the default variant."""
    t_pick = t_best = t_default = 0.0
    over = 0
    for m, n, k in shapes:
        cands = L.lbgemm_candidates(bits, m, n, k)
        t = L.lbgemm_time_candidates(bits, m, n, k, A, B, C, cands, warmup=1, reps=reps,
                                     flush_l2=True)
        pick = tuple(L.lbgemm_dispatch_for(sm_count, bits, m, n, k))
        tp = t[cands.index(pick)] if pick in cands else t[DEFAULT]
        t_pick += tp
        t_best += min(t)
        t_default += t[DEFAULT]
        over += tp > min(t) * 1.10
    return {"shapes": len(shapes), "pick_over_best": t_pick / t_best,
            "default_over_best": t_default / t_best, "pick_speedup_over_default": t_default / t_pick,
            "shapes_over_best_by_10pct": over}


def write_grid_csv(path, bits, recs, sm_count):
    """The nine tensor-core medians per shape (the selector network's data)."""
    with open(path, "w") as f:
        f.write("M,N,K,sm_count," + ",".join(f"t{v}" for v in range(9)) + "\n")
        for r in recs:
            m, n, k = r["shape"]
            f.write(f"{m},{n},{k},{sm_count}," + ",".join(f"{x:.5f}" for x in r["ms"][:9]) + "\n")


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--bits", type=int, nargs="+", default=[8, 4, 1], choices=(8, 4, 1))
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--confirm-reps", type=int, default=20)
    ap.add_argument("--out", required=True, help="table file to write")
    ap.add_argument("--csv-dir", default="", help="write grid_<gpu>_s<bits>.csv here")
    ap.add_argument("--dump", default="", help="write every record (JSON) here")
    ap.add_argument("--shapes", type=int, default=0, help="debug: only the first N grid shapes")
    ap.add_argument("--merge", action="store_true",
                    help="keep the loaded table's entries of the bit widths not swept")
    ap.add_argument("--offgrid", type=int, default=0, metavar="COUNT",
                    help="instead of tuning: judge the dispatch on COUNT random shapes the "
                         "loaded table does not hold (prints one JSON line per bit width)")
    a = ap.parse_args(argv)
    import json  # noqa: PLC0415

    import torch  # noqa: PLC0415  (device memory only)

    from . import build as bld  # noqa: PLC0415
    from . import lbgemm as L  # noqa: PLC0415
    from . import synth  # noqa: PLC0415
    bld.build()
    L.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    sm = torch.cuda.get_device_properties(dev).multi_processor_count
    shapes = GRID[: a.shapes] if a.shapes else GRID
    if a.offgrid:
        for bits in a.bits:
            shp = random_shapes(a.offgrid, 2027 + bits)
            A, B, C = device_operands(bits, shp, dev,
                                      synth.config_seed({8: 2, 4: 3, 1: 4}[bits]))
            print(json.dumps({"bits": bits, **offgrid_check(L, bits, shp, A, B, C, sm)}),
                  flush=True)
            del A, B, C
        L.lbgemm_device_status()
        return 0
    if not a.merge:
        L.lbgemm_table_clear()
    dump = {}
    for bits in a.bits:
        A, B, C = device_operands(bits, shapes, dev, synth.config_seed({8: 2, 4: 3, 1: 4}[bits]))
        recs = sweep(L, bits, shapes, A, B, C, sm, a.reps, a.confirm_reps, log=sys.stderr)
        dump[bits] = recs
        if a.csv_dir:
            write_grid_csv(os.path.join(a.csv_dir, f"grid_gb300_s{bits}.csv"), bits, recs, sm)
        del A, B, C
        torch.cuda.empty_cache()
    L.lbgemm_device_status()
    L.lbgemm_table_save(a.out)
    if a.dump:
        with open(a.dump, "w") as f:
            json.dump({"sm_count": sm, "records": dump}, f)
    return 0


if __name__ == "__main__":
    sys.exit(main())
