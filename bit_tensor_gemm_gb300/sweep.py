"""The timing sweep that builds the selector's dataset.

Method: "Leveraging Large-Scale Data for Efficient Low-Bit CUTLASS GEMM
Optimization via Neural Networks" (press summary page), section 2: every
(M, N, K) sample is timed under all nine templates and labelled with the
fastest.  Here each sample is timed on this GPU through lbgemm_time_variants
(the L2 is flushed before every timed run, the variants interleaved) and
written as one CSV row:
    M,N,K,sm_count,t0,...,t8     (median milliseconds per variant)

    python -m bit_tensor_gemm_gb300.sweep --bits 8 --out data.csv [--count 1500] [--seed 7]

Shapes are drawn log-uniformly in [64, 16384] per dimension (seeded; K a
multiple of 16, of 32 for 1-bit), keeping M*N*K <= 2^37 so the sweep ends in
minutes.  Every drawn shape is kept, the ones the library's shape rules send
to other kernels included: the label is the tensor-core tile x stage choice,
which the dispatch uses wherever the variant table runs.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np


def shapes(count: int, seed: int, max_work: float = 2.0 ** 37, k_multiple: int = 16):
    g = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        m, n, k = (int(round(2 ** g.uniform(6, 14))) for _ in range(3))
        m, n = (max(16, (x // 16) * 16) for x in (m, n))
        k = max(k_multiple, (k // k_multiple) * k_multiple)
        if float(m) * n * k > max_work:
            continue
        out.append((m, n, k))
    return out


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--out", required=True)
    ap.add_argument("--bits", type=int, default=8, choices=(8, 4, 1))
    ap.add_argument("--count", type=int, default=1500)
    ap.add_argument("--seed", type=int, default=7)
    ap.add_argument("--reps", type=int, default=5)
    a = ap.parse_args(argv)
    import torch  # noqa: PLC0415  (device memory only)

    from . import build as bld  # noqa: PLC0415
    from . import lbgemm as L  # noqa: PLC0415
    bld.build()
    L.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    sm = torch.cuda.get_device_properties(dev).multi_processor_count
    shp = shapes(a.count, a.seed, k_multiple=32 if a.bits == 1 else 16)
    from . import synth, tune  # noqa: PLC0415
    A, B, C = tune.device_operands(a.bits, shp, dev, synth.config_seed({8: 2, 4: 3, 1: 4}[a.bits]))
    with open(a.out, "w") as f:
        f.write("M,N,K,sm_count," + ",".join(f"t{v}" for v in range(9)) + "\n")
        for i, (m, n, k) in enumerate(shp):
            t = L.lbgemm_time_variants(a.bits, m, n, k, A, B, C, warmup=1, reps=a.reps,
                                       flush_l2=True)
            f.write(f"{m},{n},{k},{sm}," + ",".join(f"{x:.5f}" for x in t) + "\n")
            if i % 200 == 0:
                print(f"{i}/{len(shp)}", file=sys.stderr, flush=True)
    L.lbgemm_device_status()
    return 0


if __name__ == "__main__":
    sys.exit(main())
