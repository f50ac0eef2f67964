"""Run one GEMM (or linear layer) through the C ABI on seeded random operands.

A command-line tool for profiling one kernel in isolation: it draws the
operands (uniform codes, as in the library's synthetic workloads), makes
`--reps` calls and prints the CUDA-event time of each.  Nothing is checked
against a reference here; the tests do that.

    python -m bit_tensor_gemm_gb300.run_gemm --bits 8 -M 8192 -N 8192 -K 8192 \
        [--variant 7] [--encoded] [--linear] [--reps 2]

--variant forces a tile x stage variant of the tensor-core kernel
(lbgemm_run_variant); --fused forces the kernel that converts the larger
operand itself (lbgemm_run_fused); --warpmma the warp-level fp16 MMA kernel
for a small side (lbgemm_run_warpmma); without these the library's own
dispatch runs (lbgemm_run).  --encoded re-encodes A and B once and times only the GEMM
kernel (lbgemm_run_encoded).  --linear runs lbgemm_linear (bits 8).  --popc
runs the 1-bit XOR-popcount kernel (lbgemm_run_popc, bits 1).
"""
from __future__ import annotations

import argparse
import sys


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--bits", type=int, default=8, choices=(8, 4, 1))
    ap.add_argument("-M", type=int, required=True)
    ap.add_argument("-N", type=int, required=True)
    ap.add_argument("-K", type=int, required=True)
    ap.add_argument("--variant", type=int, default=-1)
    ap.add_argument("--encoded", action="store_true")
    ap.add_argument("--fused", type=int, default=0, metavar="TILE_N",
                    help="run lbgemm_run_fused with this tile width (64, 128 or 256)")
    ap.add_argument("--warpmma", action="store_true",
                    help="run lbgemm_run_warpmma (small side <= 32 rows)")
    ap.add_argument("--linear", action="store_true")
    ap.add_argument("--popc", action="store_true",
                    help="run lbgemm_run_popc (bits 1) with the default tile and stages")
    ap.add_argument("--reps", type=int, default=2)
    ap.add_argument("--seed", type=int, default=1)
    a = ap.parse_args(argv)
    import numpy as np  # noqa: PLC0415
    import torch  # noqa: PLC0415  (device memory and streams only)

    from . import lbgemm as L  # noqa: PLC0415
    from . import synth  # noqa: PLC0415

    L.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    M, N, K = a.M, a.N, a.K
    g = synth.rng(a.seed)
    if a.linear:
        X, sx, W, sw = synth.linear_operands(M, N, K, a.seed)
        ops = [torch.from_numpy(x).to(dev) for x in (X, sx, W, sw)]
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

        def call():
            L.lbgemm_linear(M, N, K, ops[0], ops[1], ops[2], ops[3], Y)
    else:
        if a.bits == 8:
            A, B = synth.s8(g, M, K), synth.s8(g, N, K)
        elif a.bits == 4:
            A, B = synth.s4(g, M, K), synth.s4(g, N, K)
        else:
            A, B = synth.b1(g, M, K).view(np.int32), synth.b1(g, N, K).view(np.int32)
        dA, dB = torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev)
        C = torch.empty((M, N), dtype=torch.int32, device=dev)
        if a.encoded:
            eA = torch.empty(L.lbgemm_encoded_size(a.bits, M, K), dtype=torch.uint8, device=dev)
            eB = torch.empty(L.lbgemm_encoded_size(a.bits, N, K), dtype=torch.uint8, device=dev)
            L.lbgemm_encode(a.bits, M, K, dA, eA)
            L.lbgemm_encode(a.bits, N, K, dB, eB)

            def call():
                L.lbgemm_run_encoded(a.bits, M, N, K, eA, eB, C, a.variant)
        elif a.warpmma:
            def call():
                L.lbgemm_run_warpmma(M, N, K, dA, dB, C)
        elif a.popc:
            if a.bits != 1:
                ap.error("--popc needs --bits 1")

            def call():
                L.lbgemm_run_popc(M, N, K, dA, dB, C)
        elif a.fused:
            def call():
                L.lbgemm_run_fused(M, N, K, dA, dB, C, a.fused)
        elif a.variant >= 0:
            def call():
                L.lbgemm_run_variant(a.bits, M, N, K, dA, dB, C, a.variant)
        else:
            def call():
                L.lbgemm_run(a.bits, M, N, K, dA, dB, C)
    stream = torch.cuda.current_stream()
    for r in range(a.reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        e1.synchronize()
        ms = e0.elapsed_time(e1)
        print(f"rep {r}: {ms * 1e3:.1f} us  {2.0 * M * N * K / ms / 1e9:.1f} TOPS", flush=True)
    L.lbgemm_device_status()
    return 0


if __name__ == "__main__":
    sys.exit(main())
