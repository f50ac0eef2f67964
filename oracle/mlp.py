"""Oracle of the learned selector's forward pass -- TEST INFRASTRUCTURE ONLY.

Source [LBG]: "Leveraging Large-Scale Data for Efficient Low-Bit CUTLASS GEMM
Optimization via Neural Networks" (press summary page), section 3: a
feed-forward network with three hidden layers maps (M, N, K, SM count) to
scores of the nine templates; the selected template is the top score.

Readings (where the page is silent): inputs log2 M, log2 N, log2 K and the SM
count, standardised with the stored means and deviations; ReLU after every
layer but the last.  This module reads the weight file with its own parser and
evaluates the network in float64 from that definition.
"""
from __future__ import annotations

import math


def read(path: str):
    tok = open(path).read().split()
    assert tok[0] == "lbgemm-mlp" and tok[1] == "1" and tok[2] == "bits"
    bits = int(tok[3])
    assert tok[4] == "norm"
    norm = [float(t) for t in tok[5:13]]
    assert tok[13] == "layers"
    nl = int(tok[14])
    pos = 15
    layers = []
    for _ in range(nl):
        assert tok[pos] == "layer"
        n_in, n_out = int(tok[pos + 1]), int(tok[pos + 2])
        pos += 3
        W = [[float(tok[pos + o * n_in + i]) for i in range(n_in)] for o in range(n_out)]
        pos += n_in * n_out
        b = [float(tok[pos + o]) for o in range(n_out)]
        pos += n_out
        layers.append((W, b))
    return {"bits": bits, "mean": norm[:4], "std": norm[4:], "layers": layers}


def scores(net, M: int, N: int, K: int, sm_count: int) -> list[float]:
    x = [math.log2(M), math.log2(N), math.log2(K), float(sm_count)]
    h = [(x[i] - net["mean"][i]) / net["std"][i] for i in range(4)]
    for li, (W, b) in enumerate(net["layers"]):
        out = []
        for o in range(len(W)):
            s = b[o] + sum(W[o][i] * h[i] for i in range(len(h)))
            out.append(max(s, 0.0) if li < len(net["layers"]) - 1 else s)
        h = out
    return h


def top2(net, M, N, K, sm_count) -> tuple[int, int, float]:
    """(top class, second class, score gap between them)."""
    s = scores(net, M, N, K, sm_count)
    order = sorted(range(len(s)), key=lambda i: (-s[i], i))
    return order[0], order[1], s[order[0]] - s[order[1]]
