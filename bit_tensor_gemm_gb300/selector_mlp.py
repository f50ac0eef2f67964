"""Training of the variant selector MLP, and its weight file.

Method: "Leveraging Large-Scale Data for Efficient Low-Bit CUTLASS GEMM
Optimization via Neural Networks" (press summary page).  Section 2: each
(M, N, K) sample is labelled with the index of its fastest template among
nine.  Section 3: a feed-forward network with an input layer, three hidden
layers of width 128 and a nine-way output, inputs M, N, K and the GPU's SM
count, trained with cross-entropy and Adam (batch 32, learning rate 0.001) and
judged by top-2 accuracy (the best two templates are close in time).

Readings where the page is silent: the inputs are log2(M), log2(N), log2(K)
and the SM count, each standardised with the training set's mean and
standard deviation (a constant feature keeps standard deviation 1); hidden
layers use ReLU; weights start He-normal, biases at zero.

The weight file is plain text, read by the library (lbgemm_mlp_load):
    lbgemm-mlp 1
    bits <b>
    norm <mean x4> <std x4>
    layers <L>
    layer <in> <out>      then <out> lines of <in> weights, then one line of <out> biases
    ...
The network runs on the host (float32); the library answers
lbgemm_select for shapes that are not in the timing table with its argmax.
"""
from __future__ import annotations

import math

import numpy as np

HIDDEN = (128, 128, 128)
NUM_CLASSES = 9


def features(M, N, K, sm_count) -> np.ndarray:
    M, N, K, S = (np.asarray(x, dtype=np.float64) for x in (M, N, K, sm_count))
    return np.stack([np.log2(M), np.log2(N), np.log2(K), S * np.ones_like(M)], axis=-1)


class MLP:
    def __init__(self, bits: int, n_in: int = 4, hidden=HIDDEN, n_out: int = NUM_CLASSES,
                 seed: int = 0):
        g = np.random.default_rng(seed)
        sizes = (n_in,) + tuple(hidden) + (n_out,)
        self.bits = bits
        self.W = [g.standard_normal((o, i)) * math.sqrt(2.0 / i) for i, o in zip(sizes, sizes[1:])]
        self.b = [np.zeros(o) for o in sizes[1:]]
        self.mean = np.zeros(n_in)
        self.std = np.ones(n_in)

    # -- inference -------------------------------------------------------------
    def logits(self, X: np.ndarray) -> np.ndarray:
        h = (X - self.mean) / self.std
        for li, (W, b) in enumerate(zip(self.W, self.b)):
            h = h @ W.T + b
            if li < len(self.W) - 1:
                h = np.maximum(h, 0.0)
        return h

    def predict_top2(self, X: np.ndarray) -> np.ndarray:
        z = self.logits(X)
        return np.argsort(-z, axis=1, kind="stable")[:, :2]

    # -- training ----------------------------------------------------------------
    def fit(self, X: np.ndarray, y: np.ndarray, epochs: int = 300, batch: int = 32,
            lr: float = 1e-3, seed: int = 0, log=None) -> "MLP":
        """Cross-entropy, Adam (beta 0.9 / 0.999, eps 1e-8), mini-batches of `batch`."""
        self.mean = X.mean(axis=0)
        sd = X.std(axis=0)
        self.std = np.where(sd > 1e-12, sd, 1.0)
        params = self.W + self.b
        m1 = [np.zeros_like(p) for p in params]
        m2 = [np.zeros_like(p) for p in params]
        g = np.random.default_rng(seed)
        step = 0
        n = len(X)
        for ep in range(epochs):
            order = g.permutation(n)
            total = 0.0
            for s in range(0, n, batch):
                idx = order[s:s + batch]
                grads, loss = self._grads(X[idx], y[idx])
                total += loss * len(idx)
                step += 1
                for i, (p, gr) in enumerate(zip(params, grads)):
                    m1[i] = 0.9 * m1[i] + 0.1 * gr
                    m2[i] = 0.999 * m2[i] + 0.001 * gr * gr
                    mh = m1[i] / (1 - 0.9 ** step)
                    vh = m2[i] / (1 - 0.999 ** step)
                    p -= lr * mh / (np.sqrt(vh) + 1e-8)
            if log and (ep % 50 == 0 or ep == epochs - 1):
                log(f"epoch {ep}: loss {total / n:.4f}")
        return self

    def _grads(self, X, y):
        h = (X - self.mean) / self.std
        acts = [h]
        for li, (W, b) in enumerate(zip(self.W, self.b)):
            h = h @ W.T + b
            if li < len(self.W) - 1:
                h = np.maximum(h, 0.0)
            acts.append(h)
        z = acts[-1]
        z = z - z.max(axis=1, keepdims=True)
        p = np.exp(z)
        p /= p.sum(axis=1, keepdims=True)
        nb = len(X)
        loss = float(-np.log(p[np.arange(nb), y] + 1e-12).mean())
        d = p
        d[np.arange(nb), y] -= 1.0
        d /= nb
        gW = [None] * len(self.W)
        gb = [None] * len(self.W)
        for li in range(len(self.W) - 1, -1, -1):
            gW[li] = d.T @ acts[li]
            gb[li] = d.sum(axis=0)
            if li > 0:
                d = (d @ self.W[li]) * (acts[li] > 0)
        return gW + gb, loss

    # -- file format ------------------------------------------------------------
    def save(self, path: str) -> None:
        with open(path, "w") as f:
            f.write("lbgemm-mlp 1\n")
            f.write(f"bits {self.bits}\n")
            f.write("norm " + " ".join(f"{v:.9g}" for v in list(self.mean) + list(self.std)) + "\n")
            f.write(f"layers {len(self.W)}\n")
            for W, b in zip(self.W, self.b):
                f.write(f"layer {W.shape[1]} {W.shape[0]}\n")
                for row in W:
                    f.write(" ".join(f"{v:.9g}" for v in row) + "\n")
                f.write(" ".join(f"{v:.9g}" for v in b) + "\n")

    @classmethod
    def load(cls, path: str) -> "MLP":
        with open(path) as f:
            tok = f.read().split()
        pos = 0

        def take(n=1):
            nonlocal pos
            out = tok[pos:pos + n]
            pos += n
            return out

        assert take(2) == ["lbgemm-mlp", "1"]
        assert take()[0] == "bits"
        bits = int(take()[0])
        assert take()[0] == "norm"
        norm = [float(v) for v in take(8)]
        assert take()[0] == "layers"
        L = int(take()[0])
        net = cls.__new__(cls)
        net.bits = bits
        net.mean, net.std = np.array(norm[:4]), np.array(norm[4:])
        net.W, net.b = [], []
        for _ in range(L):
            assert take()[0] == "layer"
            n_in, n_out = int(take()[0]), int(take()[0])
            net.W.append(np.array([float(v) for v in take(n_in * n_out)]).reshape(n_out, n_in))
            net.b.append(np.array([float(v) for v in take(n_out)]))
        return net


def labels_from_times(times: np.ndarray) -> np.ndarray:
    """Index of the fastest variant per sample, lowest index on ties (section 2)."""
    return np.argmin(times, axis=1)


def within_accuracy(pred: np.ndarray, times: np.ndarray, tol: float = 0.02) -> float:
    """Fraction of samples whose predicted variant is within tol of the fastest."""
    t = times[np.arange(len(times)), pred]
    return float(np.mean(t <= times.min(axis=1) * (1.0 + tol)))


def near_best_top2(top2: np.ndarray, times: np.ndarray, tol: float = 0.02) -> float:
    """Fraction of samples whose two predicted variants include one within
    tol of the fastest (the page judges top-2 because the best two templates
    are often nearly tied)."""
    idx = np.arange(len(times))
    t = np.minimum(times[idx, top2[:, 0]], times[idx, top2[:, 1]])
    return float(np.mean(t <= times.min(axis=1) * (1.0 + tol)))


def tie_rate(times: np.ndarray, tol: float = 0.02) -> float:
    """Fraction of samples whose two fastest variants lie within tol of each
    other: there the argmin label is decided by timing noise."""
    s = np.sort(times, axis=1)
    return float(np.mean(s[:, 1] <= s[:, 0] * (1.0 + tol)))


def report(net: "MLP", X: np.ndarray, y: np.ndarray, T: np.ndarray) -> dict:
    """Accuracy figures of a network on labelled samples with their times."""
    p = net.predict_top2(X)
    t1, t2 = topk_accuracy(p, y)
    tp = T[np.arange(len(T)), p[:, 0]]
    return {"samples": int(len(X)), "top1": t1, "top2": t2,
            "top2_near_best": near_best_top2(p, T), "top1_within_2pct": within_accuracy(p[:, 0], T),
            "time_pred_over_best": float(tp.sum() / T.min(axis=1).sum()),
            "time_default_over_best": float(T[:, 7].sum() / T.min(axis=1).sum()),
            "best_two_within_2pct": tie_rate(T)}


def load_dataset(path: str):
    """(features, labels, times) of a CSV written by bit_tensor_gemm_gb300.sweep."""
    D = np.loadtxt(path, delimiter=",", skiprows=1, ndmin=2)
    return features(D[:, 0], D[:, 1], D[:, 2], D[:, 3]), labels_from_times(D[:, 4:13]), D[:, 4:13]


def main(argv=None) -> int:
    import argparse  # noqa: PLC0415
    import json  # noqa: PLC0415
    ap = argparse.ArgumentParser(description="train the variant selector on a sweep CSV")
    ap.add_argument("--data", required=True, help="training CSV (random shapes)")
    ap.add_argument("--eval", default="", help="held-out CSV (e.g. the 729-shape grid)")
    ap.add_argument("--out", required=True)
    ap.add_argument("--bits", type=int, default=8)
    ap.add_argument("--epochs", type=int, default=100)
    ap.add_argument("--seed", type=int, default=0)
    a = ap.parse_args(argv)
    X, y, T = load_dataset(a.data)
    g = np.random.default_rng(a.seed)
    perm = g.permutation(len(X))
    ntr = int(0.8 * len(X))
    tr, te = perm[:ntr], perm[ntr:]
    probe = MLP(a.bits, seed=a.seed).fit(X[tr], y[tr], epochs=a.epochs)
    out = {"held_out_20pct": report(probe, X[te], y[te], T[te])}
    net = MLP(a.bits, seed=a.seed).fit(X, y, epochs=a.epochs)
    net.save(a.out)
    if a.eval:
        Xe, ye, Te = load_dataset(a.eval)
        out["eval"] = report(net, Xe, ye, Te)
    out["trained_on"] = f"{len(X)} samples of {a.data}"
    print(json.dumps(out, indent=1))
    return 0


def topk_accuracy(top2: np.ndarray, y: np.ndarray) -> tuple[float, float]:
    top1 = float(np.mean(top2[:, 0] == y))
    top2a = float(np.mean((top2[:, 0] == y) | (top2[:, 1] == y)))
    return top1, top2a


if __name__ == "__main__":
    import sys  # noqa: PLC0415
    sys.exit(main())
