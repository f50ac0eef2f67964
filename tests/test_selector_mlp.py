"""The learned selector ("Leveraging Large-Scale Data for Efficient Low-Bit
CUTLASS GEMM Optimization via Neural Networks", press summary page, section 3):
the oracle's forward pass is pinned to a hand-worked network, the library's
predictor agrees with the oracle on trained-shape networks, and the trainer
learns a separable labelling.  CPU only."""
import os

import numpy as np
import pytest

from bit_tensor_gemm_gb300 import build as bld
from bit_tensor_gemm_gb300 import lbgemm as L
from bit_tensor_gemm_gb300 import selector_mlp as S
from oracle import mlp as omlp

TINY = os.path.join(os.path.dirname(__file__), "golden", "mlp_tiny.txt")


@pytest.fixture(scope="module")
def lib():
    bld.build()
    return L.load()


def test_oracle_forward_hand_worked():
    """Two-layer network of tests/golden/mlp_tiny.txt, worked by hand:
    h = relu([x0, x1 - 1]); scores = [h0, h1, 10 - h0 - h1], x = (log2 M,
    log2 N, log2 K, sm)."""
    net = omlp.read(TINY)
    assert omlp.scores(net, 8, 4, 2, 5) == [3.0, 1.0, 6.0]      # h = (3, 1)
    assert omlp.top2(net, 8, 4, 2, 5)[:2] == (2, 0)
    assert omlp.scores(net, 2, 16, 2, 1) == [1.0, 3.0, 6.0]     # h = (1, 3)
    assert omlp.top2(net, 1024, 1024, 8, 1)[:2] == (0, 1)        # h = (10, 9): -9 last
    assert omlp.scores(net, 1, 1, 1, 0) == [0.0, 0.0, 10.0]     # relu clips x1 - 1 = -1


def test_library_matches_hand_worked(lib):
    L.lbgemm_mlp_clear()  # the shipped networks load by default
    L.lbgemm_mlp_load(TINY)
    assert L.lbgemm_mlp_predict(8, 8, 4, 2, 5) == (2, 0)
    assert L.lbgemm_mlp_predict(8, 2, 16, 2, 1) == (2, 1)
    assert L.lbgemm_mlp_predict(8, 1024, 1024, 8, 1) == (0, 1)
    assert L.lbgemm_mlp_predict(4, 8, 4, 2, 5) == (-1, -1)      # nothing loaded for 4-bit
    # a three-class network is not used by selection
    assert L.lbgemm_select_for(4343, 8, 100, 100, 100) == 7
    L.lbgemm_mlp_clear()


def test_library_matches_oracle_on_a_random_network(lib, tmp_path):
    net = S.MLP(8, seed=3)
    g = np.random.default_rng(4)
    for W in net.W:
        W *= 1.5
    net.b = [g.standard_normal(b.shape) * 0.5 for b in net.b]
    net.mean = np.array([9.0, 9.0, 9.0, 152.0])
    net.std = np.array([2.5, 2.5, 2.5, 1.0])
    path = str(tmp_path / "net.txt")
    net.save(path)
    L.lbgemm_mlp_load(path)
    ref = omlp.read(path)
    checked = 0
    for _ in range(300):
        M, N, K = (int(v) for v in np.exp2(g.uniform(6, 14, 3)).round())
        first, second = L.lbgemm_mlp_predict(8, M, N, K, 152)
        o1, o2, gap = omlp.top2(ref, M, N, K, 152)
        if gap > 1e-3:  # fp32 vs fp64 may order near-ties differently
            assert first == o1, (M, N, K)
            checked += 1
        assert first in (o1, o2)
        # selection uses the network for shapes outside the table
        assert L.lbgemm_select_for(152, 8, M, N, K) == first
    assert checked > 250
    # the numpy trainer's own forward pass agrees too
    X = S.features([64, 4096], [128, 8192], [1024, 256], 152)
    assert (net.predict_top2(X)[:, 0] == [omlp.top2(ref, 64, 128, 1024, 152)[0],
                                          omlp.top2(ref, 4096, 8192, 256, 152)[0]]).all()
    L.lbgemm_mlp_clear()
    assert L.lbgemm_mlp_predict(8, 64, 64, 64, 152) == (-1, -1)


def test_malformed_network_file(lib, tmp_path):
    bad = tmp_path / "bad.txt"
    bad.write_text("lbgemm-mlp 1\nbits 8\nnorm 0 0 0 0 1 1 1 0\nlayers 1\n")
    with pytest.raises(L.LbgemmError):
        L.lbgemm_mlp_load(str(bad))
    bad.write_text("lbgemm-mlp 1\nbits 8\nnorm 0 0 0 0 1 1 1 1\nlayers 1\nlayer 4 2\n1 2 3\n")
    with pytest.raises(L.LbgemmError):
        L.lbgemm_mlp_load(str(bad))


def test_trainer_learns_a_separable_labelling():
    """Labels that depend on the shape only (the class is the bucket of
    log2(M) + log2(N)): the trained network must get nearly all of them."""
    g = np.random.default_rng(5)
    M, N, K = (np.exp2(g.integers(6, 15, 400)) for _ in range(3))
    X = S.features(M, N, K, 152)
    y = np.clip(((np.log2(M) + np.log2(N)) - 12) // 2, 0, 8).astype(int)
    net = S.MLP(8, seed=1).fit(X, y, epochs=120)
    top1, top2 = S.topk_accuracy(net.predict_top2(X), y)
    assert top1 > 0.9 and top2 > 0.97


def test_save_load_roundtrip(tmp_path):
    net = S.MLP(4, seed=2)
    net.mean = np.array([1.0, 2.0, 3.0, 4.0])
    p = str(tmp_path / "n.txt")
    net.save(p)
    back = S.MLP.load(p)
    X = S.features([100, 7], [300, 9000], [64, 4096], 152)
    assert np.allclose(back.logits(X), net.logits(X), rtol=1e-6, atol=1e-6)
    assert back.bits == 4


def test_shipped_networks_load_by_default_and_answer_their_sm_count(lib):
    """A fresh process has the GB300 networks of every bit width; a network
    trained on one SM count does not answer for another."""
    import json  # noqa: PLC0415
    import subprocess  # noqa: PLC0415
    import sys  # noqa: PLC0415
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import sys, json; sys.path.insert(0, %r)\n"
            "from bit_tensor_gemm_gb300 import lbgemm as L\n"
            "print(json.dumps([L.lbgemm_mlp_predict(b, 300, 5000, 700, 152)[0] for b in (8, 4, 1)]"
            " + [L.lbgemm_select_for(150, 8, 300, 5000, 700)]))" % root)
    env = {k: v for k, v in os.environ.items() if k not in ("LBGEMM_MLP", "LBGEMM_TABLE")}
    got = json.loads(subprocess.run([sys.executable, "-c", code], env=env, capture_output=True,
                                    text=True, check=True).stdout)
    for bits, v in zip((8, 4, 1), got[:3]):
        net = S.MLP.load(os.path.join(root, "bit_tensor_gemm_gb300", "data",
                                      f"mlp_gb300_s{bits}.txt"))
        assert v == int(net.predict_top2(S.features([300], [5000], [700], 152))[0, 0]), bits
    # SM count 150: no table entries, the network does not apply: the default
    assert got[3] == 7
    env["LBGEMM_MLP"] = "none"
    got = json.loads(subprocess.run([sys.executable, "-c", code], env=env, capture_output=True,
                                    text=True, check=True).stdout)
    assert got[:3] == [-1, -1, -1]
