"""GPU parity at the benchmark's full sizes, in the launch configuration the
benchmark times (lbgemm_run / lbgemm_linear), on sampled outputs that the
oracle computes one by one: whole first and last rows plus random entries.
Also every shape of the 729-shape int8 sweep, on shared prefix buffers like
the benchmark, under the default and a rotating forced variant."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from bit_tensor_gemm_gb300 import build as bld  # noqa: E402
from bit_tensor_gemm_gb300 import lbgemm as L  # noqa: E402
from bit_tensor_gemm_gb300 import synth  # noqa: E402

SIZES = [64, 128, 256, 512, 1024, 2048, 4096, 8192, 16384]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bld.build()
    L.load()


def _dev(a):
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _positions(M, N, count, seed):
    g = np.random.default_rng(seed)
    rows = np.concatenate([np.zeros(N, np.int64), np.full(N, M - 1, np.int64),
                           g.integers(0, M, count)])
    cols = np.concatenate([np.arange(N), np.arange(N), g.integers(0, N, count)])
    return rows, cols


def _check_sampled(bits, A, B, K, C_dev, seed, count=4096):
    M, N = C_dev.shape
    rows, cols = _positions(M, N, count, seed)
    got = C_dev[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().numpy()
    want = oracle.entries(bits, A, B, K, rows, cols)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, (f"bits={bits} {M}x{N}x{K}: {bad.size} sampled entries differ, first "
                           f"({rows[bad[0]]},{cols[bad[0]]}) got {got[bad[0]]} want {want[bad[0]]}")


def test_int8_16384_cube():
    M = N = K = 16384
    A, B = synth.operands(8, M, N, K, synth.config_seed(2))
    C = torch.empty((M, N), dtype=torch.int32, device="cuda")
    L.lbgemm_run(8, M, N, K, _dev(A), _dev(B), C)
    L.lbgemm_device_status()
    _check_sampled(8, A, B, K, C, 1)


def test_int4_8192_cube():
    M = N = K = 8192
    A, B = synth.operands(4, M, N, K, synth.config_seed(3))
    C = torch.empty((M, N), dtype=torch.int32, device="cuda")
    L.lbgemm_run(4, M, N, K, _dev(A), _dev(B), C)
    L.lbgemm_device_status()
    _check_sampled(4, A, B, K, C, 2)


def test_b1_8192_square_k65536():
    M = N = 8192
    K = 65536
    A, B = synth.operands(1, M, N, K, synth.config_seed(4))
    C = torch.empty((M, N), dtype=torch.int32, device="cuda")
    dA, dB = _dev(A), _dev(B)
    L.lbgemm_run(1, M, N, K, dA, dB, C)  # tensor-core route
    L.lbgemm_device_status()
    _check_sampled(1, A, B, K, C, 3, count=2048)
    C.fill_(-1)
    L.lbgemm_run_popc(M, N, K, dA, dB, C)  # XOR-popcount route
    L.lbgemm_device_status()
    _check_sampled(1, A, B, K, C, 4, count=2048)


@pytest.mark.parametrize("M", [1, 16, 128, 2048])
def test_linear_full_width(M):
    N, K = 11008, 4096
    X, sx, W, sw = synth.linear_operands(M, N, K, synth.config_seed(5) + M)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    L.lbgemm_linear(M, N, K, _dev(X), _dev(sx), _dev(W), _dev(sw), Y)
    L.lbgemm_device_status()
    rows, cols = _positions(M, N, 4096, 10 + M)
    acc = oracle.entries(8, X, W, K, rows, cols).astype(np.float64)
    ref = acc * sx[rows].astype(np.float64) * sw[cols].astype(np.float64)
    got = Y.float()[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]
    got = got.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 1e-2 * np.abs(ref))
    assert np.all(got[acc == 0] == 0)


def test_int8_sweep_every_shape():
    """All 729 sweep shapes on shared prefix buffers (as the benchmark runs
    them): the default dispatch and one forced variant per shape (rotating
    through all nine), 64 random entries plus the corners checked each."""
    D = SIZES[-1]
    g = synth.rng(synth.config_seed(2))
    A = synth.s8(g, D, D).reshape(-1)
    B = synth.s8(g, D, D).reshape(-1)
    dA, dB = _dev(A), _dev(B)
    C = torch.empty(D * D, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(99)
    shapes = [(m, n, k) for m in SIZES for n in SIZES for k in SIZES]
    for idx, (m, n, k) in enumerate(shapes):
        a = A[: m * k].reshape(m, k)
        b = B[: n * k].reshape(n, k)
        rows = np.concatenate([[0, m - 1, 0, m - 1], rng.integers(0, m, 64)])
        cols = np.concatenate([[0, n - 1, n - 1, 0], rng.integers(0, n, 64)])
        want = oracle.entries(8, a, b, k, rows, cols)
        for variant in (-1, idx % 9):
            if variant < 0:
                L.lbgemm_run(8, m, n, k, dA, dB, C)
            else:
                L.lbgemm_run_variant(8, m, n, k, dA, dB, C, variant)
            got = C[: m * n].view(m, n)[torch.from_numpy(rows).cuda(),
                                        torch.from_numpy(cols).cuda()].cpu().numpy()
            assert np.array_equal(got, want), f"sweep shape {m}x{n}x{k} variant {variant}"
    L.lbgemm_device_status()
