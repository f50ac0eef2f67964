"""GPU parity of the streaming warp-MMA kernel (small side <= 16 rows, the
large operand streamed once through a bulk-copy ring): the 8-bit GEMM
bit-exact against the oracle in both orientations, with ragged row blocks,
K tails of one 16-byte chunk, extremes and an adversarial order; the linear
layer within 1e-2 relative per element (exact zeros where acc = 0)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from bit_tensor_gemm_gb300 import build as bld  # noqa: E402
from bit_tensor_gemm_gb300 import lbgemm as L  # noqa: E402
from bit_tensor_gemm_gb300 import synth  # noqa: E402

LINEAR_RTOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bld.build()
    L.load()


def G():
    import gpu_util  # noqa: PLC0415
    return gpu_util


def stream_gemm(A, B, K):
    M, N = A.shape[0], B.shape[0]
    dA, dB = G().to_dev(A), G().to_dev(B)
    dC = torch.full((M, N), -7, dtype=torch.int32, device="cuda")
    L.lbgemm_run_candidate(8, M, N, K, dA, dB, dC, L.ROUTE_STREAM, 0)
    L.lbgemm_device_status()
    return dC.cpu().numpy()


def assert_exact(got, want, what):
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        m, n = bad[0]
        raise AssertionError(f"{what}: {len(bad)} entries differ; first at ({m},{n}): "
                             f"got {got[m, n]} want {want[m, n]}")


# (M, N, K): one token and 16 tokens against the linear layer's weights, a
# block of rows that is not a multiple of 8 per CTA, fewer rows than one
# stage, more CTAs' worth of rows than SMs, K of one 16-byte chunk, K that
# leaves most warps' slices past K, the largest K, and the small side on B
STREAM_SHAPES = [(1, 11008, 4096), (16, 11008, 4096), (5, 77, 16), (16, 300, 1040), (1, 1, 16),
                 (16, 9, 4096), (9, 1219, 2048), (3, 5000, 48), (7, 2100, 4096),
                 (3000, 7, 512), (2048, 16, 4096), (100, 1, 1024)]


def test_stream_gemm_shapes():
    for i, (M, N, K) in enumerate(STREAM_SHAPES):
        A, B = synth.operands(8, M, N, K, 1700 + i)
        assert_exact(stream_gemm(A, B, K), oracle.gemm(8, A, B, K), f"stream {M}x{N}x{K}")


def test_stream_gemm_extremes_and_order():
    K = 4096
    A = np.full((16, K), -128, np.int8)
    B = np.full((300, K), -128, np.int8)
    assert np.all(stream_gemm(A, B, K) == 16384 * K)
    assert np.all(stream_gemm(B[:40], A[:3], K) == 16384 * K)
    A = np.ones((16, K), np.int8)
    B = np.ones((64, K), np.int8)
    A[:, :511] = -128
    B[:, :511] = -128
    A[:, 1024:2047] = 127
    B[:, 1024:2047] = -128
    B[1::2, 600:1000] = -1
    assert_exact(stream_gemm(A, B, K), oracle.gemm(8, A, B, K), "stream adversarial")


def test_stream_gemm_two_calls_reuse_nothing():
    """A second, smaller call right after a larger one (the same CTAs' rings
    and reduction slots) must not see the first call's data."""
    A, B = synth.operands(8, 16, 5000, 4096, 1800)
    assert_exact(stream_gemm(A, B, 4096), oracle.gemm(8, A, B, 4096), "stream first")
    A, B = synth.operands(8, 3, 700, 272, 1801)
    assert_exact(stream_gemm(A, B, 272), oracle.gemm(8, A, B, 272), "stream second")


def check_linear(got, ref, zero, what):
    assert np.all(got[zero] == 0), f"{what}: nonzero where acc == 0"
    nz = ~zero
    rel = np.abs(got[nz] - ref[nz]) / np.abs(ref[nz])
    assert rel.max() <= LINEAR_RTOL, f"{what}: max rel err {rel.max():.3g}"


@pytest.mark.parametrize("M,N", [(1, 11008), (5, 2100), (16, 11008), (16, 2101)])
def test_stream_linear(M, N):
    K = 4096
    X, sx, W, sw = synth.linear_operands(M, N, K, 1900 + M)
    if M > 1:
        X[1, :] = 0
    ref = oracle.linear(X, sx, W, sw)
    acc = oracle.gemm(8, X, W, K)
    dY = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.lbgemm_linear_candidate(M, N, K, G().to_dev(X), G().to_dev(sx), G().to_dev(W), G().to_dev(sw),
                              dY, L.ROUTE_STREAM, 0)
    L.lbgemm_device_status()
    got = dY.float().cpu().numpy().astype(np.float64)
    check_linear(got, ref, acc == 0, f"stream linear M={M} N={N}")


def test_stream_route_limits():
    dA = torch.zeros(64 * 4112, dtype=torch.int8, device="cuda")
    dC = torch.zeros(64 * 64, dtype=torch.int32, device="cuda")
    for M, N, K in [(17, 64, 1024), (16, 64, 4112), (16, 64, 40)]:
        with pytest.raises(L.LbgemmError) as e:
            L.lbgemm_run_candidate(8, M, N, K, dA, dA, dC, L.ROUTE_STREAM, 0)
        assert e.value.status == L.ERR_INVALID_ARG
