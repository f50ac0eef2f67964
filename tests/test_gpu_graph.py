"""CUDA graphs: library calls captured on a stream and replayed.  While a
stream is captured the library takes its scratch from stream-ordered
allocations of the graph itself, so a captured call needs no warm-up of the
per-device buffer and stays valid after that buffer is reallocated by a
larger call.  Every replay is checked against the oracle (bit-exact for the
GEMM; within 1e-2 for the linear layer), on fresh operand values copied into
the captured buffers between replays."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from bit_tensor_gemm_gb300 import build as bld  # noqa: E402
from bit_tensor_gemm_gb300 import lbgemm as L  # noqa: E402
from bit_tensor_gemm_gb300 import synth  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bld.build()
    L.load()
    # the library's per-device state exists before any capture
    a = torch.zeros(64 * 64, dtype=torch.int8, device="cuda")
    c = torch.zeros(64 * 64, dtype=torch.int32, device="cuda")
    L.lbgemm_run(8, 64, 64, 64, a, a, c)
    torch.cuda.synchronize()


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _grow_shared_scratch():
    """A call that needs more scratch than anything before it (the shared
    buffer is freed and allocated again)."""
    M = N = K = 8192
    a = torch.zeros(M * K, dtype=torch.int8, device="cuda")
    c = torch.empty(M * N, dtype=torch.int32, device="cuda")
    L.lbgemm_run_variant(8, M, N, K, a, a, c, 7)
    torch.cuda.synchronize()


# (bits, M, N, K): the tensor-core table route with re-encoding, the
# in-kernel conversion route, the one-launch dp4a route, 4-bit and 1-bit on
# the tensor cores, and the 1-bit popcount route
GEMM_CASES = [(8, 1024, 1024, 4096), (8, 64, 8192, 4096), (8, 256, 256, 256),
              (4, 512, 512, 1024), (1, 256, 256, 2048), (1, 64, 64, 1024)]


@pytest.mark.parametrize("bits,M,N,K", GEMM_CASES)
def test_gemm_captured_and_replayed(bits, M, N, K):
    A, B = synth.operands(bits, M, N, K, 31)
    dA, dB = _dev(A), _dev(B)
    C = torch.full((M, N), -7, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        L.lbgemm_run(bits, M, N, K, dA, dB, C, stream=s)
    for rep in range(2):
        if rep:
            A, B = synth.operands(bits, M, N, K, 32)
            dA.copy_(_dev(A))
            dB.copy_(_dev(B))
            _grow_shared_scratch()
        C.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        L.lbgemm_device_status()
        assert np.array_equal(C.cpu().numpy(), oracle.gemm(bits, A, B, K)), (bits, M, N, K, rep)


# token counts on the dp4a, streaming, split-K, stream-K and variant-table routes
LINEAR_CASES = [(1, 4096, 4096), (16, 11008, 4096), (64, 4096, 4096), (128, 11008, 4096),
                (1024, 2048, 1024)]


@pytest.mark.parametrize("M,N,K", LINEAR_CASES)
def test_linear_captured_and_replayed(M, N, K):
    X, sx, W, sw = synth.linear_operands(M, N, K, 41)
    dX, dsx, dW, dsw = _dev(X), _dev(sx), _dev(W), _dev(sw)
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        L.lbgemm_linear(M, N, K, dX, dsx, dW, dsw, Y, stream=s)
    for rep in range(2):
        if rep:
            X, sx, W, sw = synth.linear_operands(M, N, K, 42)
            dX.copy_(_dev(X))
            dsx.copy_(_dev(sx))
            dW.copy_(_dev(W))
            dsw.copy_(_dev(sw))
            _grow_shared_scratch()
        Y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        L.lbgemm_device_status()
        ref = oracle.linear(X, sx, W, sw)
        got = Y.float().cpu().numpy().astype(np.float64)
        acc = oracle.gemm(8, X, W, K)
        assert np.all(got[acc == 0] == 0)
        nz = acc != 0
        assert np.all(np.abs(got[nz] - ref[nz]) <= 1e-2 * np.abs(ref[nz])), (M, N, K, rep)


def test_quantised_linear_captured():
    M, N, K = 64, 4096, 4096
    g0 = np.random.default_rng(5)
    xf = (g0.standard_normal((M, K))).astype(np.float32)
    xt = torch.from_numpy(xf).to(torch.bfloat16)
    xf = xt.float().numpy()
    W = g0.integers(-127, 128, (N, K)).astype(np.int8)
    sw = (g0.random(N) * 0.01).astype(np.float32)
    dX, dW, dsw = xt.cuda(), _dev(W), _dev(sw)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        L.lbgemm_linear_quant(M, N, K, dX, dW, dsw, Y, stream=s)
    g.replay()
    torch.cuda.synchronize()
    L.lbgemm_device_status()
    ref = oracle.linear_quant(xf, W, sw)
    q, _ = oracle.quantize_rows(xf)
    acc = oracle.gemm(8, q, W, K)
    got = Y.float().cpu().numpy().astype(np.float64)
    nz = acc != 0
    assert np.all(np.abs(got[nz] - ref[nz]) <= 1e-2 * np.abs(ref[nz]))


def test_caller_workspace_entry_captured():
    """lbgemm_run_ws inside a graph: the caller's workspace, no library
    scratch at all."""
    bits, M, N, K = 8, 512, 768, 2048
    A, B = synth.operands(bits, M, N, K, 51)
    dA, dB = _dev(A), _dev(B)
    C = torch.full((M, N), -7, dtype=torch.int32, device="cuda")
    need = L.lbgemm_workspace_size(bits, M, N, K)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        L.lbgemm_run_ws(bits, M, N, K, dA, dB, C, -1, ws, need, stream=s)
    g.replay()
    torch.cuda.synchronize()
    L.lbgemm_device_status()
    assert np.array_equal(C.cpu().numpy(), oracle.gemm(bits, A, B, K))
