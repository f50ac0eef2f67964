"""lbgemm_run_static: the entry point for callers that cannot allocate GPU
memory (code running where cudaMalloc is off limits and no workspace can be
handed over).  It must give the oracle's exact product, call after call,
while its scratch lives in one array compiled into the library, and it must
allocate nothing.  This file is named to run last, so a failure here comes
after every other test has run."""
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


def _dev(a):
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


# (bits, M, N, K, seed, variant, route): forced variants of the tensor-core
# route, a large problem before a smaller one with another padded row length
# (no leftovers may leak), 4-bit and 1-bit, and variant -1 with a table entry
# naming the route: the in-kernel conversion kernel (scratch for one operand
# only: both would not fit), the warp-MMA kernel on a 16-token linear-layer
# shape (no scratch) and the popcount kernel (no scratch)
CASES = [(8, 1024, 768, 4104, 901, 8, None), (8, 200, 136, 264, 902, 4, None),
         (4, 512, 640, 2050, 903, 7, None), (4, 130, 70, 514, 904, 0, None),
         (1, 96, 80, 2048, 905, 2, None), (8, 256, 8192, 2048, 906, -1, (5, 128)),
         (8, 16, 11008, 4096, 907, -1, (3, 0)), (1, 64, 64, 1024, 908, -1, (1, 4))]


def _problems():
    out = []
    for bits, M, N, K, seed, v, _ in CASES:
        A, B = synth.operands(bits, M, N, K, seed)
        out.append((bits, M, N, K, v, _dev(A), _dev(B), oracle.gemm(bits, A, B, K),
                    torch.empty((M, N), dtype=torch.int32, device="cuda")))
    return out


@pytest.fixture
def routed_entries():
    """Table entries that send the variant -1 cases to their routes; the
    previous entries come back afterwards."""
    sm = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    saved = []
    for bits, M, N, K, _, v, route in CASES:
        if route is not None:
            saved.append(((bits, M, N, K), L.lbgemm_table_get_for(sm, bits, M, N, K)))
            L.lbgemm_table_set_choice_for(sm, bits, M, N, K, 7, *route)
            assert L.lbgemm_dispatch_for(sm, bits, M, N, K) == route
    yield
    for shape, entry in saved:
        L.lbgemm_table_set_choice_for(sm, *shape, *(entry or (7, -1, 0)))


def test_static_matches_oracle_two_calls_in_a_row_and_allocates_nothing(routed_entries):
    # the in-kernel conversion case needs more than the array on the
    # tensor-core route, and fits on its own route
    assert L.lbgemm_workspace_size(8, 256, 8192, 2048) > L.STATIC_SCRATCH_BYTES
    probs = _problems()
    # the first call of each kernel may load its code into the device (lazy
    # module loading, the library's and torch's fill and copy kernels alike);
    # device memory is compared from the second round of calls on
    for bits, M, N, K, v, dA, dB, want, dC in probs:
        dC.fill_(-2)
        L.lbgemm_run_static(bits, M, N, K, dA, dB, dC, v)
        dC.cpu()
    L.lbgemm_device_status()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for call in range(2):
        for bits, M, N, K, v, dA, dB, want, dC in probs:
            dC.fill_(-3 - call)
            L.lbgemm_run_static(bits, M, N, K, dA, dB, dC, v)
            L.lbgemm_device_status()
            got = dC.cpu().numpy()
            assert np.array_equal(got, want), f"call {call}: {bits}-bit {M}x{N}x{K} v={v} differs"
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "device memory changed across the calls"


def test_static_limit_is_enforced_before_running():
    M = N = 4096
    K = 4096  # (M + N) * K * 2 bytes = 64 MiB of scratch > 32 MiB
    assert L.lbgemm_workspace_size(8, M, N, K) > L.STATIC_SCRATCH_BYTES
    dummy = torch.empty(16, dtype=torch.int8, device="cuda")
    with pytest.raises(L.LbgemmError) as e:
        L.lbgemm_run_static(8, M, N, K, dummy, dummy, dummy, 7)
    assert e.value.status == L.ERR_WORKSPACE
    assert "static" in L.lbgemm_last_error()


def test_static_entry_captured_in_a_graph():
    """Captured into a CUDA graph after one call outside capture (the array's
    address is looked up then), the static entry replays exactly; the graph
    holds no allocation node, as the call allocates nothing."""
    bits, M, N, K = 8, 1024, 768, 4104
    A, B = synth.operands(bits, M, N, K, 911)
    dA, dB = _dev(A), _dev(B)
    dC = torch.full((M, N), -5, dtype=torch.int32, device="cuda")
    L.lbgemm_run_static(bits, M, N, K, dA, dB, dC, 8)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        L.lbgemm_run_static(bits, M, N, K, dA, dB, dC, 8, stream=s)
    for call in range(2):
        dC.fill_(-5 - call)
        g.replay()
        torch.cuda.synchronize()
        L.lbgemm_device_status()
        assert np.array_equal(dC.cpu().numpy(), oracle.gemm(bits, A, B, K)), call
