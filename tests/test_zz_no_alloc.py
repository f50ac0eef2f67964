"""lbgemm_run_static: the entry point for callers that cannot allocate GPU
memory (code running where cudaMalloc is off limits and no workspace can be
handed over).  It must give exactly what the allocating entry point gives,
call after call, while its scratch lives in one array compiled into the
library.  This file is named to run last, so a failure here comes after every
other test has run."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

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


def _pair(bits, M, N, K, seed, variant):
    """Run the same problem through lbgemm_run_static and lbgemm_run_variant."""
    A, B = synth.operands(bits, M, N, K, seed)
    dA, dB = _dev(A), _dev(B)
    c_static = torch.full((M, N), -3, dtype=torch.int32, device="cuda")
    c_ref = torch.full((M, N), -5, dtype=torch.int32, device="cuda")
    L.lbgemm_run_static(bits, M, N, K, dA, dB, c_static, variant)
    L.lbgemm_run_variant(bits, M, N, K, dA, dB, c_ref, variant)
    L.lbgemm_device_status()
    return c_static.cpu().numpy(), c_ref.cpu().numpy()


def test_static_matches_allocating_entry_two_calls_in_a_row():
    # First call: a larger problem fills much of the array; the second, smaller
    # one (different K, so a different padded row length) must not see leftovers.
    for bits, M, N, K, seed, v in [(8, 1024, 768, 4104, 901, 8), (8, 200, 136, 264, 902, 4),
                                   (4, 512, 640, 2050, 903, 7), (4, 130, 70, 514, 904, 0)]:
        got, want = _pair(bits, M, N, K, seed, v)
        assert np.array_equal(got, want), f"bits={bits} {M}x{N}x{K}: static result differs"


def test_static_limit_is_enforced_before_running():
    M = N = 4096
    K = 4096  # (M + N) * K * 2 bytes = 64 MiB of scratch > 32 MiB
    assert L.lbgemm_workspace_size(8, M, N, K) > L.STATIC_SCRATCH_BYTES
    dummy = torch.empty(16, dtype=torch.int8, device="cuda")
    with pytest.raises(L.LbgemmError) as e:
        L.lbgemm_run_static(8, M, N, K, dummy, dummy, dummy, -1)
    assert e.value.status == L.ERR_WORKSPACE
    assert "static" in L.lbgemm_last_error()


def test_static_one_bit():
    got, want = _pair(1, 96, 80, 2048, 905, 2)
    assert np.array_equal(got, want)
