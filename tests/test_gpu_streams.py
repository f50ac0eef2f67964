"""Concurrent calls: two host threads, each with its own stream, issue GEMMs
and linear layers on the tensor-core routes at the same time.  The library's
per-device scratch is shared between them (a host lock around its use, an
event ordering each stream's use after the other's), so every result must
still match the oracle exactly (GEMM) or within 1e-2 (linear layer)."""
import threading

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


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def test_two_threads_two_streams_share_the_scratch():
    # shapes on the variant-table route (both operands re-encoded into the
    # scratch), the in-kernel conversion route and the split linear layer
    jobs = []
    for i, (M, N, K) in enumerate([(1024, 1024, 2048), (64, 8192, 4096), (768, 512, 4096),
                                   (2048, 256, 1024)] * 2):
        A, B = synth.operands(8, M, N, K, 60 + i)
        jobs.append(("gemm", M, N, K, A, B, _dev(A), _dev(B),
                     torch.full((M, N), -7, dtype=torch.int32, device="cuda")))
    for i, (M, N, K) in enumerate([(64, 4096, 4096), (24, 4096, 11008)] * 2):
        X, sx, W, sw = synth.linear_operands(M, N, K, 80 + i)
        jobs.append(("linear", M, N, K, (X, sx, W, sw), [_dev(v) for v in (X, sx, W, sw)], None,
                     None, torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    errors = []

    def worker(t):
        try:
            s = streams[t]
            for rep in range(3):
                for j in jobs[t::2]:
                    if j[0] == "gemm":
                        _, M, N, K, _, _, dA, dB, C = j
                        L.lbgemm_run(8, M, N, K, dA, dB, C, stream=s)
                    else:
                        _, M, N, K, _, dv, _, _, Y = j
                        L.lbgemm_linear(M, N, K, dv[0], dv[1], dv[2], dv[3], Y, stream=s)
        except Exception as e:  # noqa: BLE001
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    L.lbgemm_device_status()
    for j in jobs:
        if j[0] == "gemm":
            _, M, N, K, A, B, _, _, C = j
            assert np.array_equal(C.cpu().numpy(), oracle.gemm(8, A, B, K)), (M, N, K)
        else:
            _, M, N, K, (X, sx, W, sw), _, _, _, Y = j
            ref = oracle.linear(X, sx, W, sw)
            acc = oracle.gemm(8, X, W, K)
            got = Y.float().cpu().numpy().astype(np.float64)
            nz = acc != 0
            assert np.all(got[~nz] == 0)
            assert np.all(np.abs(got[nz] - ref[nz]) <= 1e-2 * np.abs(ref[nz])), (M, N, K)
