"""GPU tests of the selection machinery: the timing entry points leave a
correct product and sane medians behind, every candidate kernel the sweep
measures is bit-exact against the oracle, and the dispatch runs a table
entry's measured route correctly.  Through the C ABI only."""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from bit_tensor_gemm_gb300 import build as bld  # noqa: E402
from bit_tensor_gemm_gb300 import lbgemm as L  # noqa: E402
from bit_tensor_gemm_gb300 import synth  # noqa: E402
from bit_tensor_gemm_gb300 import tune  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bld.build()
    L.load()


def G():
    import gpu_util  # noqa: PLC0415
    return gpu_util


def _setup(bits, M, N, K, seed):
    A, B = synth.operands(bits, M, N, K, seed)
    dC = torch.full((M, N), -7, dtype=torch.int32, device="cuda")
    return A, B, G().to_dev(A), G().to_dev(B), dC


@pytest.mark.parametrize("flush", [True, False])
def test_time_variants_medians_and_product(flush):
    """Nine finite positive medians; C is the exact product afterwards (the
    last timed run wrote it); the stream is usable for the next GEMM."""
    bits, M, N, K = 8, 300, 520, 1040
    A, B, dA, dB, dC = _setup(bits, M, N, K, 41)
    n0 = L.lbgemm_launch_count()
    t = L.lbgemm_time_variants(bits, M, N, K, dA, dB, dC, warmup=1, reps=4, flush_l2=flush)
    assert len(t) == 9 and all(math.isfinite(x) and x > 0 for x in t), t
    # 9 variants x (1 warm-up + 4 reps) runs of two launches (re-encoding + GEMM)
    assert L.lbgemm_launch_count() - n0 == 9 * 5 * 2
    L.lbgemm_device_status()
    want = oracle.gemm(bits, A, B, K)
    assert np.array_equal(dC.cpu().numpy(), want)
    assert np.array_equal(G().gemm(bits, A, B, K), want)


@pytest.mark.parametrize("bits,M,N,K", [(8, 96, 3000, 1040), (1, 100, 70, 1024),
                                        (4, 130, 250, 514), (4, 130, 250, 512),
                                        (8, 8, 1000, 512)])
def test_every_candidate_is_exact(bits, M, N, K):
    """Each (route, param) the sweep times computes the oracle's product, via
    lbgemm_run_candidate and inside lbgemm_time_candidates."""
    A, B, dA, dB, dC = _setup(bits, M, N, K, 43 + M)
    want = oracle.gemm(bits, A, B, K)
    cands = L.lbgemm_candidates(bits, M, N, K)
    assert cands[:9] == [(L.ROUTE_TABLE, v) for v in range(9)]
    for r, p in cands:
        dC.fill_(-7)
        L.lbgemm_run_candidate(bits, M, N, K, dA, dB, dC, r, p)
        L.lbgemm_device_status()
        assert np.array_equal(dC.cpu().numpy(), want), (r, p)
    for i in range(0, len(cands), 6):  # interleaved timing of a few at a time
        dC.fill_(-7)
        t = L.lbgemm_time_candidates(bits, M, N, K, dA, dB, dC, cands[i:i + 6], warmup=0,
                                     reps=3)
        assert all(math.isfinite(x) and x > 0 for x in t)
        assert np.array_equal(dC.cpu().numpy(), want)


def test_dispatch_runs_the_measured_route():
    """A table entry's route replaces the shape rule for its exact shape."""
    dev = torch.device("cuda", torch.cuda.current_device())
    sm = torch.cuda.get_device_properties(dev).multi_processor_count
    M, N, K = 192, 2050, 1024  # rule: not the in-kernel conversion kernel
    A, B, dA, dB, dC = _setup(8, M, N, K, 47)
    want = oracle.gemm(8, A, B, K)
    saved = L.lbgemm_table_get_for(sm, 8, M, N, K)
    try:
        for route, param in [(L.ROUTE_FUSED, 256), (L.ROUTE_FUSED, 64), (L.ROUTE_WARPMMA, 0),
                             (L.ROUTE_SMALL, 0), (L.ROUTE_TABLE, 1)]:
            L.lbgemm_table_set_choice_for(sm, 8, M, N, K, 7, route, param)
            assert L.lbgemm_dispatch_for(sm, 8, M, N, K) == (route, param)
            dC.fill_(-7)
            L.lbgemm_run(8, M, N, K, dA, dB, dC)
            L.lbgemm_device_status()
            assert np.array_equal(dC.cpu().numpy(), want), (route, param)
        # misaligned operands cannot take an 8-bit route: the rules' kernel runs
        K2 = 1000  # K % 16 != 0
        A2, B2 = synth.operands(8, M, N, K2, 48)
        L.lbgemm_table_set_choice_for(sm, 8, M, N, K2, 7, L.ROUTE_TABLE, 2)
        assert np.array_equal(G().gemm(8, A2, B2, K2), oracle.gemm(8, A2, B2, K2))
    finally:
        if saved is None:
            L.lbgemm_table_set_choice_for(sm, 8, M, N, K, 7, -1, 0)
        else:
            L.lbgemm_table_set_choice_for(sm, 8, M, N, K, *saved)


def test_tuning_one_shape_stores_a_valid_entry():
    """The sweep step of one shape: its record is consistent and its entry
    makes lbgemm_run compute the exact product."""
    dev = torch.device("cuda", torch.cuda.current_device())
    sm = torch.cuda.get_device_properties(dev).multi_processor_count
    M, N, K = 128, 4096, 2048
    A, B, dA, dB, dC = _setup(8, M, N, K, 49)
    saved = L.lbgemm_table_get_for(sm, 8, M, N, K)
    try:
        recs = tune.sweep(L, 8, [(M, N, K)], dA, dB, dC, sm, reps=3, confirm_reps=4)
        r = recs[0]
        assert len(r["ms"]) == len(r["candidates"]) >= 9
        assert 0 <= r["label"] < 9
        assert r["pick"] in r["candidates"]
        entry = L.lbgemm_table_get_for(sm, 8, M, N, K)
        assert entry == (r["label"], r["pick"][0], r["pick"][1])
        dC.fill_(-7)
        L.lbgemm_run(8, M, N, K, dA, dB, dC)
        L.lbgemm_device_status()
        assert np.array_equal(dC.cpu().numpy(), oracle.gemm(8, A, B, K))
    finally:
        if saved is None:
            L.lbgemm_table_set_choice_for(sm, 8, M, N, K, 7, -1, 0)
        else:
            L.lbgemm_table_set_choice_for(sm, 8, M, N, K, *saved)


@pytest.mark.parametrize("bits", [8, 4, 1])
def test_every_compiled_tile_and_stage_count_is_exact(bits):
    """lbgemm_run_tile: the nine variants and the large tile's 2- and 3-stage
    kernels (measurement only), on a ragged shape, a split-K shape and a
    shape of more than one wave of small and medium tiles."""
    for i, (M, N, K) in enumerate([(300, 200, 1040), (129, 65, 4160), (2500, 2000, 1040)]):
        if bits == 1:
            K = (K + 31) // 32 * 32
        A, B, dA, dB, dC = _setup(bits, M, N, K, 61 + i + bits)
        want = oracle.gemm(bits, A, B, K)
        for tile in range(3):
            for stages in range(2, 7 if tile == 2 else 5):
                dC.fill_(-7)
                L.lbgemm_run_tile(bits, M, N, K, dA, dB, dC, tile, stages)
                L.lbgemm_device_status()
                assert np.array_equal(dC.cpu().numpy(), want), (bits, M, N, K, tile, stages)
    with pytest.raises(L.LbgemmError) as e:
        L.lbgemm_run_tile(bits, 64, 64, 256, dA, dB, dC, 1, 5)
    assert e.value.status == L.ERR_UNSUPPORTED


def test_small_dp4a_on_nibbles():
    """The one-launch dp4a kernel on packed 4-bit operands: ragged tiles, one
    16-byte K chunk, K tails inside a 64-byte stage, extremes and a mixed
    pattern, bit-exact."""
    for i, (M, N, K) in enumerate([(1, 1, 32), (65, 70, 32), (130, 250, 96), (64, 64, 128),
                                   (300, 200, 1024), (1000, 17, 2016), (77, 513, 4096)]):
        A, B = synth.operands(4, M, N, K, 2100 + i)
        dA, dB = G().to_dev(A), G().to_dev(B)
        dC = torch.full((M, N), -7, dtype=torch.int32, device="cuda")
        L.lbgemm_run_candidate(4, M, N, K, dA, dB, dC, L.ROUTE_SMALL, 0)
        L.lbgemm_device_status()
        want = oracle.gemm(4, A, B, K)
        assert np.array_equal(dC.cpu().numpy(), want), (M, N, K)
    K = 4096
    A = np.full((40, K // 2), 0x88, np.uint8)  # every nibble -8
    B = np.full((30, K // 2), 0x88, np.uint8)
    dC = torch.empty((40, 30), dtype=torch.int32, device="cuda")
    L.lbgemm_run_candidate(4, 40, 30, K, G().to_dev(A), G().to_dev(B), dC, L.ROUTE_SMALL, 0)
    assert np.all(dC.cpu().numpy() == 64 * K)
    A = np.full((40, K // 2), 0x78, np.uint8)  # low nibble -8, high nibble 7
    B = np.full((30, K // 2), 0x87, np.uint8)  # low 7, high -8
    L.lbgemm_run_candidate(4, 40, 30, K, G().to_dev(A), G().to_dev(B), dC, L.ROUTE_SMALL, 0)
    assert np.all(dC.cpu().numpy() == oracle.gemm(4, A, B, K))
    assert np.all(dC.cpu().numpy() == -112 * K // 2 * 1)
