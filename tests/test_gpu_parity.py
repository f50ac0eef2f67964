"""GPU parity: the library's CUDA kernels against the CPU oracle, element by
element, through the C ABI.  Integer results must be bit-exact; the bf16
linear layer must be within 1e-2 relative of the fp64 oracle per element
(fp32 scaling adds at most a few ulp, bf16 rounding at most 2^-9 relative)
and exactly zero where the exact accumulator is zero."""
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
    yield


def G():
    import gpu_util  # noqa: PLC0415
    return gpu_util


def assert_exact(got, want, what):
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        m, n = bad[0]
        raise AssertionError(f"{what}: {len(bad)} entries differ; first at ({m},{n}): "
                             f"got {got[m, n]} want {want[m, n]}")


# ---- 8-bit ---------------------------------------------------------------------

def test_int8_256_cube_config():
    """The 256^3 int8 workload, seeded like the benchmark, default dispatch."""
    A, B = synth.operands(8, 256, 256, 256, synth.config_seed(1))
    assert_exact(G().gemm(8, A, B, 256), oracle.gemm(8, A, B, 256), "int8 256^3")


SHAPES_8 = [(256, 256, 256), (300, 200, 136), (129, 65, 1000), (128, 512, 2048), (1, 1, 1),
            (17, 333, 24), (257, 129, 4104)]


@pytest.mark.parametrize("variant", range(9))
def test_int8_every_variant(variant):
    for i, (M, N, K) in enumerate(SHAPES_8):
        A, B = synth.operands(8, M, N, K, 100 + i)
        assert_exact(G().gemm(8, A, B, K, variant), oracle.gemm(8, A, B, K),
                     f"int8 variant {variant} {M}x{N}x{K}")


@pytest.mark.parametrize("M", [1, 2, 5, 16])
def test_int8_skinny_path(M):
    for N, K in [(1000, 4096), (37, 16), (11008, 512)]:
        A, B = synth.operands(8, M, N, K, 7 * M + N)
        assert_exact(G().gemm(8, A, B, K), oracle.gemm(8, A, B, K), f"int8 skinny {M}x{N}x{K}")


def test_int8_small_dp4a_path():
    """Default dispatch of small problems (K <= 512, M*N*K <= 2^28): the
    one-launch dp4a kernel (K <= 256, or both sides above 256 rows), with
    ragged M, N and K tails; with a side of at most 256 rows and K > 256 the
    warp-MMA kernel."""
    for M, N, K in [(17, 19, 16), (64, 64, 64), (100, 300, 144), (1000, 250, 512), (65, 4000, 32),
                    (300, 1000, 512), (257, 260, 272)]:
        A, B = synth.operands(8, M, N, K, 13 * M + K)
        assert_exact(G().gemm(8, A, B, K), oracle.gemm(8, A, B, K), f"int8 small {M}x{N}x{K}")
    for rows in (40, 300):
        A = np.full((rows, 512), -128, np.int8)
        assert np.all(G().gemm(8, A, A, 512) == 16384 * 512)


@pytest.mark.parametrize("M,N,K", [(64, 4096, 2048), (200, 2500, 2064), (4096, 100, 4096),
                                   (3000, 256, 2064), (17, 2048, 4096), (500, 1100, 4096),
                                   (1030, 512, 3008), (100, 9000, 1040), (8200, 400, 1024),
                                   (512, 4096, 512), (300, 5000, 1024), (64, 8192, 2048),
                                   (400, 8192, 2048), (1100, 200, 8192)])
def test_int8_fused_conversion_path(M, N, K):
    """Default dispatch of problems with one side <= 512, the other >= 1024
    and K >= 512 in the conversion kernel's domain (large side >= 4096, or
    K >= 8192, or large side >= 2048 with K >= 4096, or small side <= 256
    with K >= 2048): the kernel converts the large int8 operand itself (B
    when N >= M, giving C transposed from the accumulator), on 64-, 128- or
    256-wide tiles; ragged tiles and K tails included."""
    A, B = synth.operands(8, M, N, K, 7 * M + N + K)
    assert_exact(G().gemm(8, A, B, K), oracle.gemm(8, A, B, K), f"int8 fused {M}x{N}x{K}")


# (M, N, K): both orientations, ragged rows and columns, K that ends inside a
# 64-element slice, odd slice counts, a last group of 1-3 slices, chunk
# boundaries (1024), few tiles (split K), one tile
FUSED_SHAPES = [(300, 520, 1040), (520, 300, 1040), (129, 4100, 2048), (4100, 129, 2112),
                (130, 70, 48), (16, 300, 4160), (257, 513, 1024), (700, 900, 4096),
                (100, 1100, 16384), (1, 1, 16), (256, 256, 3008)]


@pytest.mark.parametrize("slice_k", [0, 128, 256])
@pytest.mark.parametrize("tile_n", [64, 128, 256])
def test_int8_fused_every_tile(tile_n, slice_k):
    """lbgemm_run_fused with each tile width (64 and 128: double-buffered
    accumulators, K slices of 128 or 256 elements; 256: one accumulator, K in
    groups of 4 slices of 64)."""
    try:
        L.lbgemm_set_fused_slice(slice_k)
        for i, (M, N, K) in enumerate(FUSED_SHAPES):
            A, B = synth.operands(8, M, N, K, 900 + 17 * i + tile_n)
            assert_exact(G().fused(A, B, K, tile_n), oracle.gemm(8, A, B, K),
                         f"fused tile {tile_n} slice {slice_k} {M}x{N}x{K}")
    finally:
        L.lbgemm_set_fused_slice(0)


@pytest.mark.parametrize("tile_n", [64, 128, 256])
def test_int8_fused_extremes(tile_n):
    """Every value -128 (chunk sums exactly 2^24) and the adversarial order
    of large then +-1 products, on the in-kernel conversion."""
    K = 4096
    A = np.full((200, K), -128, np.int8)
    B = np.full((300, K), -128, np.int8)
    assert np.all(G().fused(A, B, K, tile_n) == 16384 * K)
    A = np.ones((128, K), np.int8)
    B = np.ones((64, K), np.int8)
    A[:, :511] = -128
    B[:, :511] = -128
    A[:, 1024:2047] = -128
    B[:, 1024:2047] = -128
    B[1::2, 600:1000] = -1
    assert_exact(G().fused(A, B, K, tile_n), oracle.gemm(8, A, B, K), "fused adversarial")
    assert_exact(G().fused(B, A, K, tile_n), oracle.gemm(8, B, A, K), "fused adversarial (T)")


@pytest.mark.parametrize("tile_n", [64, 128])
def test_int8_fused_stream_k(tile_n):
    """Stream-K forced on the 64/128-wide conversion kernels: every CTA takes
    an equal run of the tile-major K slices, cut at tile ends, the pieces of a
    tile added into C.  B converted (C written transposed by atomics) and A
    converted (TMA reduce-adds), ragged tiles, K not a multiple of the slice;
    bit-exact.  The linear layer on the same schedule (int32 sums, then the
    scaling grid) within 1e-2."""
    L.lbgemm_set_fused_stream_k(1)
    try:
        assert L.lbgemm_get_fused_stream_k() == 1
        for i, (M, N, K) in enumerate([(64, 4100, 4096), (4096, 100, 2064), (200, 3000, 1040),
                                       (33, 16384, 1024)]):
            A, B = synth.operands(8, M, N, K, 2100 + i)
            dC = torch.full((M, N), -7, dtype=torch.int32, device="cuda")
            L.lbgemm_run_candidate(8, M, N, K, G().to_dev(A), G().to_dev(B), dC, L.ROUTE_FUSED,
                                   tile_n)
            L.lbgemm_device_status()
            assert_exact(dC.cpu().numpy(), oracle.gemm(8, A, B, K),
                         f"stream-K tile {tile_n} {M}x{N}x{K}")
        for i, (M, N, K) in enumerate([(100, 4096, 4096), (40, 11008, 2048)]):
            X, sx, W, sw = synth.linear_operands(M, N, K, 2200 + i)
            X[1, :] = 0
            dY = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
            L.lbgemm_linear_candidate(M, N, K, G().to_dev(X), G().to_dev(sx), G().to_dev(W),
                                      G().to_dev(sw), dY, L.ROUTE_FUSED, tile_n)
            L.lbgemm_device_status()
            got = dY.float().cpu().numpy().astype(np.float64)
            check_linear(got, oracle.linear(X, sx, W, sw), oracle.gemm(8, X, W, K) == 0,
                         f"stream-K linear tile {tile_n} {M}x{N}x{K}")
    finally:
        L.lbgemm_set_fused_stream_k(0)


def test_int8_fused_short_chunks():
    """A shorter exact chunk (512 elements) changes where the accumulator is
    read out; the result must not change."""
    M, N, K = 200, 1500, 5120
    A, B = synth.operands(8, M, N, K, 31)
    want = oracle.gemm(8, A, B, K)
    try:
        L.lbgemm_set_exact_chunk(8, 512)
        for tile_n in (64, 256):
            assert_exact(G().fused(A, B, K, tile_n), want, f"fused chunk 512 tile {tile_n}")
        L.lbgemm_set_fused_slice(256)
        for tile_n in (64, 128):
            assert_exact(G().fused(A, B, K, tile_n), want, f"fused chunk 512 slice 256 {tile_n}")
    finally:
        L.lbgemm_set_exact_chunk(8, 1024)
        L.lbgemm_set_fused_slice(0)


@pytest.mark.parametrize("tile_n", [64, 128])
def test_int8_fused_slice_256_extremes(tile_n):
    """256-element slices: every value -128 and the adversarial order."""
    try:
        L.lbgemm_set_fused_slice(256)
        K = 4096
        A = np.full((200, K), -128, np.int8)
        B = np.full((300, K), -128, np.int8)
        assert np.all(G().fused(A, B, K, tile_n) == 16384 * K)
        A = np.ones((128, K), np.int8)
        B = np.ones((64, K), np.int8)
        A[:, :511] = -128
        B[:, :511] = -128
        A[:, 1024:2047] = -128
        B[:, 1024:2047] = -128
        B[1::2, 600:1000] = -1
        assert_exact(G().fused(A, B, K, tile_n), oracle.gemm(8, A, B, K), "slice 256 adversarial")
        assert_exact(G().fused(B, A, K, tile_n), oracle.gemm(8, B, A, K), "slice 256 adv. (T)")
        # the linear layer through the same kernel
        X, sx, W, sw = synth.linear_operands(128, 2100, 4096, 640)
        ref = oracle.linear(X, sx, W, sw)
        acc = oracle.gemm(8, X, W, 4096)
        check_linear(G().linear(X, sx, W, sw), ref, acc == 0, "linear fused slice 256")
    finally:
        L.lbgemm_set_fused_slice(0)


# (M, N, K): small side 1..32 on either operand, ragged W tiles (N % 16 != 0),
# K of one 16-byte piece, K ending inside a 256-element step, the K limits
WARPMMA_SHAPES = [(1, 1000, 4096), (5, 77, 16), (16, 300, 1040), (32, 4100, 2048),
                  (20, 1000, 2048), (300, 16, 1040), (4100, 30, 2000), (32, 32, 128),
                  (17, 11008, 576), (16, 9, 4224), (3, 5000, 4224), (30, 700, 2048),
                  (7, 300, 4160), (9, 1000, 272), (1, 1, 16),
                  # more than 32 rows on the small side: several row blocks of 32
                  (33, 1000, 512), (64, 1024, 1024), (100, 700, 2048), (1500, 128, 1040),
                  (256, 256, 64), (200, 3000, 16)]


def test_int8_warpmma_forced():
    """lbgemm_run_warpmma on every shape class it takes."""
    for i, (M, N, K) in enumerate(WARPMMA_SHAPES):
        A, B = synth.operands(8, M, N, K, 1300 + i)
        assert_exact(G().warpmma(A, B, K), oracle.gemm(8, A, B, K), f"warp-MMA {M}x{N}x{K}")


def test_int8_warpmma_extremes():
    """Every value -128 (int32 sums at 16384 K), the adversarial order of
    large then +-1 products, and a shorter exact chunk."""
    for K in (1024, 4096):
        A = np.full((16, K), -128, np.int8)
        B = np.full((100, K), -128, np.int8)
        assert np.all(G().warpmma(A, B, K) == 16384 * K)
        assert np.all(G().warpmma(B[:20], A, K) == 16384 * K)
    K = 4096
    A = np.ones((16, K), np.int8)
    B = np.ones((64, K), np.int8)
    A[:, :511] = -128
    B[:, :511] = -128
    A[:, 1024:2047] = -128
    B[:, 1024:2047] = -128
    B[1::2, 600:1000] = -1
    assert_exact(G().warpmma(A, B, K), oracle.gemm(8, A, B, K), "warp-MMA adversarial")
    try:
        L.lbgemm_set_exact_chunk(8, 512)
        assert_exact(G().warpmma(A, B, K), oracle.gemm(8, A, B, K), "warp-MMA chunk 512")
    finally:
        L.lbgemm_set_exact_chunk(8, 1024)


@pytest.mark.parametrize("M,N,K", [(8, 2000, 1024), (32, 700, 2048), (2000, 24, 512),
                                   (3000, 5, 64), (64, 1024, 1024), (4096, 128, 2048),
                                   (250, 2000, 1040), (16000, 64, 512)])
def test_int8_warpmma_dispatch(M, N, K):
    """Default dispatch of problems with a side of 5..32 rows, and of small
    problems with a side of up to 256 rows (M*N <= 2^19, K <= 2048)."""
    A, B = synth.operands(8, M, N, K, 11 * M + N)
    assert_exact(G().gemm(8, A, B, K), oracle.gemm(8, A, B, K), f"int8 warp-MMA {M}x{N}x{K}")


# (M, N, K): one tile, ragged tiles, K tails, a single K slice per tile, more
# pieces than K slices allow, N % 4 != 0 (no splits), and more than one wave
# of tiles on every tile class (2500 x 2000: 80 large, 320 medium, 640 small)
TAIL_SHAPES = [(256, 256, 256), (300, 200, 136), (1000, 1000, 2064), (129, 65, 4104),
               (2048, 520, 1024), (700, 900, 8192), (64, 64, 64), (100, 203, 1000),
               (2500, 2000, 1040)]


@pytest.mark.parametrize("variant", range(9))
def test_int8_tail_split_forced(variant):
    """Mode 2 on every tile x stage variant: the tiles of the last wave cut
    into K pieces added into C, the tiles before them stored whole (C starts
    filled with -7, so a piece outside the cleared part shows)."""
    try:
        L.lbgemm_set_tail_split(2)
        for i, (M, N, K) in enumerate(TAIL_SHAPES):
            A, B = synth.operands(8, M, N, K, 1700 + 13 * i + variant)
            assert_exact(G().gemm(8, A, B, K, variant), oracle.gemm(8, A, B, K),
                         f"tail split variant {variant} {M}x{N}x{K}")
    finally:
        L.lbgemm_set_tail_split(1)


def test_tail_split_modes_widths_and_chunks():
    """The default mode on shapes with one or more whole waves and a small
    last wave (2560 x 2048 and a ragged 2500 x 2000, every variant), mode 0
    on the same, mode 2 on the 4-bit and 1-bit (e4m3) kernels and with a
    shorter exact chunk."""
    for M, N, K in [(2560, 2048, 1024), (2500, 2000, 1040)]:
        A, B = synth.operands(8, M, N, K, 1960 + M)
        want = oracle.gemm(8, A, B, K)
        for variant in range(9):
            assert_exact(G().gemm(8, A, B, K, variant), want,
                         f"tail split (default mode) v{variant} {M}x{N}x{K}")
        try:
            L.lbgemm_set_tail_split(0)
            for variant in (1, 7):
                assert_exact(G().gemm(8, A, B, K, variant), want, f"mode 0 v{variant}")
        finally:
            L.lbgemm_set_tail_split(1)
    try:
        L.lbgemm_set_tail_split(2)
        for bits, M, N, K in [(4, 700, 900, 8192), (4, 129, 300, 1000), (1, 500, 260, 20000),
                              (1, 129, 65, 4000), (4, 2500, 2000, 1024)]:
            A, B = synth.operands(bits, M, N, K, 1900 + M)
            want = oracle.gemm(bits, A, B, K)
            for variant in (1, 4, 7):
                assert_exact(G().gemm(bits, A, B, K, variant), want,
                             f"tail split bits {bits} variant {variant} {M}x{N}x{K}")
        L.lbgemm_set_exact_chunk(8, 512)
        M, N, K = 2500, 2000, 3008
        A, B = synth.operands(8, M, N, K, 1950)
        want = oracle.gemm(8, A, B, K)
        for variant in (2, 5, 8):
            assert_exact(G().gemm(8, A, B, K, variant), want, f"tail split chunk 512 v{variant}")
    finally:
        L.lbgemm_set_exact_chunk(8, 1024)
        L.lbgemm_set_tail_split(1)


def test_int8_full_range_and_extremes():
    g = np.random.default_rng(5)
    M, N, K = 130, 70, 3000
    A = g.integers(-128, 128, (M, K)).astype(np.int8)
    B = g.integers(-128, 128, (N, K)).astype(np.int8)
    A[0] = -128
    B[0] = -128
    B[1] = 127
    assert_exact(G().gemm(8, A, B, K, 7), oracle.gemm(8, A, B, K), "int8 full range")


def test_int8_max_k_all_min():
    """K = 131071 with every value -128: C = 16384 K = 2147467264, the largest
    result the 8-bit path accepts; every chunk and the int32 sum are at their
    limits."""
    K = 131071
    A = np.full((3, K), -128, np.int8)
    B = np.full((2, K), -128, np.int8)
    C = G().gemm(8, A, B, K, 1)
    assert np.all(C == 16384 * K)


def test_int8_exact_accumulation_adversarial():
    """Large products first, then +-1 terms: a truncating fp32 sum would drop
    the small terms.  The per-chunk magnitude reaches 2^23 + 2^9 and, in the
    second chunk, 2^24 - 2^14 + 1."""
    K = 4096
    A = np.ones((128, K), np.int8)
    B = np.ones((64, K), np.int8)
    A[:, :511] = -128
    B[:, :511] = -128
    A[:, 1024:2047] = -128
    B[:, 1024:2047] = -128
    B[1::2, 600:1000] = -1
    assert_exact(G().gemm(8, A, B, K, 4), oracle.gemm(8, A, B, K), "int8 adversarial")


def test_int8_workspace_entry_matches():
    M, N, K = 200, 300, 520
    A, B = synth.operands(8, M, N, K, 77)
    need = L.lbgemm_workspace_size(8, M, N, K)
    ws = torch.empty(need, dtype=torch.uint8, device=G().DEV)
    dC = torch.empty((M, N), dtype=torch.int32, device=G().DEV)
    L.lbgemm_run_ws(8, M, N, K, G().to_dev(A), G().to_dev(B), dC, 5, ws, need)
    L.lbgemm_device_status()
    assert_exact(dC.cpu().numpy(), oracle.gemm(8, A, B, K), "int8 run_ws")
    with pytest.raises(L.LbgemmError) as e:
        L.lbgemm_run_ws(8, M, N, K, G().to_dev(A), G().to_dev(B), dC, 5, ws, need - 1)
    assert e.value.status == L.ERR_WORKSPACE


@pytest.mark.parametrize("bits", [8, 4, 1])
def test_encode_then_run_encoded(bits):
    """lbgemm_encode + lbgemm_run_encoded (operands kept re-encoded, e.g.
    weights): the table's variant and forced ones, few tiles (split K: C is
    cleared by a memset here, there being no encoder launch), ragged shapes,
    and a forced split of the last wave."""
    Ks = {8: (1000, 4104), 4: (1002, 4096), 1: (1024, 8192)}[bits]
    for i, (M, N) in enumerate([(300, 200), (129, 65), (2500, 2000)]):
        K = Ks[i % 2]
        A, B = synth.operands(bits, M, N, K, 60 + 7 * i + bits)
        want = oracle.gemm(bits, A, B, K)
        for variant in (-1, 1, 7):
            assert_exact(G().encoded(bits, A, B, K, variant), want,
                         f"encoded bits {bits} v{variant} {M}x{N}x{K}")
    try:
        L.lbgemm_set_tail_split(2)
        M, N, K = 2500, 2000, Ks[0]
        A, B = synth.operands(bits, M, N, K, 90 + bits)
        want = oracle.gemm(bits, A, B, K)
        for variant in (2, 5, 8):
            assert_exact(G().encoded(bits, A, B, K, variant), want,
                         f"encoded tail split bits {bits} v{variant}")
    finally:
        L.lbgemm_set_tail_split(1)


def test_int8_host_buffers():
    M, N, K = 96, 160, 640
    A, B = synth.operands(8, M, N, K, 78)
    C = np.zeros((M, N), np.int32)
    L.lbgemm_run_host(8, M, N, K, A, B, C, -1, 0)
    assert_exact(C, oracle.gemm(8, A, B, K), "int8 host buffers")


@pytest.mark.parametrize("bits,M,N,K", [(8, 4500, 4000, 256), (8, 20000, 64, 4096),
                                        (8, 9000, 4000, 64),
                                        (8, 300, 9000, 1024), (8, 2000, 2100, 512),
                                        (4, 4500, 4000, 128), (4, 300, 6000, 4096),
                                        (1, 5000, 4000, 64), (1, 300, 9000, 8192)])
def test_host_buffers_in_blocks(bits, M, N, K):
    """Problems that copy more than 8 MB run in blocks of the larger side
    (copies in and out on their own streams, overlapping the blocks' GEMMs):
    row blocks and column blocks (C out by 2-D copies), ragged last blocks,
    the block count at its cap (9000 x 4000 x 64: 144 MB of copies in twelve
    blocks of 768 rows), a large A with a small C, and every bit width."""
    A, B = synth.operands(bits, M, N, K, 80 + bits)
    C = np.zeros((M, N), np.int32)
    L.lbgemm_run_host(bits, M, N, K, A, B, C, -1, 0)
    assert_exact(C, oracle.gemm(bits, A, B, K), f"host buffers bits {bits} {M}x{N}x{K}")


# ---- 4-bit ---------------------------------------------------------------------

SHAPES_4 = [(256, 256, 256), (300, 200, 138), (129, 65, 1000), (128, 512, 4096), (3, 5, 2)]


@pytest.mark.parametrize("variant", range(9))
def test_int4_every_variant(variant):
    for i, (M, N, K) in enumerate(SHAPES_4):
        A, B = synth.operands(4, M, N, K, 200 + i)
        assert_exact(G().gemm(4, A, B, K, variant), oracle.gemm(4, A, B, K),
                     f"int4 variant {variant} {M}x{N}x{K}")


def test_int4_extremes_long_k():
    K = 65536
    A = np.full((2, K // 2), 0x88, np.uint8)   # all -8
    B = np.full((3, K // 2), 0x88, np.uint8)
    B[1] = 0x77                                # all 7
    C = G().gemm(4, A, B, K)
    assert np.all(C[:, 0] == 64 * K) and np.all(C[:, 1] == -56 * K) and np.all(C[:, 2] == 64 * K)


# ---- 1-bit ---------------------------------------------------------------------

SHAPES_1 = [(64, 64, 1024), (100, 70, 4096), (129, 257, 96), (5, 3, 32), (200, 130, 65536)]


@pytest.mark.parametrize("variant", range(9))
def test_b1_every_variant(variant):
    for i, (M, N, K) in enumerate(SHAPES_1):
        A, B = synth.operands(1, M, N, K, 300 + i)
        assert_exact(G().gemm(1, A, B, K, variant), oracle.gemm(1, A, B, K),
                     f"b1 variant {variant} {M}x{N}x{K}")


@pytest.mark.parametrize("variant", range(9))
def test_b1_popc_every_variant(variant):
    """The XOR-popcount CUDA-core kernel, each of its tile x stage variants."""
    for i, (M, N, K) in enumerate(SHAPES_1):
        A, B = synth.operands(1, M, N, K, 300 + i)
        dC = torch.full((M, N), -7, dtype=torch.int32, device=G().DEV)
        L.lbgemm_run_popc(M, N, K, G().to_dev(A), G().to_dev(B), dC, variant)
        L.lbgemm_device_status()
        assert_exact(dC.cpu().numpy(), oracle.gemm(1, A, B, K), f"b1 popc v{variant} {M}x{N}x{K}")


def test_b1_auto_routes():
    """Default dispatch: small problems on the popcount kernel, large ones on
    the tensor cores; both exact."""
    for M, N, K in [(64, 64, 1024), (256, 256, 32768)]:
        A, B = synth.operands(1, M, N, K, M + K)
        assert_exact(G().gemm(1, A, B, K), oracle.gemm(1, A, B, K), f"b1 auto {M}x{N}x{K}")


def test_b1_closed_forms():
    K = 4096
    g = np.random.default_rng(9)
    A = g.integers(0, 1 << 32, (40, K // 32), dtype=np.uint64).astype(np.uint32)
    B = np.concatenate([A, ~A])
    C = G().gemm(1, A, B, K)
    assert np.all(np.diag(C[:, :40]) == K) and np.all(np.diag(C[:, 40:]) == -K)


# ---- linear layer -----------------------------------------------------------------

def check_linear(Y, ref, acc_zero, what):
    assert np.all(np.isfinite(Y)), what
    err = np.abs(Y - ref)
    tol = LINEAR_RTOL * np.abs(ref)
    bad = err > tol
    assert not bad.any(), f"{what}: {bad.sum()} entries beyond 1e-2 relative"
    assert np.all(Y[acc_zero] == 0), f"{what}: nonzero output where the accumulator is zero"


@pytest.mark.parametrize("M", [1, 16, 128, 200, 40])
def test_linear_small(M):
    N, K = 1000, 4096
    X, sx, W, sw = synth.linear_operands(M, N, K, 400 + M)
    X[0, :] = 0  # an all-zero token gives exact zeros
    ref = oracle.linear(X, sx, W, sw)
    acc = oracle.gemm(8, X, W, K)
    check_linear(G().linear(X, sx, W, sw), ref, acc == 0, f"linear M={M}")


@pytest.mark.parametrize("M", [5, 16, 32])
def test_linear_warpmma_route(M):
    """Token counts 5..32: the warp-level fp16 MMA kernel, Y scaled in its
    final reduction."""
    N, K = 2100, 4096 if M <= 16 else 2048
    X, sx, W, sw = synth.linear_operands(M, N, K, 700 + M)
    X[1, :] = 0
    ref = oracle.linear(X, sx, W, sw)
    acc = oracle.gemm(8, X, W, K)
    check_linear(G().linear(X, sx, W, sw), ref, acc == 0, f"linear warp-MMA M={M}")


@pytest.mark.parametrize("M,N,K", [(33, 2100, 4096), (128, 2100, 4096), (300, 2100, 4096),
                                   (450, 8200, 2048), (40, 2102, 4096), (128, 11008, 4096),
                                   (400, 8200, 8192)])
def test_linear_fused_route(M, N, K):
    """Token counts 33..512 in the conversion kernel's domain: the weights are
    converted in the kernel and Y is written transposed from the accumulator
    (64- and 128-wide tiles by the dispatch, also past 384 tokens at K = 8192;
    CTA pairs forced with 400 and 450 tokens;
    N % 4 != 0 included)."""
    X, sx, W, sw = synth.linear_operands(M, N, K, 600 + M)
    X[1, :] = 0
    ref = oracle.linear(X, sx, W, sw)
    acc = oracle.gemm(8, X, W, K)
    check_linear(G().linear(X, sx, W, sw), ref, acc == 0, f"linear fused M={M}")
    if M > 384:
        dY = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=G().DEV)
        L.lbgemm_linear_candidate(M, N, K, G().to_dev(X), G().to_dev(sx), G().to_dev(W),
                                  G().to_dev(sw), dY, L.ROUTE_FUSED, 256)
        L.lbgemm_device_status()
        got = dY.float().cpu().numpy().astype(np.float64)
        check_linear(got, ref, acc == 0, f"linear fused pairs M={M}")


@pytest.mark.parametrize("tile", [64, 128])
@pytest.mark.parametrize("M,N,K", [(24, 4096, 4096), (64, 4096, 4096), (100, 2102, 4096),
                                   (17, 11008, 4096), (200, 1030, 8192), (64, 1000, 512),
                                   (100, 2102, 1040)])
def test_linear_fused_split_k(tile, M, N, K):
    """The conversion kernel's linear layer, K split over CTAs where the
    unsplit grid would leave most SMs idle: partial sums added into an int32
    workspace, then scaled into Y by a second grid (ragged tiles of W rows and
    tokens; N % 4 != 0 on the scalar scaling path; a K with a ragged last
    slice); unsplit where the split would not pay (11008 rows, 512-long K).  A second call right after the
    first must not see the first one's sums."""
    for rep in range(2):
        X, sx, W, sw = synth.linear_operands(M, N, K, 610 + M + 7 * rep)
        X[1, :] = 0
        ref = oracle.linear(X, sx, W, sw)
        acc = oracle.gemm(8, X, W, K)
        dY = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=G().DEV)
        L.lbgemm_linear_candidate(M, N, K, G().to_dev(X), G().to_dev(sx), G().to_dev(W),
                                  G().to_dev(sw), dY, L.ROUTE_FUSED, tile)
        L.lbgemm_device_status()
        got = dY.float().cpu().numpy().astype(np.float64)
        check_linear(got, ref, acc == 0, f"linear split-K tile {tile} {M}x{N}x{K} call {rep}")


@pytest.mark.parametrize("slice_k", [128, 256])
@pytest.mark.parametrize("M,N,K", [(128, 2100, 4096), (200, 1030, 8192), (192, 4100, 2064),
                                   (300, 9800, 1040)])
def test_linear_fused_slice_forced(slice_k, M, N, K):
    """The 128-wide conversion kernel's linear layer with either K slice
    forced (256 elements is its default for the linear layer, 128 for the
    GEMM): whole tiles, split and stream-K schedules, a ragged last slice."""
    X, sx, W, sw = synth.linear_operands(M, N, K, 680 + M + slice_k)
    X[2, :] = 0
    ref = oracle.linear(X, sx, W, sw)
    acc = oracle.gemm(8, X, W, K)
    L.lbgemm_set_fused_slice(slice_k)
    try:
        dY = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=G().DEV)
        L.lbgemm_linear_candidate(M, N, K, G().to_dev(X), G().to_dev(sx), G().to_dev(W),
                                  G().to_dev(sw), dY, L.ROUTE_FUSED, 128)
        L.lbgemm_device_status()
    finally:
        L.lbgemm_set_fused_slice(0)
    got = dY.float().cpu().numpy().astype(np.float64)
    check_linear(got, ref, acc == 0, f"linear slice {slice_k} {M}x{N}x{K}")


def test_linear_fused_split_k_extremes():
    """Sums of K products of -128 x -128 (2^14 each) summed over K pieces in
    int32: 16384 * 8192 = 2^27, exact in the workspace and in fp32."""
    M, N, K = 40, 4096, 8192
    X = np.full((M, K), -128, np.int8)
    W = np.full((N, K), -128, np.int8)
    W[::3] = 127
    sx = np.full(M, 2.0 ** -20, np.float32)
    sw = np.full(N, 0.5, np.float32)
    dY = torch.empty((M, N), dtype=torch.bfloat16, device=G().DEV)
    L.lbgemm_linear_candidate(M, N, K, G().to_dev(X), G().to_dev(sx), G().to_dev(W),
                              G().to_dev(sw), dY, L.ROUTE_FUSED, 64)
    L.lbgemm_device_status()
    got = dY.float().cpu().numpy().astype(np.float64)
    ref = oracle.linear(X, sx, W, sw)
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("variant", [0, 4, 8])
def test_linear_variants(variant):
    M, N, K = 160, 520, 1024
    X, sx, W, sw = synth.linear_operands(M, N, K, 500 + variant)
    ref = oracle.linear(X, sx, W, sw)
    acc = oracle.gemm(8, X, W, K)
    check_linear(G().linear(X, sx, W, sw, variant), ref, acc == 0, f"linear v{variant}")


# ---- quantised activations ------------------------------------------------------

def _bf16_rows(M, K, seed):
    g = np.random.default_rng(seed)
    x = (g.standard_normal((M, K)) * g.uniform(0.05, 20, (M, 1))).astype(np.float32)
    x[min(1, M - 1)] = 0.0  # a zero row
    xt = torch.from_numpy(x).to(torch.bfloat16)
    return xt, xt.float().numpy()  # the exact values the GPU reads


@pytest.mark.parametrize("M,K", [(37, 4096), (5, 100), (130, 1000), (1, 8), (1100, 264),
                                 (8200, 40), (8195, 30)])
def test_quantize_rows_bit_exact(M, K):
    """Eight warps per row up to 8192 rows, one warp per row beyond (with a
    ragged last block); 16-byte loads when K % 8 == 0, else one element per
    thread."""
    xt, xf = _bf16_rows(M, K, M + K)
    Q = torch.empty((M, K), dtype=torch.int8, device=G().DEV)
    S = torch.empty(M, dtype=torch.float32, device=G().DEV)
    L.lbgemm_quantize_rows(M, K, xt.to(G().DEV), Q, S)
    L.lbgemm_device_status()
    q, s = oracle.quantize_rows(xf)
    np.testing.assert_array_equal(S.cpu().numpy(), s)
    assert_exact(Q.cpu().numpy(), q, f"quantize {M}x{K}")


@pytest.mark.parametrize("M", [1, 16, 128, 300])
def test_linear_quant(M):
    N, K = 1024, 4096
    xt, xf = _bf16_rows(M, K, 600 + M)
    g = np.random.default_rng(M)
    W = g.integers(-127, 128, (N, K)).astype(np.int8)
    sw = (g.random(N) * 0.01).astype(np.float32)
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=G().DEV)
    L.lbgemm_linear_quant(M, N, K, xt.to(G().DEV), G().to_dev(W), G().to_dev(sw), Y)
    L.lbgemm_device_status()
    ref = oracle.linear_quant(xf, W, sw)
    q, s = oracle.quantize_rows(xf)
    check_linear(Y.float().cpu().numpy().astype(np.float64), ref, oracle.gemm(8, q, W, K) == 0,
                 f"linear_quant M={M}")


# ---- status word ------------------------------------------------------------------

def test_wait_timeout_is_reported_and_recovers():
    """A wait that nothing signals gives up after its limit: the status word
    reports the time-out once, and the next GEMM runs and is exact."""
    L.lbgemm_device_status()
    L.lbgemm_selftest_timeout()
    with pytest.raises(L.LbgemmError) as e:
        L.lbgemm_device_status()
    assert e.value.status == L.ERR_TIMEOUT
    L.lbgemm_device_status()  # cleared
    A, B = synth.operands(8, 130, 70, 300, 4242)
    assert_exact(G().gemm(8, A, B, 300, 7), oracle.gemm(8, A, B, 300), "after time-out")


def test_device_status_clean_after_runs():
    L.lbgemm_device_status()
    assert L.lbgemm_launch_count() > 0
