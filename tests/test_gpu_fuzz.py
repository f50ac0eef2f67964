"""GPU parity on seeded random shapes through the default dispatch.

The other parity tests pin each kernel and each shape rule on chosen shapes;
here the shapes are drawn at random (sides log-uniform from 1 to ~6000, K
log-uniform up to 16384 with the bit width's alignment, 8-bit K also
unaligned), so that every boundary between the routes, and ragged tiles of
every kernel the dispatch reaches, are crossed without being picked by hand.
C must equal the oracle bit for bit; the linear layer must be within 1e-2
relative of the fp64 oracle per element and exactly zero where the exact
accumulator is.  The drawn shapes must reach several routes, so that a
change of the rules cannot leave the test exercising only one kernel."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from bit_tensor_gemm_gb300 import build as bld  # noqa: E402
from bit_tensor_gemm_gb300 import lbgemm as L  # noqa: E402
from bit_tensor_gemm_gb300 import synth  # noqa: E402

# per shape and per test, in multiply-adds, so that the oracle finishes in
# seconds on a few cores
SHAPE_MACS = 1 << 33
TEST_MACS = 1 << 35


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


def draw_shapes(seed, count, k_align, k_free=False):
    """count shapes (M, N, K): M, N log-uniform in [1, 2^12.5], K log-uniform
    in [k_align, 16384] rounded to k_align (to any K >= 1 for a quarter of the
    shapes when k_free); within the multiply-add budgets."""
    g = np.random.default_rng(seed)
    out, total = [], 0
    while len(out) < count:
        M = int(round(2 ** g.uniform(0, 12.5)))
        N = int(round(2 ** g.uniform(0, 12.5)))
        k = 2 ** g.uniform(np.log2(k_align), 14)
        K = int(round(k)) if (k_free and g.random() < 0.25) else max(k_align, int(round(k / k_align)) * k_align)
        macs = M * N * K
        if macs > SHAPE_MACS or total + macs > TEST_MACS:
            continue
        total += macs
        out.append((M, N, K))
    return out


def routes_of(bits, shapes):
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    return {L.lbgemm_dispatch_for(sm, bits, M, N, K)[0] for M, N, K in shapes}


@pytest.mark.parametrize("bits,k_align,seed", [(8, 16, 9001), (4, 2, 9002), (1, 32, 9003)])
def test_dispatch_random_shapes(bits, k_align, seed):
    shapes = draw_shapes(seed, 40, k_align, k_free=(bits == 8))
    for i, (M, N, K) in enumerate(shapes):
        A, B = synth.operands(bits, M, N, K, seed * 100 + i)
        got = G().gemm(bits, A, B, K)
        want = oracle.gemm(bits, A, B, K)
        if not np.array_equal(got, want):
            bad = np.argwhere(got != want)
            m, n = bad[0]
            raise AssertionError(f"{bits}-bit {M}x{N}x{K}: {len(bad)} entries differ; first at "
                                 f"({m},{n}): got {got[m, n]} want {want[m, n]}")
    # the draw reaches more than one kernel of the dispatch
    assert len(routes_of(bits, shapes)) >= 2, routes_of(bits, shapes)


def test_linear_random_shapes():
    g = np.random.default_rng(9010)
    seen = set()
    total = 0
    for i in range(24):
        while True:
            M = int(round(2 ** g.uniform(0, 10)))           # 1..1024 tokens
            N = int(round(2 ** g.uniform(6, 14)))           # 64..16384 output channels
            K = 16 * int(round(2 ** g.uniform(6, 13) / 16))  # 64..8192
            K = max(K, 16)
            if M * N * K <= SHAPE_MACS and total + M * N * K <= TEST_MACS:
                break
        total += M * N * K
        X, sx, W, sw = synth.linear_operands(M, N, K, 9100 + i)
        X[0, :] = 0  # an all-zero token: exact zeros in Y
        ref = oracle.linear(X, sx, W, sw)
        acc = oracle.gemm(8, X, W, K)
        Y = G().linear(X, sx, W, sw)
        bad = np.abs(Y - ref) > 1e-2 * np.abs(ref)
        assert not bad.any(), f"linear {M}x{N}x{K}: {bad.sum()} entries beyond 1e-2 relative"
        assert np.all(Y[acc == 0] == 0), f"linear {M}x{N}x{K}: nonzero output where acc = 0"
        seen.add(L.lbgemm_route(8, M, N, K, linear=True)[0])
    assert len(seen) >= 3, seen
