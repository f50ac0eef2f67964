"""Host-side tests of the C ABI: the library loads, exports every declared
symbol, and its host logic (argument checks, selection rule, table, chunk
settings) agrees with the oracle of the selection rules.  No GPU needed."""
import os
import re

import numpy as np
import pytest

from bit_tensor_gemm_gb300 import build as bld
from bit_tensor_gemm_gb300 import lbgemm as L
from oracle import select as osel

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "lbgemm.h")


@pytest.fixture(scope="module")
def lib():
    bld.build()
    return L.load()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lbgemm_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = header_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), f"{n} declared in lbgemm.h but not exported"


def test_binding_matches_header():
    assert L.exported_symbols() == header_functions()


def test_variant_space(lib):
    assert L.lbgemm_num_variants() == osel.NUM_VARIANTS == 9
    assert L.lbgemm_default_variant() == osel.DEFAULT_VARIANT
    for v in range(9):
        tile, stages = osel.variant_of(v)
        info = L.lbgemm_variant_info(8, v)
        assert info["stages"] == stages
        assert info["tile_n"] == (64, 128, 256)[tile]
        assert info["tile_m"] == (128, 128, 256)[tile]
        assert L.lbgemm_variant_info(4, v)["tile_k"] == 128
        b1 = L.lbgemm_variant_info(1, v)
        assert (b1["tile_m"], b1["tile_n"], b1["tile_k"]) == (info["tile_m"], info["tile_n"], 128)
    with pytest.raises(L.LbgemmError):
        L.lbgemm_variant_info(8, 9)


def test_choose_matches_oracle(lib):
    g = np.random.default_rng(11)
    for trial in range(500):
        t = g.uniform(1.0, 2.0, 9).astype(np.float32)
        if trial % 3 == 0:  # ties and near-ties around the default
            t[g.integers(0, 9)] = t.min()
            t[7] = t.min() * np.float32(1.0 + g.choice([0.0, 0.01, 0.019, 0.03]))
        want = osel.table_choice([float(x) for x in t], 7, 0.02)
        assert L.lbgemm_choose(t, 7, 0.02) == want, t
    assert L.lbgemm_choose([1.0] * 8 + [float("nan")]) == -1


def test_select_nearest_matches_oracle(lib):
    g = np.random.default_rng(12)
    sm = 4242  # an SM count no real device has, so no other test's entries interfere
    sizes = [64, 128, 256, 512, 1024, 2048, 4096, 8192, 16384]
    entries = {}
    for _ in range(40):
        key = tuple(int(x) for x in g.choice(sizes, 3))
        entries[key] = int(g.integers(0, 9))
    for (m, n, k), v in entries.items():
        L.lbgemm_table_set_for(sm, 8, m, n, k, v)
    ent = list(entries.items())
    for _ in range(300):
        q = [int(x) for x in g.integers(1, 20000, 3)]
        assert L.lbgemm_select_for(sm, 8, *q) == osel.nearest(ent, *q), q
    for (m, n, k), v in ent:
        assert L.lbgemm_select_for(sm, 8, m, n, k) == v
    # other bit widths and SM counts see none of these entries
    assert L.lbgemm_select_for(sm, 4, 64, 64, 64) == osel.DEFAULT_VARIANT
    assert L.lbgemm_select_for(sm + 1, 8, 64, 64, 64) == osel.DEFAULT_VARIANT


def test_table_roundtrip(lib, tmp_path):
    L.lbgemm_table_clear()
    L.lbgemm_table_set_for(152, 8, 64, 128, 256, 3)
    L.lbgemm_table_set_for(152, 1, 8192, 8192, 65536, 8)
    L.lbgemm_table_set_for(148, 4, 8192, 8192, 8192, 0)
    p = str(tmp_path / "table.txt")
    L.lbgemm_table_save(p)
    L.lbgemm_table_clear()
    assert L.lbgemm_table_size() == 0
    L.lbgemm_table_load(p)
    assert L.lbgemm_table_size() == 3
    assert L.lbgemm_select_for(152, 8, 64, 128, 256) == 3
    assert L.lbgemm_select_for(152, 1, 8192, 8192, 65536) == 8
    assert L.lbgemm_select_for(148, 4, 8192, 8192, 8192) == 0
    bad = tmp_path / "bad.txt"
    bad.write_text("152 8 64 64 64 9\n")
    with pytest.raises(L.LbgemmError):
        L.lbgemm_table_load(str(bad))
    L.lbgemm_table_clear()


def test_exact_chunk_settings(lib):
    assert L.lbgemm_get_exact_chunk(8) == 1024
    assert L.lbgemm_get_exact_chunk(4) == 131072
    assert L.lbgemm_get_exact_chunk(1) == 1 << 23
    for bits, bad in [(8, 1088), (8, 100), (4, 64), (4, 1 << 20), (1, 64), (1, 1 << 25), (2, 128)]:
        with pytest.raises(L.LbgemmError):
            L.lbgemm_set_exact_chunk(bits, bad)
    L.lbgemm_set_exact_chunk(8, 512)
    assert L.lbgemm_get_exact_chunk(8) == 512
    L.lbgemm_set_exact_chunk(8, 1024)


def test_tail_split_settings(lib):
    assert L.lbgemm_get_tail_split() == 1
    for bad in (-1, 3):
        with pytest.raises(L.LbgemmError):
            L.lbgemm_set_tail_split(bad)
    assert L.lbgemm_get_tail_split() == 1
    for mode in (0, 2, 1):
        L.lbgemm_set_tail_split(mode)
        assert L.lbgemm_get_tail_split() == mode


@pytest.mark.parametrize("args,status", [
    ((3, 4, 4, 4, 16, 16, 16), L.ERR_INVALID_ARG),           # bits
    ((8, -1, 4, 4, 16, 16, 16), L.ERR_INVALID_ARG),          # negative M
    ((8, 4, 4, 0, 16, 16, 16), L.ERR_INVALID_ARG),           # K = 0
    ((8, 4, 4, 131072, 16, 16, 16), L.ERR_INVALID_ARG),      # int32 overflow possible
    ((4, 4, 4, 7, 16, 16, 16), L.ERR_ALIGNMENT),             # odd K, 4-bit
    ((1, 4, 4, 48, 16, 16, 16), L.ERR_ALIGNMENT),            # K % 32, 1-bit
    ((8, 4, 4, 16, 0, 16, 16), L.ERR_INVALID_ARG),           # null A
    ((8, 4, 4, 16, 16, 24, 16), L.ERR_ALIGNMENT),            # misaligned B
])
def test_argument_errors_need_no_device(lib, args, status):
    bits, M, N, K, a, b, c = args
    with pytest.raises(L.LbgemmError) as e:
        L.lbgemm_run_variant(bits, M, N, K, a or None, b, c, 0, 0)
    assert e.value.status == status
    assert L.lbgemm_last_error()


@pytest.mark.parametrize("M,N,K,tile,status", [
    (16, 100, 4240, 0, L.ERR_INVALID_ARG),   # warp-MMA: K above its limit at 16 rows
    (32, 100, 2064, 0, L.ERR_INVALID_ARG),   # warp-MMA: K above its limit at 32 rows
    (257, 300, 64, 0, L.ERR_INVALID_ARG),    # warp-MMA: small side above 256 rows
    (200, 300, 2064, 0, L.ERR_INVALID_ARG),  # warp-MMA: K above its limit past 16 rows
    (16, 100, 40, 0, L.ERR_ALIGNMENT),       # warp-MMA: K % 16
    (16, 100, 64, 96, L.ERR_INVALID_ARG),    # fused: tile width
    (16, 100, 40, 128, L.ERR_ALIGNMENT),     # fused: K % 16
])
def test_forced_route_errors_need_no_device(lib, M, N, K, tile, status):
    with pytest.raises(L.LbgemmError) as e:
        if tile:
            L.lbgemm_run_fused(M, N, K, 16, 16, 16, tile, 0)
        else:
            L.lbgemm_run_warpmma(M, N, K, 16, 16, 16, 0)
    assert e.value.status == status


def test_empty_problem_is_a_noop(lib):
    L.lbgemm_run(8, 0, 5, 16, 16, 16, 16, 0)
    L.lbgemm_run(1, 7, 0, 32, None, None, None, 0)


def test_workspace_size(lib):
    assert L.lbgemm_workspace_size(1, 64, 64, 48) == 0   # K % 32 != 0: not a 1-bit problem
    assert L.lbgemm_workspace_size(1, 64, 64, 64) == 2 * 64 * 64  # one e4m3 byte per bit
    # int8: fp16 copies, rows padded to a multiple of 8 halves, each buffer to 256 bytes
    assert L.lbgemm_workspace_size(8, 3, 5, 9) == 256 + 256
    assert L.lbgemm_workspace_size(8, 256, 256, 256) == 2 * 256 * 256 * 2
    assert L.lbgemm_workspace_size(4, 256, 128, 256) == 256 * 256 + 128 * 256


# ---- dispatch routes (host only) ----------------------------------------------

def _pairs(lo, hi, K):
    if 128 < lo <= 256:
        return (hi >= 16384 and K >= 1024) or (hi >= 8192 and K >= 16384)
    if lo > 384:
        return (hi >= 8192 and K >= 2048) or (hi >= 16384 and K >= 1024) or K >= 16384
    return False


def _route8(M, N, K, linear=False):
    """The shape rules that include/lbgemm.h states for lbgemm_run and
    lbgemm_linear, written out from that text (16-byte-aligned operands)."""
    if M == 0 or N == 0:
        return L.ROUTE_NONE, 0
    lo, hi = min(M, N), max(M, N)
    k16 = K % 16 == 0
    if k16 and (M <= 4 or (linear and M <= 8 and 4096 < K <= 8192)):
        return L.ROUTE_SKINNY, 0
    if lo <= 16 and hi >= 1024 and k16 and K <= 4096 and (not linear or M <= 16):
        return L.ROUTE_STREAM, 0
    if lo <= 32 and k16 and K <= (4224 if lo <= 16 else 2048):
        return L.ROUTE_WARPMMA, 0
    if not linear:
        cap = 2 ** 19 if K <= 1024 else 2 ** 18
        if (lo <= 256 and 256 < K <= 2048 and k16
                and (lo * hi <= cap or (K <= 512 and M * N * K <= 2 ** 28))):
            return L.ROUTE_WARPMMA, 0
        if K <= 512 and M * N * K <= 2 ** 28 and k16:
            return L.ROUTE_SMALL, 0
    if (k16 and lo <= 512 and hi >= 1024 and K >= 512 and (not linear or M <= N)
            and (hi >= 4096 or K >= 8192 or (hi >= 2048 and K >= 4096)
                 or (lo <= 256 and K >= 2048))):
        # the linear layer never on CTA pairs
        pairs = _pairs(lo, hi, K) and not linear
        return L.ROUTE_FUSED, 64 if lo <= 64 else 256 if pairs else 128
    return L.ROUTE_TABLE, 0


def test_routes_follow_the_stated_rules(lib):
    sides = [1, 2, 4, 5, 16, 17, 32, 33, 64, 65, 100, 128, 129, 200, 256, 257, 300, 384, 385, 512,
             513, 1024, 2048, 4096, 8192, 16384]
    ks = [16, 48, 64, 256, 272, 512, 528, 1024, 1040, 2048, 2064, 4096, 4224, 4240, 8192, 16384]
    for M in sides:
        for N in sides:
            for K in ks:
                assert L.lbgemm_route(8, M, N, K) == _route8(M, N, K), (M, N, K)
                assert L.lbgemm_route(8, M, N, K, linear=True) == _route8(M, N, K, True), (M, N, K)


def test_routes_of_measured_examples(lib):
    R = L
    cases = [((8, 1, 11008, 4096), (R.ROUTE_SKINNY, 0)),
             ((8, 16, 11008, 4096), (R.ROUTE_STREAM, 0)),
             ((8, 11008, 5, 4096), (R.ROUTE_STREAM, 0)),
             ((8, 16, 11008, 4224), (R.ROUTE_WARPMMA, 0)),
             ((8, 64, 1024, 1024), (R.ROUTE_WARPMMA, 0)),
             ((8, 256, 256, 256), (R.ROUTE_SMALL, 0)),
             ((8, 64, 8192, 2048), (R.ROUTE_FUSED, 64)),
             ((8, 512, 4096, 1024), (R.ROUTE_FUSED, 128)),
             ((8, 8192, 256, 2048), (R.ROUTE_FUSED, 128)),
             ((8, 256, 16384, 16384), (R.ROUTE_FUSED, 256)),
             ((8, 8192, 8192, 8192), (R.ROUTE_TABLE, 0)),
             ((8, 0, 5, 16), (R.ROUTE_NONE, 0)),
             ((4, 8192, 8192, 8192), (R.ROUTE_TABLE, 0)),
             ((1, 64, 64, 1024), (R.ROUTE_POPC, 0)),
             ((1, 256, 256, 1024), (R.ROUTE_POPC, 0)),      # 2^26 bit-MACs
             ((1, 512, 512, 512), (R.ROUTE_TABLE, 0)),      # 2^27: the tensor cores
             ((4, 256, 256, 256), (R.ROUTE_SMALL, 0)),      # 2^24 MACs, K <= 256
             ((4, 512, 512, 256), (R.ROUTE_SMALL, 0)),      # 2^26 exactly
             ((4, 1024, 512, 256), (R.ROUTE_TABLE, 0)),     # 2^27 > 2^26
             ((4, 256, 256, 512), (R.ROUTE_TABLE, 0)),      # K > 256
             ((4, 64, 64, 48), (R.ROUTE_TABLE, 0)),         # K % 32 != 0
             ((1, 8192, 8192, 65536), (R.ROUTE_TABLE, 0))]
    for args, want in cases:
        assert L.lbgemm_route(*args) == want, args
    # the linear layer on the 11008 x 4096 weights, token counts of the benchmark
    for M, want in [(1, (R.ROUTE_SKINNY, 0)), (16, (R.ROUTE_STREAM, 0)), (17, (R.ROUTE_FUSED, 64)),
                    (128, (R.ROUTE_FUSED, 128)), (512, (R.ROUTE_FUSED, 128)),
                    (2048, (R.ROUTE_TABLE, 0))]:
        assert L.lbgemm_route(8, M, 11008, 4096, linear=True) == want, M
    # the GEMM of the same shape takes CTA pairs, the linear layer does not
    assert L.lbgemm_route(8, 512, 11008, 4096) == (R.ROUTE_FUSED, 256)
    for bad in [(3, 4, 4, 16), (8, -1, 4, 16), (8, 4, 4, 0)]:
        with pytest.raises(L.LbgemmError):
            L.lbgemm_route(*bad)
    with pytest.raises(L.LbgemmError):
        L.lbgemm_route(4, 16, 16, 32, linear=True)


def test_bench_route_histogram(lib):
    """bench.py's per-route summary of the 729-shape sweep covers every shape
    once and names the in-kernel conversion kernel with its tile."""
    import bench  # noqa: PLC0415
    h = bench.route_histogram(L, bench.SWEEP)
    assert sum(e["shapes"] for e in h.values()) == 729
    assert set(h) <= {"table", "skinny_dp4a", "stream_mma", "warp_mma", "small_dp4a",
                      "in_kernel_conversion_64",
                      "in_kernel_conversion_128", "in_kernel_conversion_256"}
    assert h["table"]["shapes"] > 200 and "ms" not in h["table"]
    t = bench.route_histogram(L, bench.SWEEP[:3], [1.0, 2.0, 3.0])
    assert sum(e["ms"] for e in t.values()) == 6.0


# every entry point rejects bad arguments before it touches a device
P = 4096  # a 16-byte-aligned stand-in address (never dereferenced: the checks fail first)


@pytest.mark.parametrize("call,status", [
    (lambda: L.lbgemm_run_host(3, 4, 4, 16, P, P, P), L.ERR_INVALID_ARG),
    (lambda: L.lbgemm_run_host(8, 4, 4, 0, P, P, P), L.ERR_INVALID_ARG),
    (lambda: L.lbgemm_run_host(8, 4, 4, 16, None, P, P), L.ERR_INVALID_ARG),
    (lambda: L.lbgemm_run_host(1, 4, 4, 48, P, P, P), L.ERR_ALIGNMENT),
    (lambda: L.lbgemm_linear(4, 4, 16, P, None, P, P, P), L.ERR_INVALID_ARG),
    (lambda: L.lbgemm_linear(4, 4, 131072, P, P, P, P, P), L.ERR_INVALID_ARG),
    (lambda: L.lbgemm_linear_variant(4, 4, 16, P, P, P, P, P, 9), L.ERR_INVALID_ARG),
    (lambda: L.lbgemm_linear_quant(4, 4, 16, P, P, None, P), L.ERR_INVALID_ARG),
    (lambda: L.lbgemm_quantize_rows(-1, 16, P, P, P), L.ERR_INVALID_ARG),
    (lambda: L.lbgemm_quantize_rows(4, 0, P, P, P), L.ERR_INVALID_ARG),
    (lambda: L.lbgemm_quantize_rows(4, 16, P, None, P), L.ERR_INVALID_ARG),
    (lambda: L.lbgemm_run_popc(4, 4, 48, P, P, P), L.ERR_ALIGNMENT),
    (lambda: L.lbgemm_run_popc(4, 4, 64, P, P, P, 9), L.ERR_INVALID_ARG),
    (lambda: L.lbgemm_run_encoded(2, 4, 4, 64, P, P, P), L.ERR_INVALID_ARG),
    (lambda: L.lbgemm_run_encoded(8, 4, 4, 64, P, P, P, -2), L.ERR_INVALID_ARG),
    (lambda: L.lbgemm_encode(3, 4, 64, P, P), L.ERR_INVALID_ARG),
])
def test_entry_points_reject_bad_arguments_without_a_device(lib, call, status):
    with pytest.raises(L.LbgemmError) as e:
        call()
    assert e.value.status == status
    assert L.lbgemm_last_error()


def test_empty_problems_need_no_device(lib):
    L.lbgemm_run_host(8, 0, 4, 16, P, P, P)
    L.lbgemm_linear(0, 4, 16, P, P, P, P, P)
    L.lbgemm_quantize_rows(0, 16, P, P, P)
    L.lbgemm_run_popc(4, 0, 64, P, P, P)
    L.lbgemm_run_encoded(8, 4, 0, 64, P, P, P)


C_PROGRAM = r"""
#include <stdio.h>
#include "lbgemm.h"
int main(void) {
  int tm = 0, tn = 0, tk = 0, st = 0, tile = -1;
  if (lbgemm_num_variants() != 9) return 1;
  if (lbgemm_variant_info(8, lbgemm_default_variant(), &tm, &tn, &tk, &st) != LBGEMM_OK) return 2;
  int route = lbgemm_route(8, 16, 11008, 4096, 1, &tile);
  lbgemm_status bad = lbgemm_run(3, 4, 4, 16, (const void*)0, (const void*)0, (int32_t*)0,
                                 (void*)0);
  const char* msg = lbgemm_last_error();
  printf("%d %d %d %d %d %d %d %d\n", tm, tn, tk, st, route, tile, (int)bad, msg && msg[0] ? 1 : 0);
  return 0;
}
"""


def test_header_is_plain_c_and_links(lib, tmp_path):
    """The boundary is a C ABI: a C99 program includes the header, links the
    library and calls host-side entry points (no device needed)."""
    import shutil  # noqa: PLC0415
    import subprocess  # noqa: PLC0415
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    libdir = os.path.dirname(L.LIBRARY)
    exe = tmp_path / "abi"
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", str(src),
                    "-I", os.path.dirname(HEADER), "-L", libdir, "-llbgemm",
                    f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    tm, tn, tk, stages, route, tile, bad, has_msg = map(int, out)
    info = L.lbgemm_variant_info(8, L.lbgemm_default_variant())
    assert (tm, tn, tk, stages) == (info["tile_m"], info["tile_n"], info["tile_k"], info["stages"])
    assert (route, tile) == (L.ROUTE_STREAM, 0)
    assert bad == L.ERR_INVALID_ARG and has_msg == 1


# ---- measured routes in the table (host only) -------------------------------------

def test_choose_candidate_matches_oracle(lib):
    g = np.random.default_rng(31)
    for trial in range(400):
        n = int(g.integers(1, 20))
        t = g.uniform(1.0, 2.0, n).astype(np.float32)
        d = int(g.integers(0, n))
        if trial % 3 == 0:  # ties and near-ties around the default
            t[g.integers(0, n)] = t.min()
            t[d] = t.min() * np.float32(1.0 + g.choice([0.0, 0.01, 0.019, 0.03]))
        want = osel.candidate_choice([float(x) for x in t], d, 0.02)
        assert L.lbgemm_choose_candidate(list(t), d, 0.02) == want, (t, d)
    # the nine-variant rule is the same rule
    t = [3.0, 2.0, 1.0, 1.5, 1.01, 4.0, 1.0, 1.02, 2.0]
    assert L.lbgemm_choose(t, 7, 0.02) == L.lbgemm_choose_candidate(t, 7, 0.02) == 7
    assert L.lbgemm_choose_candidate([1.0, float("nan")], 0, 0.02) == -1
    assert L.lbgemm_choose_candidate([1.0, 2.0], 2, 0.02) == -1


def test_candidates_cover_the_routes_that_run(lib):
    T, POPC, SK, WM, SM, FU = (L.ROUTE_TABLE, L.ROUTE_POPC, L.ROUTE_SKINNY, L.ROUTE_WARPMMA,
                               L.ROUTE_SMALL, L.ROUTE_FUSED)
    tc = [(T, v) for v in range(9)]
    assert L.lbgemm_candidates(4, 8192, 8192, 8192) == tc
    assert L.lbgemm_candidates(4, 256, 512, 1024) == tc + [(SM, 0)]
    assert L.lbgemm_candidates(4, 256, 512, 1040) == tc  # K % 32 != 0
    assert L.lbgemm_candidates(1, 8192, 8192, 65536) == tc  # 2^42 bit-MACs: no popcount
    assert L.lbgemm_candidates(1, 64, 64, 1024) == tc + [(POPC, v) for v in range(9)]
    assert L.lbgemm_candidates(8, 16384, 16384, 16384) == tc
    assert L.lbgemm_candidates(8, 64, 16384, 4096) == tc + [(FU, 64), (FU, 128)]
    assert L.lbgemm_candidates(8, 8, 1024, 1024) == tc + [(SK, 0), (L.ROUTE_STREAM, 0), (WM, 0),
                                                          (SM, 0), (FU, 64), (FU, 128)]
    assert (L.ROUTE_STREAM, 0) in L.lbgemm_candidates(8, 4096, 16, 4096)
    assert (L.ROUTE_STREAM, 0) not in L.lbgemm_candidates(8, 4096, 16, 4112)  # K <= 4096
    assert (L.ROUTE_STREAM, 0) not in L.lbgemm_candidates(8, 17, 4096, 1024)
    assert L.lbgemm_candidates(8, 256, 512, 2048) == tc + [(WM, 0), (SM, 0), (FU, 64), (FU, 128),
                                                           (FU, 256)]
    assert L.lbgemm_candidates(8, 256, 512, 4096) == tc + [(SM, 0), (FU, 64), (FU, 128), (FU, 256)]
    assert L.lbgemm_candidates(8, 100, 100, 100) == tc  # K % 16 != 0: the 8-bit routes need it
    with pytest.raises(L.LbgemmError):
        L.lbgemm_candidates(3, 64, 64, 64)


def test_table_routes_drive_the_dispatch(lib, tmp_path):
    sm = 4545  # an SM count no device has
    T, POPC, WM, FU = L.ROUTE_TABLE, L.ROUTE_POPC, L.ROUTE_WARPMMA, L.ROUTE_FUSED
    # no entry: the shape rules (lbgemm_route), the variant from selection
    assert L.lbgemm_dispatch_for(sm, 1, 64, 64, 1024) == (POPC, 1)  # the rule's 64 x 64 variant
    for bits, shape in [(8, (16, 11008, 4096)), (8, (4096, 4096, 4096)), (1, (64, 64, 1024)),
                        (4, (256, 256, 256))]:
        r, p = L.lbgemm_dispatch_for(sm, bits, *shape)
        rule, tile = L.lbgemm_route(bits, *shape)
        assert r == rule
        if r == T:
            assert p == L.lbgemm_select_for(sm, bits, *shape)
        if r == FU:
            assert p == tile
    # measured entries take over for their exact shape only
    L.lbgemm_table_set_choice_for(sm, 8, 4096, 4096, 4096, 3, T, 5)
    L.lbgemm_table_set_choice_for(sm, 8, 256, 8192, 2048, 1, FU, 256)
    L.lbgemm_table_set_choice_for(sm, 8, 128, 1024, 1024, 4, WM, 0)
    L.lbgemm_table_set_choice_for(sm, 1, 64, 64, 1024, 2, POPC, 4)
    L.lbgemm_table_set_for(sm, 4, 512, 512, 512, 6)  # a label without a route
    assert L.lbgemm_dispatch_for(sm, 8, 4096, 4096, 4096) == (T, 5)
    assert L.lbgemm_select_for(sm, 8, 4096, 4096, 4096) == 3  # the label stays the variant
    assert L.lbgemm_dispatch_for(sm, 8, 256, 8192, 2048) == (FU, 256)
    assert L.lbgemm_dispatch_for(sm, 8, 128, 1024, 1024) == (WM, 0)
    assert L.lbgemm_dispatch_for(sm, 1, 64, 64, 1024) == (POPC, 4)
    assert L.lbgemm_dispatch_for(sm, 4, 512, 512, 512) == (T, 6)
    assert L.lbgemm_table_get_for(sm, 8, 256, 8192, 2048) == (1, FU, 256)
    assert L.lbgemm_table_get_for(sm, 4, 512, 512, 512) == (6, -1, 0)
    assert L.lbgemm_table_get_for(sm, 4, 512, 512, 1024) is None
    # a neighbour of a measured shape follows the rules again
    assert L.lbgemm_dispatch_for(sm, 8, 256, 8192, 4096)[0] == L.lbgemm_route(8, 256, 8192, 4096)[0]
    # routes that cannot run the shape are refused
    for bad in [(8, 512, 512, 512, 0, WM, 0),      # warp-MMA: small side above 256
                (4, 64, 64, 64, 0, FU, 128),       # 8-bit routes only
                (8, 64, 64, 40, 0, FU, 128),       # K % 16
                (8, 64, 64, 64, 0, FU, 96),        # no such tile
                (8, 64, 64, 64, 0, POPC, 1),       # popcount: 1-bit only
                (8, 64, 64, 64, 0, T, 9),
                (8, 64, 64, 64, 0, 6, 0)]:
        with pytest.raises(L.LbgemmError):
            L.lbgemm_table_set_choice_for(sm, *bad)
    # the file keeps the routes; old six-column lines still load
    p = str(tmp_path / "t.txt")
    L.lbgemm_table_save(p)
    text = open(p).read()
    assert f"{sm} 8 256 8192 2048 1 {FU} 256\n" in text and f"{sm} 4 512 512 512 6\n" in text
    L.lbgemm_table_clear()
    L.lbgemm_table_load(p)
    assert L.lbgemm_dispatch_for(sm, 8, 256, 8192, 2048) == (FU, 256)
    assert L.lbgemm_table_get_for(sm, 4, 512, 512, 512) == (6, -1, 0)
    n = L.lbgemm_table_size()
    for bad_line in [f"{sm} 8 64 64 64 7 {WM}\n",            # route without its parameter
                     f"{sm} 8 512 512 512 7 {WM} 0\n",      # a route that cannot run it
                     f"{sm} 8 64 64 64 7 0 7 1\n"]:         # trailing field
        bad = tmp_path / "bad.txt"
        bad.write_text("# header\n" + bad_line)
        with pytest.raises(L.LbgemmError):
            L.lbgemm_table_load(str(bad))
        assert L.lbgemm_table_size() == n  # nothing merged
    L.lbgemm_table_clear()


def test_oracle_dispatch_rule():
    assert osel.dispatch(None, (3, 0)) == (3, 0)
    assert osel.dispatch((5, 128), (0, 7)) == (5, 128)


# ---- the GB300 table shipped with the library ----------------------------------------

SHIPPED = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                       "bit_tensor_gemm_gb300", "data", "lbgemm_table_gb300.txt")

PROBE = r"""
import json, sys
sys.path.insert(0, {root!r})
from bit_tensor_gemm_gb300 import lbgemm as L
L.load()
out = {{"path": L.lbgemm_table_default_path(), "size": L.lbgemm_table_size(), "q": []}}
for sm, bits, m, n, k in json.loads(sys.argv[1]):
    out["q"].append([L.lbgemm_select_for(sm, bits, m, n, k),
                     list(L.lbgemm_dispatch_for(sm, bits, m, n, k))])
print(json.dumps(out))
"""


def _fresh_process(queries, env_table=None):
    """Answers of a fresh process (the table is loaded at first use)."""
    import json  # noqa: PLC0415
    import subprocess  # noqa: PLC0415
    import sys  # noqa: PLC0415
    env = dict(os.environ)
    env.pop("LBGEMM_TABLE", None)
    if env_table is not None:
        env["LBGEMM_TABLE"] = env_table
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", PROBE.format(root=root), json.dumps(queries)],
                       env=env, capture_output=True, text=True, check=True)
    return json.loads(r.stdout)


def _shipped_entries():
    rows = []
    for line in open(SHIPPED):
        w = line.split()
        if w and not w[0].startswith("#"):
            rows.append([int(x) for x in w])
    return rows


def test_shipped_table_is_loaded_by_default(lib):
    rows = _shipped_entries()
    assert len(rows) == 3 * 729  # the 729-shape grid for 8-, 4- and 1-bit operands
    assert {r[1] for r in rows} == {8, 4, 1} and all(len(r) == 8 for r in rows)
    g = np.random.default_rng(5)
    picks = [rows[i] for i in g.choice(len(rows), 60, replace=False)]
    picks += [r for r in rows if r[1] in (4, 1)][:20]
    queries = [r[:5] for r in picks]
    got = _fresh_process(queries)
    assert os.path.realpath(got["path"]) == os.path.realpath(SHIPPED)
    assert got["size"] == len(rows)
    for r, (sel, disp) in zip(picks, got["q"]):
        assert sel == r[5], r  # lbgemm_select gives the stored label
        assert disp == [r[6], r[7]], r  # and lbgemm_run the stored route


def test_table_file_from_the_environment(lib, tmp_path):
    assert _fresh_process([], env_table="none")["size"] == 0
    assert _fresh_process([], env_table="")["size"] == 0
    p = tmp_path / "mine.txt"
    p.write_text("# mine\n4242 4 100 200 300 5\n4242 8 64 4096 1024 2 5 64\n")
    got = _fresh_process([[4242, 4, 100, 200, 300], [4242, 8, 64, 4096, 1024]], env_table=str(p))
    assert got["size"] == 2 and got["path"] == str(p)
    assert got["q"] == [[5, [L.ROUTE_TABLE, 5]], [2, [L.ROUTE_FUSED, 64]]]


def test_fused_slice_setting(lib):
    assert L.lbgemm_get_fused_slice() == 0
    for v in (128, 256, 0):
        L.lbgemm_set_fused_slice(v)
        assert L.lbgemm_get_fused_slice() == v
    for bad in (64, 512, -1):
        with pytest.raises(L.LbgemmError) as e:
            L.lbgemm_set_fused_slice(bad)
        assert e.value.status == L.ERR_INVALID_ARG
    assert L.lbgemm_get_fused_slice() == 0


def test_fused_stream_k_setting(lib):
    """The conversion kernels' schedule knob: 0 (split K, the default) or 1
    (stream-K); anything else is rejected and leaves the setting alone."""
    assert L.lbgemm_get_fused_stream_k() == 0
    for v in (1, 0):
        L.lbgemm_set_fused_stream_k(v)
        assert L.lbgemm_get_fused_stream_k() == v
    for bad in (2, -1):
        with pytest.raises(L.LbgemmError) as e:
            L.lbgemm_set_fused_stream_k(bad)
        assert e.value.status == L.ERR_INVALID_ARG
    assert L.lbgemm_get_fused_stream_k() == 0


def _fused_schedule(M, N, K, tile_n, linear, sm, slice_, force=False):
    """The schedule include/lbgemm.h states for lbgemm_fused_schedule, written
    out from that text."""
    import math  # noqa: PLC0415
    large_b = linear or N >= M
    if not linear and not large_b and N % 4:
        return 1, 0
    R, S = (N, M) if large_b else (M, N)
    tiles = math.ceil(R / 128) * math.ceil(S / tile_n)
    c = 4 * tile_n / K
    nkb = math.ceil(K / 64)
    best, splits = None, 1
    for p in range(1, 17):
        if p > 1 and nkb // p < 4:
            break
        cost = math.ceil(tiles * p / sm) * (1 / p + (c if p > 1 else 0))
        if best is None or cost < best - 1e-9:
            best, splits = cost, p
    k = math.ceil((K + 7) // 8 * 8 / slice_)
    r = math.ceil(tiles * k / sm) if tiles * k >= 2 * sm else 0
    sk = r / k + (r / k + 1) * c if r else None
    stream = force and r > 0
    if linear and not stream:
        chosen = best
        if best > 0.7 * math.ceil(tiles / sm):
            splits, chosen = 1, math.ceil(tiles / sm)
        stream = sk is not None and sk <= 0.85 * chosen
    if stream:
        return 1, math.ceil(r / k) + 1
    return splits, 0


def test_fused_schedule_follows_the_stated_model(lib):
    """The split / stream-K plan of the 64- and 128-wide conversion kernels,
    against the header's formula on a grid of GEMM and linear shapes and SM
    counts, plus the measured cases the model was fitted on."""
    assert L.lbgemm_get_fused_slice() == 0 and L.lbgemm_get_fused_stream_k() == 0
    sides = [1, 16, 64, 100, 128, 192, 256, 512, 1024, 4096, 11008, 28672]
    for M in sides:
        for N in sides:
            for K in (256, 1040, 4096, 16384):
                for tile in (64, 128):
                    for linear in (False, True):
                        if linear and M > N:
                            continue
                        for sm in (152, 148):
                            want = _fused_schedule(M, N, K, tile, linear, sm,
                                                   256 if tile == 64 or linear else 128)
                            assert L.lbgemm_fused_schedule(M, N, K, tile, linear, sm) == want, \
                                (M, N, K, tile, linear, sm)
    # measured on GB300 (152 SMs): 64 x 16384 x 16384 GEMM in 7 pieces (114 ->
    # 106 us); the linear layer split where the grid is short (64 x 4096 x
    # 4096: 27 -> 19.5 us), stream-K where the tiles make a fractional wave
    # (192 x 11008 x 4096: 53 -> 45 us), whole tiles where neither pays
    # (256 x 28672 x 8192)
    assert L.lbgemm_fused_schedule(64, 16384, 16384, 64) == (7, 0)
    assert L.lbgemm_fused_schedule(64, 4096, 4096, 64, True) == (4, 0)
    assert L.lbgemm_fused_schedule(192, 11008, 4096, 128, True)[1] > 0
    assert L.lbgemm_fused_schedule(256, 28672, 8192, 128, True) == (1, 0)
    # forced stream-K, and the slice setting feeding the slice count
    L.lbgemm_set_fused_stream_k(1)
    try:
        assert L.lbgemm_fused_schedule(64, 16384, 16384, 64) == \
            _fused_schedule(64, 16384, 16384, 64, False, 152, 256, force=True)
    finally:
        L.lbgemm_set_fused_stream_k(0)
    L.lbgemm_set_fused_slice(128)
    try:
        assert L.lbgemm_fused_schedule(128, 11008, 4096, 128, True) == \
            _fused_schedule(128, 11008, 4096, 128, True, 152, 128)
        assert L.lbgemm_fused_schedule(512, 4096, 4096, 64) == \
            _fused_schedule(512, 4096, 4096, 64, False, 152, 128)
    finally:
        L.lbgemm_set_fused_slice(0)
    for bad in [(64, 64, 64, 256, False, 152), (0, 64, 64, 64, False, 152),
                (64, 64, 64, 64, False, 0), (128, 64, 64, 64, True, 152)]:
        with pytest.raises(L.LbgemmError):
            L.lbgemm_fused_schedule(*bad)
