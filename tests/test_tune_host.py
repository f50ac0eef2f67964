"""Host tests of the selection procedure (tune.py) and of bench.py's summary
arithmetic, with a stand-in for the library's timing calls: the decisions
(label, pick, head-to-head confirmation) follow the stated rules, checked
against the selection oracle.  No GPU."""
import numpy as np
import pytest

import bench
from bit_tensor_gemm_gb300 import lbgemm as L
from bit_tensor_gemm_gb300 import tune
from oracle import select as osel

T, FU, WM = 0, 5, 3


class FakeLib:
    """The library's selection entry points with scripted timings."""

    def __init__(self, cands, sweep_ms, confirm_ms):
        self.cands = cands
        self.sweep_ms = sweep_ms
        self.confirm_ms = confirm_ms  # {(route, param): (t_candidate, t_default)}
        self.table = {}
        self.confirm_calls = []

    def lbgemm_candidates(self, bits, m, n, k):
        return list(self.cands)

    def lbgemm_time_candidates(self, bits, m, n, k, A, B, C, cands, warmup=1, reps=5,
                               flush_l2=True):
        if len(cands) == 2 and tuple(cands[1]) == (T, 7):  # a head-to-head check
            self.confirm_calls.append((tuple(cands[0]), reps))
            return list(self.confirm_ms[tuple(cands[0])])
        assert [tuple(c) for c in cands] == [tuple(c) for c in self.cands]
        return list(self.sweep_ms)

    def lbgemm_choose(self, times, default, keep):
        if not all(t >= 0 for t in times):  # the library rejects NaN and negatives with -1
            return -1
        return osel.table_choice(list(times), default, keep)

    def lbgemm_choose_candidate(self, times, default, keep):
        if not all(t >= 0 for t in times):
            return -1
        return osel.candidate_choice(list(times), default, keep)

    def lbgemm_table_set_choice_for(self, sm, bits, m, n, k, label, route, param):
        self.table[(sm, bits, m, n, k)] = (label, route, param)


CANDS = [(T, v) for v in range(9)] + [(WM, 0), (FU, 128)]


def test_pick_confirmed_and_label_confirmed():
    ms = [1.0, 1.0, 1.0, 1.0, 0.80, 1.0, 1.0, 1.0, 1.0, 0.50, 0.90]  # label 4, pick warp-MMA
    lib = FakeLib(CANDS, ms, {(T, 4): (0.8, 1.0), (WM, 0): (0.5, 1.0)})
    recs = tune.sweep(lib, 8, [(64, 4096, 1024)], None, None, None, 152, reps=10,
                      confirm_reps=20)
    r = recs[0]
    assert r["label"] == 4 and tuple(r["pick"]) == (WM, 0)
    assert lib.table[(152, 8, 64, 4096, 1024)] == (4, WM, 0)
    assert sorted(lib.confirm_calls) == [((T, 4), 20), ((WM, 0), 20)]


def test_a_pick_that_loses_head_to_head_falls_back_to_the_default():
    ms = [1.0] * 9 + [0.50, 0.90]
    ms[7] = 1.0
    # the sweep saw warp-MMA twice as fast; the fresh head-to-head sees a tie
    lib = FakeLib(CANDS, ms, {(WM, 0): (0.99, 1.0)})
    r = tune.sweep(lib, 8, [(64, 4096, 1024)], None, None, None, 152)[0]
    assert r["label"] == 7  # the nine variants tie: the default is kept
    assert tuple(r["pick"]) == (T, 7)
    assert lib.table[(152, 8, 64, 4096, 1024)] == (7, T, 7)


def test_keep_margin_covers_the_timer_resolution():
    assert tune.keep_margin(1.0) == pytest.approx(0.02)
    assert tune.keep_margin(0.010) == pytest.approx(0.1)  # 1 us of 10 us
    # a candidate 5 % faster at 10 us is within the timer's resolution: no pick
    ms = [0.0100] * 9 + [0.0095, 0.0200]
    lib = FakeLib(CANDS, ms, {})
    r = tune.sweep(lib, 8, [(64, 64, 64)], None, None, None, 152)[0]
    assert tuple(r["pick"]) == (T, 7) and r["label"] == 7 and lib.confirm_calls == []


def test_selection_summary_arithmetic():
    shapes = [(64, 64, 64), (8192, 8192, 8192)]
    recs = [{"label": 7, "pick": [T, 7]}, {"label": 5, "pick": [T, 5]}]
    disp = [(T, 7), (T, 5)]
    # arms: default, label, dispatch, default again
    Tm = np.array([[0.010, 0.011, 0.010, 0.0105], [0.70, 0.60, 0.60, 0.70]])
    peaks = {"bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
    summ, roof = bench.selection_summary(8, shapes, recs, disp, Tm, 1.0, peaks, 20)
    assert summ["speedup_min"] == pytest.approx(0.010 / 0.011)
    assert summ["speedup_max"] == pytest.approx(0.70 / 0.60)
    assert summ["noise_floor_max"] == pytest.approx(0.05)
    assert summ["label_ne_default"] == 1 and summ["pick_ne_default"] == 1
    assert summ["dispatch_speedup_geomean"] == pytest.approx(np.sqrt(1.0 * 0.70 / 0.60))
    ops = 2.0 * (64 ** 3 + 8192 ** 3)
    assert summ["sweep_tops_dispatch"] == pytest.approx(ops / 0.610e-3 / 1e12)
    t_roof = bench.shape_roofline_ms(8, shapes, peaks)
    assert t_roof[1] == pytest.approx(2.0 * 8192 ** 3 / 1700e12 * 1e3)  # tensor-bound
    assert t_roof[0] == pytest.approx((2 * 64 * 64 + 4 * 64 * 64) / 6800e9 * 1e3)  # bytes
    assert roof["frac"] == pytest.approx(t_roof.sum() / 0.610)
    # 4-bit operands: half the bytes, twice the tensor rate
    t4 = bench.shape_roofline_ms(4, shapes, peaks)
    assert t4[1] == pytest.approx(t_roof[1] / 2)
    assert t4[0] == pytest.approx((64 * 64 + 4 * 64 * 64) / 6800e9 * 1e3)


def test_route_names():
    assert bench.route_name(L.ROUTE_FUSED, 256) == "in_kernel_conversion_256"
    assert bench.route_name(L.ROUTE_POPC, 4) == "popcount_v4"
    assert bench.route_name(L.ROUTE_STREAM, 0) == "stream_mma"
    h = bench.route_histogram(None, [(1, 2, 3), (4, 5, 6)], [1.0, 2.0],
                              [(L.ROUTE_FUSED, 128), (L.ROUTE_TABLE, 7)])
    assert h == {"in_kernel_conversion_128": {"shapes": 1, "ms": 1.0},
                 "table": {"shapes": 1, "ms": 2.0}}


def test_unusable_timings_stop_the_sweep():
    ms = [1.0] * 8 + [float("nan"), 0.5, 0.9]
    lib = FakeLib(CANDS, ms, {})
    with pytest.raises(RuntimeError):
        tune.sweep(lib, 8, [(64, 64, 64)], None, None, None, 152)
    assert lib.table == {}


def test_random_shapes_are_off_the_grid():
    shp = tune.random_shapes(200, 5)
    assert len(shp) == 200 and len(set(shp)) > 190
    for m, n, k in shp:
        assert (m, n, k) not in tune.GRID and m % 16 == 0 and n % 16 == 0 and k % 32 == 0
        assert 16 <= min(m, n) and max(m, n, k) <= 16384 and m * n * k <= 2 ** 37
