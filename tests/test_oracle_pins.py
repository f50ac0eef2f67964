"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Method: "Leveraging Large-Scale Data for Efficient Low-Bit CUTLASS GEMM
Optimization via Neural Networks" (press summary page), intro (1-, 4- and
8-bit GEMM) and section 1 (A x B = C accumulated along K); section 4 for the
linear layer.

Each pin is a plain function taking an optional compiled oracle, so the
mutation tests at the bottom can run the same pins against copies of the
oracle with a plausible mistake planted, and check that some pin fails.
"""
import glob
import json
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from oracle import select as osel

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---- independent references (numpy library routines, own unpacking) --------

def ref_unpack_s4(packed: np.ndarray, K: int) -> np.ndarray:
    """Nibbles -> int64 values, written differently from the oracle: a code c
    in [8, 15] stands for c - 16."""
    p = packed.astype(np.int64)
    codes = np.empty((p.shape[0], 2 * p.shape[1]), dtype=np.int64)
    codes[:, 0::2] = p & 15
    codes[:, 1::2] = p >> 4
    vals = np.where(codes >= 8, codes - 16, codes)
    return vals[:, :K]


def ref_unpack_b1(words: np.ndarray, K: int) -> np.ndarray:
    """Words -> +-1 int64 values via numpy's little-endian bit unpacking."""
    by = np.ascontiguousarray(words.astype("<u4")).view(np.uint8)
    bits = np.unpackbits(by, axis=1, bitorder="little")[:, :K].astype(np.int64)
    return 2 * bits - 1


def ref_matmul(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.matmul(a.astype(np.int64), b.astype(np.int64).T)


def _arr(bits, rows):
    return np.array(rows, dtype={8: np.int8, 4: np.uint8, 1: np.uint32}[bits])


# ---- pins -------------------------------------------------------------------

def pin_golden(lib=None):
    files = sorted(glob.glob(os.path.join(GOLDEN, "*.json")))
    assert len(files) >= 7
    for path in files:
        c = json.load(open(path))
        assert c["source"]
        if "X" in c:  # linear layer case
            X, W = np.array(c["X"], np.int8), np.array(c["W"], np.int8)
            sx, sw = np.array(c["sx"], np.float32), np.array(c["sw"], np.float32)
            ref = oracle.linear(X, sx, W, sw, lib=lib)
            np.testing.assert_array_equal(ref, np.array(c["Y"]), err_msg=path)
            acc = oracle.gemm(8, X, W, c["K"], lib=lib)
            np.testing.assert_array_equal(acc, np.array(c["acc"]), err_msg=path)
            continue
        A, B = _arr(c["bits"], c["A"]), _arr(c["bits"], c["B"])
        C = oracle.gemm(c["bits"], A, B, c["K"], lib=lib)
        np.testing.assert_array_equal(C, np.array(c["C"]), err_msg=path)
        if "values_A" in c:
            np.testing.assert_array_equal(ref_unpack_s4(A, c["K"]), np.array(c["values_A"]))
            np.testing.assert_array_equal(ref_unpack_s4(B, c["K"]), np.array(c["values_B"]))
        if c["bits"] == 1:
            C2 = oracle.gemm(1, A, B, c["K"], b1_form="unpacked", lib=lib)
            np.testing.assert_array_equal(C2, np.array(c["C"]), err_msg=path)


def pin_s8_matches_numpy(lib=None):
    g = np.random.default_rng(1)
    for M, N, K in [(37, 29, 301), (1, 1, 1), (5, 64, 2048)]:
        A = g.integers(-128, 128, (M, K)).astype(np.int8)
        B = g.integers(-128, 128, (N, K)).astype(np.int8)
        np.testing.assert_array_equal(oracle.gemm(8, A, B, K, lib=lib), ref_matmul(A, B))


def pin_s4_bruteforce(lib=None):
    """Every pair of packed bytes at K = 2: all 16^4 value combinations."""
    allb = np.arange(256, dtype=np.uint8).reshape(256, 1)
    C = oracle.gemm(4, allb, allb, 2, lib=lib)
    v = ref_unpack_s4(allb, 2)
    np.testing.assert_array_equal(C, ref_matmul(v, v))
    # a few by hand: byte 0x88 holds (-8, -8); 0x77 holds (7, 7)
    assert C[0x88, 0x88] == 128 and C[0x77, 0x88] == -112 and C[0x01, 0x10] == 0


def pin_s4_matches_numpy(lib=None):
    g = np.random.default_rng(2)
    for M, N, K in [(13, 17, 77), (3, 40, 512), (2, 2, 1)]:
        A = g.integers(0, 256, (M, (K + 1) // 2)).astype(np.uint8)
        B = g.integers(0, 256, (N, (K + 1) // 2)).astype(np.uint8)
        np.testing.assert_array_equal(oracle.gemm(4, A, B, K, lib=lib),
                                      ref_matmul(ref_unpack_s4(A, K), ref_unpack_s4(B, K)))


def pin_b1_bruteforce(lib=None):
    """Every pair of 8-bit patterns at K = 8, with garbage in the padding bits."""
    g = np.random.default_rng(3)
    pat = np.arange(256, dtype=np.uint32)
    A = (pat | (g.integers(0, 1 << 24, 256).astype(np.uint32) << 8)).reshape(256, 1)
    B = (pat | (g.integers(0, 1 << 24, 256).astype(np.uint32) << 8)).reshape(256, 1)
    want = ref_matmul(ref_unpack_b1(A, 8), ref_unpack_b1(B, 8))
    np.testing.assert_array_equal(oracle.gemm(1, A, B, 8, lib=lib), want)
    np.testing.assert_array_equal(oracle.gemm(1, A, B, 8, b1_form="unpacked", lib=lib), want)


def pin_b1_matches_numpy(lib=None):
    g = np.random.default_rng(4)
    for M, N, K in [(9, 11, 32), (7, 5, 40), (6, 6, 95), (4, 33, 1024)]:
        nw = (K + 31) // 32
        A = g.integers(0, 1 << 32, (M, nw), dtype=np.uint64).astype(np.uint32)
        B = g.integers(0, 1 << 32, (N, nw), dtype=np.uint64).astype(np.uint32)
        want = ref_matmul(ref_unpack_b1(A, K), ref_unpack_b1(B, K))
        np.testing.assert_array_equal(oracle.gemm(1, A, B, K, lib=lib), want)
        np.testing.assert_array_equal(oracle.gemm(1, A, B, K, b1_form="unpacked", lib=lib), want)


def pin_identities(lib=None):
    g = np.random.default_rng(5)
    K = 64
    A = g.integers(-128, 128, (10, K)).astype(np.int8)
    eye = np.eye(K, dtype=np.int8)
    np.testing.assert_array_equal(oracle.gemm(8, A, eye, K, lib=lib), A.astype(np.int32))
    np.testing.assert_array_equal(oracle.gemm(8, np.zeros_like(A), A, K, lib=lib), 0)
    ones = np.ones((3, K), np.int8)
    np.testing.assert_array_equal(oracle.gemm(8, ones, ones, K, lib=lib), K)
    neg = np.full((2, K), -128, np.int8)
    np.testing.assert_array_equal(oracle.gemm(8, neg, neg, K, lib=lib), 16384 * K)
    # 4-bit identity: nibble code 1 on the diagonal
    eye4 = np.zeros((K, K // 2), np.uint8)
    for k in range(K):
        eye4[k, k // 2] |= np.uint8(1 << (4 * (k % 2)))
    A4 = g.integers(0, 256, (6, K // 2)).astype(np.uint8)
    np.testing.assert_array_equal(oracle.gemm(4, A4, eye4, K, lib=lib), ref_unpack_s4(A4, K))
    m8 = np.full((2, K // 2), 0x88, np.uint8)
    np.testing.assert_array_equal(oracle.gemm(4, m8, m8, K, lib=lib), 64 * K)
    # 1-bit closed forms: a . a = K, a . ~a = -K
    Kb = 96
    a = g.integers(0, 1 << 32, (4, 3), dtype=np.uint64).astype(np.uint32)
    C = oracle.gemm(1, a, np.concatenate([a, ~a]), Kb, lib=lib)
    np.testing.assert_array_equal(np.diag(C[:, :4]), Kb)
    np.testing.assert_array_equal(np.diag(C[:, 4:]), -Kb)
    # transpose symmetry and linearity
    B = g.integers(-128, 128, (7, K)).astype(np.int8)
    np.testing.assert_array_equal(oracle.gemm(8, B, A, K, lib=lib),
                                  oracle.gemm(8, A, B, K, lib=lib).T)
    A1 = g.integers(-63, 64, (5, K)).astype(np.int8)
    A2 = g.integers(-64, 64, (5, K)).astype(np.int8)
    np.testing.assert_array_equal(oracle.gemm(8, (A1 + A2).astype(np.int8), B, K, lib=lib),
                                  oracle.gemm(8, A1, B, K, lib=lib) + oracle.gemm(8, A2, B, K, lib=lib))


def pin_overflow(lib=None):
    K = 131071  # 16384 * K = 2147467264 still fits int32
    neg = np.full((1, K), -128, np.int8)
    assert oracle.gemm(8, neg, neg, K, lib=lib)[0, 0] == 16384 * K
    K = 131072  # 2^31 does not fit
    neg = np.full((1, K), -128, np.int8)
    with pytest.raises(OverflowError):
        oracle.gemm(8, neg, neg, K, lib=lib)


def pin_entries(lib=None):
    g = np.random.default_rng(6)
    for bits, K in [(8, 200), (4, 130), (1, 320)]:
        rows = {8: K, 4: (K + 1) // 2, 1: (K + 31) // 32}[bits]
        dt = {8: np.int8, 4: np.uint8, 1: np.uint32}[bits]
        if bits == 8:
            A = g.integers(-128, 128, (21, rows)).astype(dt)
            B = g.integers(-128, 128, (19, rows)).astype(dt)
        else:
            A = g.integers(0, 1 << (8 if bits == 4 else 32), (21, rows), dtype=np.uint64).astype(dt)
            B = g.integers(0, 1 << (8 if bits == 4 else 32), (19, rows), dtype=np.uint64).astype(dt)
        r = g.integers(0, 21, 50)
        c = g.integers(0, 19, 50)
        full = oracle.gemm(bits, A, B, K, lib=lib)
        np.testing.assert_array_equal(oracle.entries(bits, A, B, K, r, c, lib=lib), full[r, c])


def pin_linear(lib=None):
    g = np.random.default_rng(7)
    M, N, K = 3, 5, 40
    X = g.integers(-127, 128, (M, K)).astype(np.int8)
    W = g.integers(-127, 128, (N, K)).astype(np.int8)
    X[1] = 0
    sx = g.random(M).astype(np.float32)
    sw = g.random(N).astype(np.float32)
    ref = oracle.linear(X, sx, W, sw, lib=lib)
    acc = ref_matmul(X, W)
    for m in range(M):
        for n in range(N):
            assert ref[m, n] == float(acc[m, n]) * float(sx[m]) * float(sw[n])
    assert np.all(ref[1] == 0)


def pin_quantize(lib=None):
    """Per-row quantiser: a hand-worked row, the zero row, and the bounds that
    hold for any row (the row's absmax maps to +-127, |q| <= 127, and q*s is
    within s/2 (plus fp32 rounding) of x)."""
    q, s = oracle.quantize_rows(np.array([[1.0, -4.0, 0.5], [0.0, 0.0, 0.0]], np.float32))
    # row 0: s = 4/127, x/s = (31.75, -127, 15.875) -> (32, -127, 16)
    assert q[0].tolist() == [32, -127, 16] and s[0] == np.float32(4.0) / np.float32(127.0)
    assert q[1].tolist() == [0, 0, 0] and s[1] == np.float32(1e-12) / np.float32(127.0)
    g = np.random.default_rng(8)
    x = (g.standard_normal((50, 333)) * g.uniform(0.01, 100, (50, 1))).astype(np.float32)
    q, s = oracle.quantize_rows(x)
    assert np.all(np.abs(q.astype(int)) <= 127)
    am = np.argmax(np.abs(x), axis=1)
    assert np.all(np.abs(q[np.arange(50), am].astype(int)) == 127)
    err = np.abs(q.astype(np.float64) * s[:, None] - x)
    assert np.all(err <= s[:, None] * (0.5 + 1e-5))
    # the quantised linear reference is the linear reference of the codes
    W = g.integers(-127, 128, (4, 333)).astype(np.int8)
    sw = g.random(4).astype(np.float32)
    np.testing.assert_array_equal(oracle.linear_quant(x[:3], W, sw, lib=lib),
                                  oracle.linear(q[:3], s[:3], W, sw, lib=lib))


PINS = [pin_golden, pin_quantize, pin_s8_matches_numpy, pin_s4_bruteforce, pin_s4_matches_numpy,
        pin_b1_bruteforce, pin_b1_matches_numpy, pin_identities, pin_overflow, pin_entries,
        pin_linear]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin()


# ---- planted mistakes: each must make at least one pin fail -----------------

MUTATIONS = {
    "dropped_last_k": ("for (int64_t k = 0; k < K; ++k) s += (int64_t)a[k] * (int64_t)b[k];",
                       "for (int64_t k = 0; k + 1 < K; ++k) s += (int64_t)a[k] * (int64_t)b[k];"),
    "b_read_unsigned": ("s += (int64_t)a[k] * (int64_t)b[k];",
                        "s += (int64_t)a[k] * (int64_t)(uint8_t)b[k];"),
    "nibble_order_swapped": ("(k % 2 == 0) ? (byte & 0xFu) : (byte >> 4)",
                             "(k % 2 == 1) ? (byte & 0xFu) : (byte >> 4)"),
    "nibble_unsigned": ("(int)(nib ^ 8u) - 8", "(int)nib"),
    "b1_missing_factor_two": ("return K - 2 * diff;", "return K - diff;"),
    "b1_padding_unmasked": ("if (valid < 32) x &= (1u << valid) - 1u;", ""),
    "b1_bit_order_reversed": ("(row[k / 32] >> (k % 32)) & 1u", "(row[k / 32] >> (31 - k % 32)) & 1u"),
    "popcount_wrong": ("x &= x - 1u;", "x >>= 1;"),
    "overflow_unchecked": ("if (s > INT32_MAX || s < INT32_MIN) j->overflow = 1;", ""),
    "linear_wrong_scale": ("* (double)sw[n]", "* (double)sw[0]"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc missing")
    old, new = MUTATIONS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "lbgemm_oracle.c")).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old}"
    mut = tmp_path / "mut.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-o", str(so), str(mut)])
    lib = oracle.load_lib(str(so))
    caught = []
    for pin in PINS:
        try:
            pin(lib)
        except (AssertionError, OverflowError, ValueError, pytest.fail.Exception) as e:
            caught.append((pin.__name__, type(e).__name__))
    assert caught, f"no pin caught the planted mistake {name}"


# ---- selection-rule oracle (definition pins, hand-worked) --------------------

def test_select_label_and_choice():
    t = [5.0, 4.0, 4.0, 9.0, 9.0, 9.0, 9.0, 4.05, 9.0]
    assert osel.label(t) == 1                      # argmin, lowest index on ties
    assert osel.table_choice(t) == osel.DEFAULT_VARIANT  # default within 2 %
    t[7] = 4.5
    assert osel.table_choice(t) == 1
    assert osel.DEFAULT_VARIANT == 7 and osel.variant_of(7) == (2, 5)
    assert osel.variant_of(0) == (0, 2) and osel.variant_of(8) == (2, 6)
    assert [osel.variant_index(*osel.variant_of(i)) for i in range(9)] == list(range(9))


def test_select_nearest():
    e = [((64, 64, 64), 0), ((4096, 4096, 4096), 8), ((4096, 64, 4096), 5)]
    assert osel.nearest(e, 64, 64, 64) == 0
    assert osel.nearest(e, 8192, 8192, 8192) == 8
    assert osel.nearest(e, 4096, 128, 4096) == 5
    assert osel.nearest([], 1, 1, 1) == osel.DEFAULT_VARIANT
