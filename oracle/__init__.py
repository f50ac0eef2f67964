"""CPU oracle for the low-bit GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library's product path never does.

The arithmetic lives in ``lbgemm_oracle.c`` (plain C, int64 sums, threads over
rows of C); this module compiles it with gcc on first use and marshals numpy
arrays through ctypes.  Method source, cited as [LBG]: "Leveraging Large-Scale
Data for Efficient Low-Bit CUTLASS GEMM Optimization via Neural Networks"
(IEEE Transactions on Big Data, press summary page), intro and section 1.

Every function here is pinned by ``tests/test_oracle_pins.py`` against hand-
worked examples, identities and brute force, except ``select.label`` whose pin
is its definition (the argmin of measured times, section 2 of the page).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lbgemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, OVERFLOW, BAD_ARG = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/liboracle.so`` (gcc, -O2, pthreads)."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-Wall", "-Wextra",
             "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def load_lib(path: str):
    """Open a compiled oracle (this one, or a copy built elsewhere) with its signatures."""
    lib = ctypes.CDLL(path)
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    for name in ("oracle_gemm_s8", "oracle_gemm_s4", "oracle_gemm_b1",
                 "oracle_gemm_b1_unpacked"):
        f = getattr(lib, name)
        f.argtypes = [i64, i64, i64, vp, vp, vp, ctypes.c_int]
        f.restype = ctypes.c_int
    lib.oracle_entries.argtypes = [ctypes.c_int, i64, i64, i64, vp, vp, i64, vp, vp, vp]
    lib.oracle_entries.restype = ctypes.c_int
    lib.oracle_linear.argtypes = [i64, i64, i64, vp, vp, vp, vp, vp, ctypes.c_int]
    lib.oracle_linear.restype = ctypes.c_int
    return lib


def _load(lib=None):
    global _lib
    if lib is not None:
        return lib
    with _lock:
        if _lib is None:
            _lib = load_lib(build())
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
               else (os.cpu_count() or 1))


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _check(rc: int, what: str) -> None:
    if rc == OVERFLOW:
        raise OverflowError(f"{what}: a result does not fit int32")
    if rc != OK:
        raise ValueError(f"{what}: bad arguments (rc={rc})")


def row_elems(bits: int, K: int) -> int:
    """Row length of an operand in its storage unit (bytes, bytes, words)."""
    return {8: K, 4: (K + 1) // 2, 1: (K + 31) // 32}[bits]


_DTYPES = {8: np.int8, 4: np.uint8, 1: np.uint32}


def _prep(bits: int, X: np.ndarray, K: int) -> np.ndarray:
    X = np.ascontiguousarray(X)
    if X.dtype != _DTYPES[bits]:
        raise TypeError(f"{bits}-bit operand must be {np.dtype(_DTYPES[bits]).name}, got {X.dtype}")
    if X.ndim != 2 or X.shape[1] != row_elems(bits, K):
        raise ValueError(f"operand shape {X.shape} does not hold rows of K={K} {bits}-bit values")
    return X


def gemm(bits: int, A: np.ndarray, B: np.ndarray, K: int, threads: int | None = None,
         b1_form: str = "popc", lib=None) -> np.ndarray:
    """C[M,N] int32 = A[M,K] . B[N,K]^T for bits in {8, 4, 1}.

    8-bit: int8 arrays [rows, K].  4-bit: uint8 arrays [rows, ceil(K/2)],
    low nibble first.  1-bit: uint32 arrays [rows, ceil(K/32)], bit 1 = +1.
    ``b1_form`` picks the popcount form ("popc") or the unpacked +-1 form
    ("unpacked") for 1-bit operands.
    """
    A = _prep(bits, A, K)
    B = _prep(bits, B, K)
    M, N = A.shape[0], B.shape[0]
    C = np.zeros((M, N), dtype=np.int32)
    lib = _load(lib)
    f = {8: lib.oracle_gemm_s8, 4: lib.oracle_gemm_s4,
         1: lib.oracle_gemm_b1 if b1_form == "popc" else lib.oracle_gemm_b1_unpacked}[bits]
    rc = f(M, N, K, _ptr(A), _ptr(B), _ptr(C), threads or default_threads())
    _check(rc, f"oracle gemm bits={bits}")
    return C


def entries(bits: int, A: np.ndarray, B: np.ndarray, K: int, rows, cols, lib=None) -> np.ndarray:
    """C[rows[i], cols[i]] for each i, computed one by one."""
    A = _prep(bits, A, K)
    B = _prep(bits, B, K)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape:
        raise ValueError("rows and cols differ in length")
    out = np.zeros(rows.shape, dtype=np.int32)
    rc = _load(lib).oracle_entries(bits, A.shape[0], B.shape[0], K, _ptr(A), _ptr(B),
                                rows.size, _ptr(rows), _ptr(cols), _ptr(out))
    _check(rc, f"oracle entries bits={bits}")
    return out


def linear(X: np.ndarray, sx: np.ndarray, W: np.ndarray, sw: np.ndarray,
           threads: int | None = None, lib=None) -> np.ndarray:
    """fp64 reference of the quantised linear layer: (X . W^T) * sx[m] * sw[n]."""
    X = np.ascontiguousarray(X, dtype=np.int8)
    W = np.ascontiguousarray(W, dtype=np.int8)
    sx = np.ascontiguousarray(sx, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    M, K = X.shape
    N = W.shape[0]
    if W.shape[1] != K or sx.shape != (M,) or sw.shape != (N,):
        raise ValueError("linear: inconsistent shapes")
    ref = np.zeros((M, N), dtype=np.float64)
    rc = _load(lib).oracle_linear(M, N, K, _ptr(X), _ptr(sx), _ptr(W), _ptr(sw), _ptr(ref),
                               threads or default_threads())
    _check(rc, "oracle linear")
    return ref


def quantize_rows(x: np.ndarray):
    """Per-row symmetric int8 quantisation, in float32 as the library states it:
    s = max(max|x|, 1e-12) / 127 and q = clamp(round_half_even(x / s), -127, 127)
    (the quantiser in front of a quantised linear layer, [LBG] section 4; the
    page gives none, this is the plainest reading).  x: float32 [M, K]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=1) if x.shape[1] else np.zeros(x.shape[0], np.float32)
    s = np.maximum(amax, np.float32(1e-12)).astype(np.float32) / np.float32(127.0)
    q = np.rint(x / s[:, None].astype(np.float32))
    q = np.clip(q, -127, 127).astype(np.int8)
    return q, s.astype(np.float32)


def linear_quant(x: np.ndarray, W: np.ndarray, sw: np.ndarray, threads: int | None = None,
                 lib=None):
    """fp64 reference of the linear layer on unquantised activations:
    quantize_rows(x), then the quantised linear layer."""
    q, s = quantize_rows(x)
    return linear(q, s, W, sw, threads=threads, lib=lib)
