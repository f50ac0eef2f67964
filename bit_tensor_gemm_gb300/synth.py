"""Seeded synthetic operands for the low-bit GEMM.

This module only draws random numbers and lays them out in the library's
operand formats; it holds none of the GEMM's arithmetic, and both the CPU
oracle and the GPU path read what it produces.

Formats (rows are K-major; A is [M, K], B is [N, K]):
  8-bit  int8 [rows, K]
  4-bit  uint8 [rows, ceil(K/2)]: two signed nibbles per byte, element 2j in
         the low nibble of byte j.  A uniform random byte holds two nibbles
         each uniform over the 16 codes, i.e. values uniform over [-8, 7].
  1-bit  uint32 [rows, ceil(K/32)]: element k is bit k%32 of word k/32, bit 1
         meaning +1.  A uniform random word holds 32 bits with p = 0.5.
Padding nibbles/bits past K in a row's last byte/word are zero.

The linear-layer recipe draws x ~ N(0, 1) and quantises it symmetrically per
row: s = max(absmax, 1e-12) / 127, q = clamp(round_half_even(x / s), -127, 127).
"""
from __future__ import annotations

import numpy as np

BASE_SEED = 20261202


def config_seed(config_id: int) -> int:
    """Seed of a named workload: the base seed plus the workload's number."""
    return BASE_SEED + config_id


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def s8(g: np.random.Generator, rows: int, K: int, lo: int = -127, hi: int = 127) -> np.ndarray:
    """int8 [rows, K], uniform over [lo, hi]."""
    return g.integers(lo, hi + 1, size=(rows, K), dtype=np.int16).astype(np.int8)


def s4(g: np.random.Generator, rows: int, K: int) -> np.ndarray:
    """uint8 [rows, ceil(K/2)] of packed nibbles, each value uniform over [-8, 7]."""
    nb = (K + 1) // 2
    out = g.integers(0, 256, size=(rows, nb), dtype=np.int16).astype(np.uint8)
    if K % 2:
        out[:, -1] &= np.uint8(0x0F)
    return out


def b1(g: np.random.Generator, rows: int, K: int) -> np.ndarray:
    """uint32 [rows, ceil(K/32)] of packed +-1 bits, p = 0.5."""
    nw = (K + 31) // 32
    out = g.integers(0, 1 << 32, size=(rows, nw), dtype=np.uint64).astype(np.uint32)
    if K % 32:
        out[:, -1] &= np.uint32((1 << (K % 32)) - 1)
    return out


def operands(bits: int, M: int, N: int, K: int, seed: int):
    """(A, B) for one GEMM, A drawn first, then B, from one seeded stream."""
    g = rng(seed)
    draw = {8: s8, 4: s4, 1: b1}[bits]
    A = draw(g, M, K)
    B = draw(g, N, K)
    return A, B


def quantize_rows(x: np.ndarray):
    """Symmetric per-row int8 quantisation: returns (q int8, scale float32)."""
    absmax = np.abs(x).max(axis=1)
    s = (np.maximum(absmax, 1e-12) / 127.0).astype(np.float32)
    q = np.clip(np.rint(x / s[:, None]), -127, 127).astype(np.int8)
    return q, s


def linear_operands(M: int, N: int, K: int, seed: int):
    """(X int8 [M,K], sx f32 [M], W int8 [N,K], sw f32 [N]) from N(0,1) draws."""
    g = rng(seed)
    x = g.standard_normal((M, K), dtype=np.float32)
    w = g.standard_normal((N, K), dtype=np.float32)
    X, sx = quantize_rows(x)
    W, sw = quantize_rows(w)
    return X, sx, W, sw
