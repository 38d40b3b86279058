"""Exact-rational brute force, used only to pin the oracle.

Written from the definitions, independently of ``oracle/``: the exact sum of
products is a ``fractions.Fraction``; rounding to binary32 follows IEEE-754
round-to-nearest-ties-to-even with gradual underflow and overflow to inf.  The
rounding routine is itself pinned against numpy's double->float32 conversion
in ``test_oracle_pins.py``.
"""
from __future__ import annotations

import struct
from fractions import Fraction

import numpy as np

F32_MIN_Q = -149          # exponent of the smallest subnormal
F32_MAX_Q = 104           # exponent of one ulp at the top binade
NAN_BITS = 0x7FC00000


def _floor_log2(x: Fraction) -> int:
    """floor(log2 x) for x > 0, by integer arithmetic."""
    n, d = x.numerator, x.denominator
    e = n.bit_length() - d.bit_length()
    # 2^e <= x < 2^(e+1) must hold; adjust by at most one step
    if e >= 0:
        if n < d << e:
            e -= 1
    else:
        if n << -e < d:
            e -= 1
    return e


def round_to_f32_bits(x: Fraction, zero_sign_of=None) -> int:
    """binary32 bit pattern of RNE(x).

    An exact zero is +0 (``zero_sign_of`` is ignored for it).  A nonzero x that
    rounds to zero keeps its sign.
    """
    if x == 0:
        return 0
    sign = 0x80000000 if x < 0 else 0
    a = -x if x < 0 else x
    e = _floor_log2(a)
    q_exp = max(e - 23, F32_MIN_Q)
    unit = Fraction(2) ** q_exp
    q = a // unit                          # floor
    rem = a - q * unit
    half = unit / 2
    if rem > half or (rem == half and q % 2 == 1):
        q += 1
    if q == 1 << 24:
        q >>= 1
        q_exp += 1
    if q_exp > F32_MAX_Q:
        return sign | 0x7F800000
    if q == 0:
        return sign
    if q < (1 << 23):                      # subnormal (q_exp == -149)
        return sign | int(q)
    biased = q_exp + 23 + 127
    return sign | (biased << 23) | (int(q) - (1 << 23))


def f32_bits_to_fraction(bits: int) -> Fraction:
    """Exact value of a finite binary32 pattern."""
    (f,) = struct.unpack("<f", struct.pack("<I", bits & 0xFFFFFFFF))
    return Fraction(f)


def bf16_to_fraction(bits: int) -> Fraction:
    return f32_bits_to_fraction((int(bits) & 0xFFFF) << 16)


def exact_dot(a_vals, b_vals) -> tuple:
    """(exact Fraction sum, any non-finite) of the products of two sequences."""
    total = Fraction(0)
    nonfinite = False
    for a, b in zip(a_vals, b_vals):
        fa, fb = float(a), float(b)
        if not (np.isfinite(fa) and np.isfinite(fb)):
            nonfinite = True
            continue
        total += Fraction(fa) * Fraction(fb)
    return total, nonfinite


def brute_gemm_bits(A, B) -> np.ndarray:
    """uint32 result patterns of the exact GEMM of f32 arrays A [M,K], B [N,K]."""
    A = np.asarray(A, np.float32)
    B = np.asarray(B, np.float32)
    M, N = A.shape[0], B.shape[0]
    out = np.zeros((M, N), np.uint32)
    for m in range(M):
        for n in range(N):
            s, nf = exact_dot(A[m].tolist(), B[n].tolist())
            out[m, n] = NAN_BITS if nf else round_to_f32_bits(s)
    return out
