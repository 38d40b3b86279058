"""Pins for the CPU oracle: tie it to things other than itself.

Each test checks the oracle against something the det-train page or plain
mathematics fixes (page section "Method": the exact sum of the exact products,
rounded to fp32 a single time; section "Correctness": K-shard/fold invariance
and the fp32 rounding floor against an fp64 matmul):
  * exact-rational brute force on tiny inputs (fractions.Fraction);
  * the small-integer special case (exact int64 GEMM + one RNE cast);
  * K = 1, which is one RNE of an exact double (numpy's cast);
  * math.fsum (correctly rounded double of the exact sum);
  * hand-derived worked cases (tests/golden/worked_cases.json);
  * invariants: K-shards, permutation, negation, transpose, 2^s scaling;
  * the accuracy bound against an fp64 matmul.
A plausible mistake anywhere in the oracle (a dropped or doubled product, a
wrong sign or index, a transposed operand, a rounding slip at ties,
subnormals or overflow) fails at least one of them.
"""
import json
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

from exact_ref import (NAN_BITS, bf16_to_fraction, brute_gemm_bits, exact_dot,
                       round_to_f32_bits)
from exact_sum_gemm_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_cases.json")


def bits(x):
    return np.asarray(x, np.float32).view(np.uint32)


def f32_to_bf16_bits(x):
    b = bits(x)
    assert np.all((b & 0xFFFF) == 0), "value is not representable in bf16"
    return (b >> 16).astype(np.uint16)


# --- the test-side rounding routine is itself pinned to a library routine ---

def test_fraction_rounding_matches_numpy_cast_of_doubles():
    g = np.random.default_rng(123)
    vals = []
    # random doubles over the whole binary32 range, incl. subnormal and overflow
    e = g.integers(-160, 130, size=4000)
    m = g.random(4000) + 1.0
    vals += list(np.ldexp(m, e) * np.where(g.random(4000) < 0.5, -1, 1))
    # exact midpoints and neighbours
    for k in range(200):
        f = np.float32(np.ldexp(g.random() + 1.0, int(g.integers(-150, 128))))
        nxt = np.nextafter(f, np.float32(np.inf))
        if np.isfinite(nxt):
            mid = (float(f) + float(nxt)) / 2
            vals += [mid, np.nextafter(mid, 0.0), np.nextafter(mid, np.inf)]
    vals += [2.0 ** -150, 2.0 ** -151, 3 * 2.0 ** -151, 2.0 ** 128 - 2.0 ** 103,
             2.0 ** 128 - 2.0 ** 102, float(np.finfo(np.float32).max)]
    for v in vals:
        want = int(np.float32(v).view(np.uint32))
        got = round_to_f32_bits(Fraction(v))
        if v != 0 and np.float32(v) == 0:      # numpy keeps the sign of tiny values
            assert got == want, v
        assert got == want, (v, hex(got), hex(want))


# --- brute force on tiny inputs ----------------------------------------------

def _tiny_f32(g, shape, mode):
    if mode == "normal":
        return g.standard_normal(shape).astype(np.float32)
    if mode == "wide":
        e = g.integers(-149, 128, size=shape)
        m = g.random(shape) + 1.0
        x = np.ldexp(m, e).astype(np.float32)
        return np.where(g.random(shape) < 0.5, -x, x).astype(np.float32)
    if mode == "subnormal":
        bitsv = g.integers(1, 1 << 23, size=shape).astype(np.uint32)
        bitsv |= (g.integers(0, 2, size=shape).astype(np.uint32) << 31)
        return bitsv.view(np.float32)
    if mode == "ties":
        # values whose products land on rounding midpoints often
        e = g.integers(-30, 30, size=shape)
        m = g.integers(1, 1 << 13, size=shape) / float(1 << 12)
        x = np.ldexp(m, e).astype(np.float32)
        return np.where(g.random(shape) < 0.5, -x, x).astype(np.float32)
    raise ValueError(mode)


@pytest.mark.parametrize("mode", ["normal", "wide", "subnormal", "ties"])
def test_oracle_matches_exact_rationals_f32(oracle_mod, mode):
    g = np.random.default_rng({"normal": 1, "wide": 2, "subnormal": 3, "ties": 4}[mode])
    for trial in range(120):
        M, N, K = (int(v) for v in g.integers(1, 5, size=3))
        K = int(g.integers(0, 9))
        A = _tiny_f32(g, (M, K), mode)
        B = _tiny_f32(g, (N, K), mode)
        if mode == "wide" and K >= 2 and trial % 3 == 0:
            # plant an exact cancellation between the first two products
            A[:, 1] = -A[:, 0]
            B[:, 1] = B[:, 0]
        got = oracle_mod.gemm(A, B).view(np.uint32)
        want = brute_gemm_bits(A, B)
        np.testing.assert_array_equal(got, want, err_msg=f"trial {trial} M{M} N{N} K{K}")


def test_oracle_matches_exact_rationals_bf16(oracle_mod):
    g = np.random.default_rng(5)
    for trial in range(150):
        M, N = (int(v) for v in g.integers(1, 4, size=2))
        K = int(g.integers(0, 9))
        a = g.integers(0, 1 << 16, size=(M, K)).astype(np.uint16)
        b = g.integers(0, 1 << 16, size=(N, K)).astype(np.uint16)
        # keep them finite: clear exponent-all-ones patterns
        a[(a & 0x7F80) == 0x7F80] &= 0xBFFF
        b[(b & 0x7F80) == 0x7F80] &= 0xBFFF
        got = oracle_mod.gemm(a, b, dtype="bf16").view(np.uint32)
        for m in range(M):
            for n in range(N):
                s = sum((bf16_to_fraction(a[m, k]) * bf16_to_fraction(b[n, k])
                         for k in range(K)), Fraction(0))
                assert int(got[m, n]) == round_to_f32_bits(s), (trial, m, n)


def test_oracle_digits_are_the_exact_sum(oracle_mod):
    g = np.random.default_rng(6)
    A = _tiny_f32(g, (3, 7), "wide")
    B = _tiny_f32(g, (2, 7), "wide")
    P = oracle_mod.gemm_digits(A, B)
    assert P.shape == (20, 3, 2)
    for m in range(3):
        for n in range(2):
            s, _ = exact_dot(A[m].tolist(), B[n].tolist())
            assert oracle_mod.digits_value(P[:, m, n]) == s
            d = P[:18, m, n]
            assert np.all((d[:17] >= 0) & (d[:17] < 2 ** 32))     # canonical form
    assert np.all(P[18] == 7) and np.all(P[19] == 0)


# --- special cases that reduce to library routines ----------------------------

def test_small_integer_case_is_int64_gemm_then_one_rounding(oracle_mod):
    g = np.random.default_rng(7)
    for K, lim in [(64, 1 << 20), (257, 1 << 23), (1000, 1 << 12)]:
        A = g.integers(-lim, lim, size=(9, K))
        B = g.integers(-lim, lim, size=(11, K))
        exact = A.astype(np.int64) @ B.astype(np.int64).T          # |.| < 2^63
        want = exact.astype(np.float32)                            # one RNE (C cast)
        got = oracle_mod.gemm(A.astype(np.float32), B.astype(np.float32))
        np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))


def test_k1_is_one_rounding_of_an_exact_double(oracle_mod):
    g = np.random.default_rng(8)
    for mode in ["normal", "wide", "subnormal"]:
        A = _tiny_f32(g, (40, 1), mode)
        B = _tiny_f32(g, (30, 1), mode)
        want = (A.astype(np.float64) @ B.astype(np.float64).T).astype(np.float32)
        got = oracle_mod.gemm(A, B)
        np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))


def _is_f32_midpoint(d):
    if not np.isfinite(d) or d == 0:
        return False
    f = np.float32(d)
    lo = f if float(f) <= d else np.nextafter(f, np.float32(-np.inf))
    hi = np.nextafter(lo, np.float32(np.inf))
    if not np.isfinite(hi):
        hi_v = 2.0 ** 128 if lo > 0 else float(hi)
    else:
        hi_v = float(hi)
    return (float(lo) + hi_v) / 2 == d


@pytest.mark.parametrize("dist", ["normal", "wide", "cancel"])
def test_fsum_cross_check(oracle_mod, dist):
    g = np.random.default_rng({"normal": 9, "wide": 10, "cancel": 11}[dist])
    M, N, K = 12, 10, 300
    if dist == "normal":
        A = g.standard_normal((M, K)).astype(np.float32)
        B = g.standard_normal((N, K)).astype(np.float32)
    else:
        A = _tiny_f32(g, (M, K), "wide")
        B = _tiny_f32(g, (N, K), "wide")
        A = np.clip(A, -1e30, 1e30).astype(np.float32)        # keep double products finite
        if dist == "cancel":
            A[:, K // 2:] = -A[:, :K // 2]
            B[:, K // 2:] = B[:, :K // 2]
            A[:, 0] = np.float32(1e-30)
    got = oracle_mod.gemm(A, B)
    checked = 0
    for m in range(M):
        for n in range(N):
            d = math.fsum(float(x) * float(y) for x, y in zip(A[m], B[n]))
            if _is_f32_midpoint(d):
                continue
            checked += 1
            assert got[m, n].view(np.uint32) == np.float32(d).view(np.uint32), (m, n, d)
    assert checked > 0.9 * M * N


# --- worked cases -------------------------------------------------------------

def _golden_cases():
    with open(GOLDEN) as f:
        data = json.load(f)
    for case in data["cases"]:
        for dt in case["dtypes"]:
            yield pytest.param(case, dt, id=f"{case['name']}-{dt}")


def _hexf(s):
    return float.fromhex(s) if s not in ("inf", "-inf", "nan") else float(s)


@pytest.mark.parametrize("case,dtype", list(_golden_cases()))
def test_worked_case(oracle_mod, case, dtype):
    a = np.array([[_hexf(v) for v in case["a"]]], np.float32)
    b = np.array([[_hexf(v) for v in case["b"]]], np.float32)
    want = int(case["expected"], 16)
    if dtype == "bf16":
        got = oracle_mod.gemm(f32_to_bf16_bits(a), f32_to_bf16_bits(b), dtype="bf16")
    else:
        got = oracle_mod.gemm(a, b)
    assert int(got.view(np.uint32)[0, 0]) == want
    # the exact-rational brute force agrees with the hand derivation
    if dtype == "f32":
        assert int(brute_gemm_bits(a, b)[0, 0]) == want


def test_top_range_cancellation_at_k_limit(oracle_mod):
    K = 1 << 19
    a = np.full((1, K), 2.0 ** 127, np.float32)
    b = np.full((1, K), 2.0 ** 127, np.float32)
    b[0, 1::2] *= -1
    got = oracle_mod.gemm(a, b)
    assert int(got.view(np.uint32)[0, 0]) == 0
    b[0, 1] = 2.0 ** 127                      # now two surplus products: 2 * 2^254
    got = oracle_mod.gemm(a, b)
    assert np.isinf(got[0, 0]) and got[0, 0] > 0
    P = oracle_mod.gemm_digits(a, b)
    assert oracle_mod.digits_value(P[:, 0, 0]) == Fraction(2) ** 255


# --- invariants -----------------------------------------------------------------

def _sum_planes(parts):
    return np.sum(np.stack(parts), axis=0)


@pytest.mark.parametrize("dist", ["normal", "bf16wide"])
def test_kshard_and_fold_invariance(oracle_mod, dist):
    if dist == "normal":
        A = wl.normal_f32((17, 200), 0, 0)
        B = wl.normal_f32((13, 200), 0, 1)
        dtype = "f32"
    else:
        A, B, _ = wl.bf16_wide_with_cancellation(17, 13, 200, seed=1)
        dtype = "bf16"
    full = oracle_mod.gemm_digits(A, B, dtype)
    fullc = oracle_mod.gemm(A, B, dtype)
    for n_sh in (2, 4, 8, 16):
        for cuts in (wl.equal_cuts(200, n_sh), wl.kshard_cuts(200, n_sh, seed=n_sh)):
            parts = [oracle_mod.gemm_digits(A[:, k0:k1], B[:, k0:k1], dtype) for k0, k1 in cuts]
            summed = oracle_mod.canonicalize(_sum_planes(parts))
            np.testing.assert_array_equal(summed, full)
            np.testing.assert_array_equal(oracle_mod.finalize(_sum_planes(parts)).view(np.uint32),
                                          fullc.view(np.uint32))


def test_permutation_negation_transpose_scaling(oracle_mod):
    A = wl.loguniform_f32((9, 150), 3, 0, lo=-40, hi=40)
    B = wl.loguniform_f32((7, 150), 3, 1, lo=-40, hi=40)
    C = oracle_mod.gemm(A, B)
    perm = np.random.default_rng(0).permutation(150)
    np.testing.assert_array_equal(oracle_mod.gemm(A[:, perm], B[:, perm]).view(np.uint32),
                                  C.view(np.uint32))
    np.testing.assert_array_equal(oracle_mod.gemm(-A, B), -C)
    np.testing.assert_array_equal(oracle_mod.gemm(B, A).view(np.uint32), C.T.view(np.uint32))
    for s in (-20, 7):
        As = np.ldexp(A, s).astype(np.float32)
        want = np.ldexp(C.astype(np.float64), s)
        ok = (np.abs(want) >= 2.0 ** -126) & (np.abs(want) < 2.0 ** 127)
        got = oracle_mod.gemm(As, B)
        np.testing.assert_array_equal(got[ok], want[ok].astype(np.float32))


def test_accuracy_against_fp64_matmul(oracle_mod):
    # det-train page, "Correctness": relative error vs an fp64 matmul sits at
    # the fp32 rounding floor.  Bound: |c - r| <= 2^-24 |r| + gamma_K sum|ab| (1 + 2^-24).
    for A, B in [(wl.normal_f32((64, 64), 0, 0), wl.normal_f32((64, 64), 0, 1)),
                 (wl.normal_f32((48, 1024), 5, 0), wl.normal_f32((40, 1024), 5, 1))]:
        K = A.shape[1]
        c = oracle_mod.gemm(A, B).astype(np.float64)
        r = A.astype(np.float64) @ B.astype(np.float64).T
        absum = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64)).T
        gamma = K * 2.0 ** -53 / (1 - K * 2.0 ** -53)
        bound = 2.0 ** -24 * np.abs(r) + gamma * absum * (1 + 2.0 ** -24)
        assert np.all(np.abs(c - r) <= bound)
        rel = np.abs(c - r) / np.abs(r)
        assert rel.max() <= 2.0 ** -24 * 1.001


def test_finalize_and_canonicalize_on_raw_digits(oracle_mod):
    g = np.random.default_rng(12)
    P = np.zeros((20, 50), np.int64)
    P[:18] = g.integers(-(2 ** 50), 2 ** 50, size=(18, 50))
    P[:18, :10] = g.integers(-3, 3, size=(18, 10))
    P[17, 10:] = g.integers(-(2 ** 20), 2 ** 20, size=40)   # keep magnitudes finite-ish
    P[19, 45:] = 1                                          # non-finite count
    out = oracle_mod.finalize(P).view(np.uint32)
    can = oracle_mod.canonicalize(P)
    assert np.all((can[:17] >= 0) & (can[:17] < 2 ** 32))
    for i in range(50):
        v = oracle_mod.digits_value(P[:, i])
        assert oracle_mod.digits_value(can[:, i]) == v
        want = NAN_BITS if i >= 45 else round_to_f32_bits(v)
        assert int(out[i]) == want, i
    np.testing.assert_array_equal(oracle_mod.canonicalize(can), can)
