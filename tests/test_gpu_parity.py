"""GPU parity: the CUDA path against the CPU oracle, bit for bit (0 ULP).

Every input comes from the seeded generators; every expected value from the
oracle.  The det-train page's "Correctness" section sets the bar: full-K
det_gemm equals the combine/finalize composition of 2/4/8/16-way K-shards in
any fold grouping, bitwise, for bf16 and f32, and every output is the exact
sum of the exact products with a single rounding to fp32.
"""
import numpy as np
import pytest
import torch

import exact_sum_gemm_gb300 as dg
from exact_sum_gemm_gb300 import workloads as wl
from gpu_util import assert_bits_equal, bits_of, dev_bf16, dev_f32, fold, np_bits

pytestmark = pytest.mark.gpu

FOLDS = ["all", "left", "right", "tree", "random", "reversed"]


def _digits_np(t):
    return t.cpu().numpy()


# --- workload: 64^3 f32 N(0,1), full-K vs 2/4/8/16-way shards ------------------

def test_small_f32_full_and_shards(oracle_mod):
    A = wl.normal_f32((64, 64), 0, 0)
    B = wl.normal_f32((64, 64), 0, 1)
    want = np_bits(oracle_mod.gemm(A, B))
    want_digits = oracle_mod.gemm_digits(A, B)
    a, b = dev_f32(A), dev_f32(B)
    full = dg.det_gemm(a, b)
    assert_bits_equal(bits_of(full), want, "det_gemm vs oracle")
    np.testing.assert_array_equal(_digits_np(dg.det_gemm_partial(a, b)), want_digits)
    for n_sh in (2, 4, 8, 16):
        for cuts in (wl.equal_cuts(64, n_sh), wl.kshard_cuts(64, n_sh, seed=n_sh)):
            parts = [dg.det_gemm_partial(a[:, k0:k1], b[:, k0:k1]) for k0, k1 in cuts]
            for how in FOLDS:
                acc = fold(parts, how, dg.det_combine, seed=n_sh)
                np.testing.assert_array_equal(_digits_np(acc), want_digits,
                                              err_msg=f"{n_sh} shards, fold {how}")
                assert_bits_equal(bits_of(dg.det_finalize(acc)), want, f"{n_sh} shards {how}")


# --- workload: bf16 512x512x4096, exponents U{-60..60}, planted cancellations -----

def test_bf16_wide_exponents_with_cancellation(oracle_mod):
    a_bits, b_bits, pairs = wl.bf16_wide_with_cancellation(512, 512, 4096, seed=1)
    want_digits = oracle_mod.gemm_digits(a_bits, b_bits, dtype="bf16")
    want = np_bits(oracle_mod.gemm(a_bits, b_bits, dtype="bf16"))
    a, b = dev_bf16(a_bits), dev_bf16(b_bits)
    got = dg.det_gemm(a, b)
    assert_bits_equal(bits_of(got), want, "bf16 det_gemm vs oracle")
    # the cancelled pairs contribute exactly nothing
    keep = np.setdiff1d(np.arange(4096), pairs.ravel())
    got_keep = dg.det_gemm(a[:, keep], b[:, keep])
    assert_bits_equal(bits_of(got_keep), want, "cancellation pairs removed")
    np.testing.assert_array_equal(_digits_np(dg.det_gemm_partial(a, b)), want_digits)
    # every output's digits through 2/4/8/16 random K-shards in six fold orders
    for n_sh in (2, 4, 8, 16):
        cuts = wl.kshard_cuts(4096, n_sh, seed=100 + n_sh)
        parts = [dg.det_gemm_partial(a[:, k0:k1], b[:, k0:k1]) for k0, k1 in cuts]
        for how in FOLDS:
            acc = fold(parts, how, dg.det_combine, seed=n_sh)
            np.testing.assert_array_equal(_digits_np(acc), want_digits,
                                          err_msg=f"{n_sh} shards, fold {how}")
            assert_bits_equal(bits_of(dg.det_finalize(acc)), want, f"{n_sh} shards {how}")


def edge_rows(M, n, seed):
    """At least n rows of an M-row output: both sides of every 128-row tile edge
    (the tensor-core tiles and the row bands start on multiples of 128 and
    256), the first and last rows, and seeded random rows to make up n."""
    rows = {0, M - 1}
    for t in range(128, M, 128):
        rows.update((t - 1, t))
    g = wl.rng(seed, 99)
    while len(rows) < n:
        rows.add(int(g.integers(0, M)))
    return np.array(sorted(rows), np.int64)


# --- workload: 4096^3 f32 N(0,1), the benchmark's launch, sampled rows ------------

def test_bench_size_sampled_rows(oracle_mod):
    A = wl.normal_f32((4096, 4096), 0, 0)
    B = wl.normal_f32((4096, 4096), 0, 1)
    got = bits_of(dg.det_gemm(dev_f32(A), dev_f32(B)))
    rows = edge_rows(4096, 128, seed=0)
    want = np_bits(oracle_mod.gemm(A[rows], B))
    assert_bits_equal(got[rows], want, "4096^3 sampled rows")
    # accuracy against an fp64 matmul on the sampled rows: the fp32 rounding floor
    ref = A[rows].astype(np.float64) @ B.astype(np.float64).T
    c = got[rows].view(np.float32).astype(np.float64)
    assert np.max(np.abs(c - ref) / np.abs(ref)) <= 2.0 ** -24 * 1.01


# --- workload: f32 256x256x2^19, |x| = 2^U[-100,100] (carry headroom) -------------

def test_k_limit_loguniform(oracle_mod):
    K = 1 << 19
    A = wl.loguniform_f32((256, K), 3, 0)
    B = wl.loguniform_f32((256, K), 3, 1)
    a, b = dev_f32(A), dev_f32(B)
    # every output: most overflow fp32, so the digits are compared as well as
    # the rounded values
    want_digits = oracle_mod.gemm_digits(A, B)
    want = np_bits(oracle_mod.finalize(want_digits))
    assert_bits_equal(bits_of(dg.det_gemm(a, b)), want, "K=2^19 all outputs")
    np.testing.assert_array_equal(dg.det_gemm_partial(a, b).cpu().numpy(), want_digits)
    # K-sharding at the limit: 4 ragged shards compose to the same digits
    rows, cols = slice(64, 128), slice(0, 256)
    cuts = wl.kshard_cuts(K, 4, seed=3)
    parts = [dg.det_gemm_partial(a[rows, k0:k1], b[cols, k0:k1]) for k0, k1 in cuts]
    np.testing.assert_array_equal(dg.det_combine(parts).cpu().numpy(),
                                  want_digits[:, rows, cols])


# --- workload: DetLinear 4096->4096 forward / dgrad / wgrad ------------------------

def test_detlinear_fwd_dgrad_wgrad(oracle_mod):
    x_np, w_np = wl.detlinear_inputs()
    x, w = dev_f32(x_np), dev_f32(w_np)
    layer = dg.DetLinear(4096, 4096, device="cuda", weight=w)
    xg = x.clone().requires_grad_(True)
    y = layer(xg)
    y.square().mean().backward()
    # forward: at least 128 of the 2048 rows, on both sides of every tile edge
    rows = edge_rows(2048, 128, seed=1)
    y_rows = oracle_mod.gemm(x_np[rows], w_np)
    assert_bits_equal(bits_of(y)[rows], np_bits(y_rows), "forward")
    # upstream gradient of y.square().mean() is 2y/numel = y * 2^-22 (numel = 2^23),
    # an exact power-of-two scaling; it is formed here from the oracle's y
    scale = np.float32(2.0 ** -22)
    dy_rows = (y_rows * scale).astype(np.float32)
    w_t = np.ascontiguousarray(w_np.T)
    assert_bits_equal(bits_of(xg.grad)[rows], np_bits(oracle_mod.gemm(dy_rows, w_t)), "dgrad")
    # wgrad rows o need dy[:, o] for the whole batch; at least 128 of the 4096
    # rows of dW, on both sides of every tile edge
    orow = edge_rows(4096, 128, seed=2)
    dy_cols = (oracle_mod.gemm(x_np, w_np[orow]) * scale).astype(np.float32)   # [2048, n]
    want_dw = oracle_mod.gemm(np.ascontiguousarray(dy_cols.T), np.ascontiguousarray(x_np.T))
    assert_bits_equal(bits_of(layer.weight.grad)[orow], np_bits(want_dw), "wgrad")


# --- repeatability -------------------------------------------------------------------

def test_repeated_runs_identical():
    A = wl.normal_f32((300, 700), 11, 0)
    B = wl.normal_f32((200, 700), 11, 1)
    a, b = dev_f32(A), dev_f32(B)
    first = bits_of(dg.det_gemm(a, b))
    for _ in range(3):
        assert_bits_equal(bits_of(dg.det_gemm(a, b)), first, "repeat")
