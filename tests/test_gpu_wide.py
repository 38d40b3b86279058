"""The wide residue path against the oracle, bit for bit.

Tiles whose operand rows span more binades than the narrow residue path's
18-binade grid (and its deep lists) covers go to the wide path: every row on
its own integer grid from its smallest element, up to 40 moduli, the same
tensor-core GEMM, a multi-limb CRT.  These tests draw such data (log-uniform
magnitudes, bf16 with exponents over +-60, subnormals, zero rows, both operand
layouts), compare every output and every digit with the oracle, and check
through det_tile_routes that the wide path (not the general kernel) computed
the tiles -- or, for rows it must not take (Inf/NaN, a spread beyond its
window), that those tiles went to the general kernel.
"""
import numpy as np
import pytest
import torch

import exact_sum_gemm_gb300 as dg
from exact_sum_gemm_gb300 import _native
from exact_sum_gemm_gb300 import workloads as wl
from gpu_util import assert_bits_equal, bits_of, dev_bf16, dev_f32, np_bits

pytestmark = pytest.mark.gpu


def _check(oracle_mod, A, B, dtype="f32", layouts=("NN",)):
    to_dev = dev_f32 if dtype == "f32" else dev_bf16
    want = np_bits(oracle_mod.gemm(A, B, dtype=dtype))
    want_digits = oracle_mod.gemm_digits(A, B, dtype=dtype)
    routes = []
    for tag in layouts:
        a = to_dev(A) if tag[0] == "N" else to_dev(np.ascontiguousarray(A.T)).t()
        b = to_dev(B) if tag[1] == "N" else to_dev(np.ascontiguousarray(B.T)).t()
        assert_bits_equal(bits_of(dg.det_gemm(a, b)), want, f"{dtype} {tag} det_gemm")
        routes.append(_native.tile_routes())
        np.testing.assert_array_equal(dg.det_gemm_partial(a, b).cpu().numpy(), want_digits,
                                      err_msg=f"{dtype} {tag} digits")
        routes.append(_native.tile_routes())
    return routes


def _all_wide(routes):
    for r in routes:
        assert r["general"] == r["tiles"] and r["wide"] == r["tiles"] and r["kulisch"] == 0, r


@pytest.mark.parametrize("M,N,K", [(300, 260, 777), (129, 257, 64), (64, 64, 4096), (1, 70, 33)])
def test_wide_f32_loguniform(oracle_mod, M, N, K):
    A = wl.loguniform_f32((M, K), 71, 0, lo=-40, hi=40)
    B = wl.loguniform_f32((N, K), 71, 1, lo=-40, hi=40)
    _all_wide(_check(oracle_mod, A, B, layouts=("NN", "TT", "NT")))


def test_wide_bf16_exponents_60_with_cancellation(oracle_mod):
    A, B, _ = wl.bf16_wide_with_cancellation(200, 130, 1000, seed=72)
    _all_wide(_check(oracle_mod, A, B, dtype="bf16", layouts=("NN", "TN")))


def test_wide_subnormals_and_zero_rows(oracle_mod):
    # magnitudes 2^U[-149, -80]: a third of them subnormal; a zero row and a
    # zero column
    A = wl.loguniform_f32((150, 300), 73, 0, lo=-149, hi=-80)
    B = wl.loguniform_f32((140, 300), 73, 1, lo=-149, hi=-80)
    A[7] = 0.0
    B[:, 11] = 0.0
    B[100] = 0.0
    routes = _check(oracle_mod, A, B)
    for r in routes:
        assert r["kulisch"] == 0 and r["wide"] > 0, r


def test_rows_the_wide_path_must_not_take(oracle_mod):
    # one row of A holds a NaN, one row of B spans 100 binades: their tiles go
    # to the general kernel, every other tile to the wide path
    A = wl.loguniform_f32((200, 500), 74, 0, lo=-30, hi=30)
    B = wl.loguniform_f32((190, 500), 74, 1, lo=-30, hi=30)
    A[70, 5] = np.nan
    B[150, 9] = np.float32(2.0 ** 60)
    B[150, 10] = np.float32(2.0 ** -40)
    routes = _check(oracle_mod, A, B)
    for r in routes:
        assert r["wide"] > 0 and r["kulisch"] > 0 and r["wide"] + r["kulisch"] == r["general"], r


def test_wide_headline_shape_sampled_rows(oracle_mod):
    A = wl.loguniform_f32((4096, 4096), 0, 0, lo=-40, hi=40)
    B = wl.loguniform_f32((4096, 4096), 0, 1, lo=-40, hi=40)
    got = bits_of(dg.det_gemm(dev_f32(A), dev_f32(B)))
    _all_wide([_native.tile_routes()])
    rows = np.array(sorted({0, 1, 127, 128, 255, 256, 2047, 2048, 2559, 2560, 2815, 2816, 4094, 4095} |
                           set(wl.rng(75, 0).integers(0, 4096, size=52).tolist())))
    assert_bits_equal(got[rows], np_bits(oracle_mod.gemm(A[rows], B)), "wide 4096^3 rows")


def test_narrow_data_takes_no_wide_tile():
    a = dev_f32(wl.normal_f32((512, 1024), 76, 0))
    b = dev_f32(wl.normal_f32((384, 1024), 76, 1))
    dg.det_gemm(a, b)
    r = _native.tile_routes()
    assert r["general"] == 0 and r["wide"] == 0 and r["kulisch"] == 0, r


def test_wide_path_switch_gives_identical_results(oracle_mod):
    # det_set_wide_path(0) sends the same tiles to the general kernel: the
    # results are the same exact sums, bit for bit
    A = wl.loguniform_f32((200, 300), 77, 0, lo=-40, hi=40)
    B = wl.loguniform_f32((150, 300), 77, 1, lo=-40, hi=40)
    a, b = dev_f32(A), dev_f32(B)
    lib = dg.library()
    on = bits_of(dg.det_gemm(a, b))
    _all_wide([_native.tile_routes()])
    assert lib.det_set_wide_path(0) == 1
    try:
        off = bits_of(dg.det_gemm(a, b))
        off_digits = dg.det_gemm_partial(a, b).cpu().numpy()
    finally:
        assert lib.det_set_wide_path(1) == 0
    assert np.array_equal(on, off)
    assert_bits_equal(off, np_bits(oracle_mod.gemm(A, B)), "wide path off")
    np.testing.assert_array_equal(off_digits, oracle_mod.gemm_digits(A, B))


def test_a_few_wide_rows_and_columns_in_narrow_data(oracle_mod):
    # N(0,1) operands with 64 rows of A and 64 rows of B spanning 80 binades:
    # only the tiles holding them are wide.  The wide GEMM computes just the
    # 256 x 256 output tiles that hold a wide tile (a device-side list), and
    # the wide norms and planes cover only the 64-row blocks such tiles hold;
    # the other outputs come from the narrow path.  Rows on both sides of the
    # wide ones are compared with the oracle, as are the wide rows themselves,
    # and partial digits alike.
    M, N, K = 1024, 768, 512
    A = wl.normal_f32((M, K), 73, 0)
    B = wl.normal_f32((N, K), 73, 1)
    A[320:384] = wl.loguniform_f32((64, K), 73, 2, lo=-40, hi=40)
    B[448:512] = wl.loguniform_f32((64, K), 73, 3, lo=-40, hi=40)
    a, b = dev_f32(A), dev_f32(B)
    got = bits_of(dg.det_gemm(a, b))
    r = _native.tile_routes()
    # the wide rows make 12 x 16 tiles wide (every tile of A's wide block and
    # of B's), and no tile is left for the general kernel
    assert r["wide"] == (N // 64) + (M // 64) - 1 and r["kulisch"] == 0, r
    rows = np.array([0, 255, 319, 320, 351, 383, 384, 511, 512, 1023])
    assert_bits_equal(got[rows], np_bits(oracle_mod.gemm(A[rows], B)), "sampled rows")
    P = dg.det_gemm_partial(a, b).cpu().numpy()
    np.testing.assert_array_equal(P[:, rows], oracle_mod.gemm_digits(A[rows], B), err_msg="digits")


@pytest.mark.parametrize("wide_rows", ["all", "upper", "lower"])
def test_wide_rows_in_a_tall_output(oracle_mod, wide_rows):
    # 2304 rows (two narrow row bands, split at row 1024): wide tiles
    # everywhere, or only in 64 rows of A in the lower or the upper part of
    # C.  Every output of the wide rows and the rows around them, and the
    # rows at the narrow band edge, equal the oracle's, and so do their
    # digits.
    M, N, K = 2304, 320, 300
    if wide_rows == "all":
        A = wl.loguniform_f32((M, K), 78, 0, lo=-40, hi=40)
        B = wl.loguniform_f32((N, K), 78, 1, lo=-40, hi=40)
        check = np.arange(M)
    else:
        A = wl.normal_f32((M, K), 79, 0)
        B = wl.normal_f32((N, K), 79, 1)
        lo = 1984 if wide_rows == "lower" else 640
        A[lo:lo + 64] = wl.loguniform_f32((64, K), 79, 2, lo=-40, hi=40)
        check = np.array(sorted(set(range(lo - 2, lo + 66)) | {0, 1023, 1024, 1025, M - 1}))
    a, b = dev_f32(A), dev_f32(B)
    got = bits_of(dg.det_gemm(a, b))
    r = _native.tile_routes()
    assert r["wide"] > 0 and r["kulisch"] == 0, r
    assert_bits_equal(got[check], np_bits(oracle_mod.gemm(A[check], B)), f"wide rows: {wide_rows}")
    edge = np.array([0, 1023, 1024, M - 1] + ([640, 700] if wide_rows == "upper" else [2000]))
    P = dg.det_gemm_partial(a, b).cpu().numpy()
    np.testing.assert_array_equal(P[:, edge], oracle_mod.gemm_digits(A[edge], B), err_msg="digits")
