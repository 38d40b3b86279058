"""det_gemm_strided_batched as one residue-path pipeline.

Where the entries' M and N are multiples of 64 and both operands are
K-contiguous rows of at most 4096 elements, the batch runs as one problem:
the entries' rows are stacked, each output tile is computed from its own
entry's operands only, and one set of launches serves every entry.  Every
entry must equal the oracle's GEMM of its operands and the single det_gemm of
the same operands, bit for bit, whatever the entry holds (deep elements,
exponent spreads that send its tiles to the general kernel, non-finite
values, zeros) and whatever the layout (padded entry strides, a shared
operand, tiles wider than an entry, ragged K and N).
"""
import numpy as np
import pytest
import torch

import exact_sum_gemm_gb300 as dg
from exact_sum_gemm_gb300 import workloads as wl
from gpu_util import assert_bits_equal, bits_of, dev_bf16, dev_f32, np_bits

pytestmark = pytest.mark.gpu


def _launches(fn):
    lib = dg.library()
    torch.cuda.synchronize()
    n0 = lib.det_kernel_launches()
    out = fn()
    torch.cuda.synchronize()
    return out, lib.det_kernel_launches() - n0


def _per_entry(fn):
    """fn() with the batched pipeline switched off (entries one after another)."""
    lib = dg.library()
    prev = lib.det_set_batched_pipeline(0)
    try:
        return fn()
    finally:
        lib.det_set_batched_pipeline(prev)


def test_sixty_four_heads_in_one_set_of_launches(oracle_mod):
    # 64 entries of 128 x 128 x 4096 (attention-like heads), f32 N(0,1)
    batch, M, N, K = 64, 128, 128, 4096
    A = wl.normal_f32((batch, M, K), 61, 0)
    B = wl.normal_f32((batch, N, K), 61, 1)
    a, b = dev_f32(A), dev_f32(B)
    got, n_batched = _launches(lambda: dg.det_gemm_batched(a, b))
    ref, n_loop = _launches(lambda: _per_entry(lambda: dg.det_gemm_batched(a, b)))
    # one pipeline: a fixed set of launches, not one set per entry
    assert n_batched < 40 and n_loop >= 10 * batch, (n_batched, n_loop)
    assert_bits_equal(bits_of(got), bits_of(ref), "batched pipeline against entry by entry")
    want = np.stack([np_bits(oracle_mod.gemm(A[i], B[i])) for i in range(batch)])
    assert_bits_equal(bits_of(got), want, "every entry against the oracle")
    for i in (0, 31, 63):
        assert_bits_equal(bits_of(got[i]), bits_of(dg.det_gemm(a[i], b[i])), f"single call {i}")


def _mixed_entries(batch, M, N, K):
    A = wl.normal_f32((batch, M, K), 62, 0)
    B = wl.normal_f32((batch, N, K), 62, 1)
    g = np.random.default_rng(62)
    # entry 0: deep elements in a few rows of A and columns of C
    for r in g.integers(0, M, size=5):
        A[0, r, g.integers(0, K)] = np.float32(3e-9)
    for c in g.integers(0, N, size=7):
        B[0, c, g.integers(0, K)] = np.float32(-2e-9)
    # entry 1: wide exponents in rows 64..127 of A and columns 0..63 of C
    # (those tiles go to the general kernel)
    A[1, 64:128] = wl.loguniform_f32((64, K), 63, 0, lo=-60, hi=60)
    B[1, 0:64] = wl.loguniform_f32((64, K), 63, 1, lo=-60, hi=60)
    # entry 2: a non-finite element in A and one in B
    A[2, 10, 5] = np.float32(np.inf)
    B[2, N - 1, 7] = np.float32(np.nan)
    # entry 3: all zeros; entry 4: far below the window (the digit route)
    A[3] = 0.0
    A[4, 3, 11] = np.float32(1e-40)
    return A, B


def test_mixed_entries_padded_strides_and_ragged_tiles(oracle_mod):
    # M = 192: an entry's rows end inside a 256-row tile; N = 320: a ragged
    # 256-column tile; K = 700: a ragged last stage.  A's entries sit 8 rows
    # apart in a larger buffer, C's rows have a padded stride.
    batch, M, N, K = 6, 192, 320, 700
    A, B = _mixed_entries(batch, M, N, K)
    Apad = np.zeros((batch, M + 8, K), dtype=np.float32)
    Apad[:, :M] = A
    a = dev_f32(Apad)[:, :M, :]
    b = dev_f32(B)
    out_full = torch.full((batch, M, N + 16), -1.0, device="cuda")
    out = out_full[:, :, :N]
    _, n = _launches(lambda: dg.det_gemm_batched(a, b, out=out))
    assert n < 40, n
    assert torch.all(out_full[:, :, N:] == -1.0), "padding of C written"
    ref = _per_entry(lambda: dg.det_gemm_batched(a, b))
    assert_bits_equal(bits_of(out), bits_of(ref), "batched pipeline against entry by entry")
    for i in range(batch):
        assert_bits_equal(bits_of(out[i]), np_bits(oracle_mod.gemm(A[i], B[i])), f"entry {i}")


def test_bf16_shared_weight(oracle_mod):
    # bf16 entries of 64 rows with one weight [N, K] shared by all (stride 0)
    batch, M, N, K = 8, 64, 128, 512
    ab, _, _ = wl.bf16_wide_with_cancellation(batch * M, 8, K, seed=64)
    _, wb, _ = wl.bf16_wide_with_cancellation(8, N, K, seed=65)
    a_bits = ab.reshape(batch, M, K)
    x, w = dev_bf16(a_bits), dev_bf16(wb)
    got, n = _launches(lambda: dg.det_gemm_batched(x, w))
    assert n < 40, n
    for i in range(batch):
        assert_bits_equal(bits_of(got[i]), np_bits(oracle_mod.gemm(a_bits[i], wb, dtype="bf16")),
                          f"bf16 entry {i}")
    assert_bits_equal(bits_of(got), bits_of(_per_entry(lambda: dg.det_gemm_batched(x, w))),
                      "against entry by entry")


def test_two_small_entries_on_the_single_cta_kernel(oracle_mod):
    # 2 x 64 stacked rows: the band fits one 128-row tile (single-CTA kernel)
    batch, M, N, K = 2, 64, 64, 256
    A = wl.normal_f32((batch, M, K), 66, 0)
    B = wl.normal_f32((batch, N, K), 66, 1)
    got = dg.det_gemm_batched(dev_f32(A), dev_f32(B))
    for i in range(batch):
        assert_bits_equal(bits_of(got[i]), np_bits(oracle_mod.gemm(A[i], B[i])), f"entry {i}")


@pytest.mark.parametrize("batch,M,N,K", [(16, 64, 64, 512), (7, 128, 128, 1000), (5, 64, 128, 256)])
def test_entries_packed_into_shared_tiles(oracle_mod, batch, M, N, K):
    # entries smaller than a tile share it: four 64 x 64 entries per
    # 256 x 256 tile, two 128 x 128 ones (seven entries: the last tile holds
    # one), two 64 x 128 ones; only each entry's own block is an output
    A = wl.normal_f32((batch, M, K), 67, 0)
    B = wl.normal_f32((batch, N, K), 67, 1)
    A[batch - 1, 0, 3] = np.float32(2e-9)                 # a deep row in the last entry
    B[0, N - 1, 5] = np.float32(-3e-9)                    # a deep column in the first
    a, b = dev_f32(A), dev_f32(B)
    got, n = _launches(lambda: dg.det_gemm_batched(a, b))
    assert n < 40, n
    for i in range(batch):
        assert_bits_equal(bits_of(got[i]), np_bits(oracle_mod.gemm(A[i], B[i])), f"entry {i}")
    assert_bits_equal(bits_of(got), bits_of(_per_entry(lambda: dg.det_gemm_batched(a, b))),
                      "against entry by entry")


def test_many_tiny_entries_and_a_shared_left_operand(oracle_mod):
    # 1000 entries of 64 x 64 x 64: 64 000 stacked rows through the planes,
    # the routing and two bands; x is one [M, K] matrix every entry shares
    # (an expanded view: entry stride 0)
    batch, M, N, K = 1000, 64, 64, 64
    x = wl.normal_f32((M, K), 68, 0)
    W = wl.normal_f32((batch, N, K), 68, 1)
    W[999, 5, 7] = np.float32(-4e-9)                      # a deep column in the last entry
    xb = dev_f32(x).unsqueeze(0).expand(batch, M, K)
    wd = dev_f32(W)
    got, n = _launches(lambda: dg.det_gemm_batched(xb, wd))
    assert n < 40, n
    for i in (0, 1, 500, 998, 999):
        assert_bits_equal(bits_of(got[i]), np_bits(oracle_mod.gemm(x, W[i])), f"entry {i}")
    assert_bits_equal(bits_of(got), bits_of(_per_entry(lambda: dg.det_gemm_batched(xb, wd))),
                      "against entry by entry")


def test_switch_returns_the_previous_setting():
    lib = dg.library()
    assert lib.det_set_batched_pipeline(0) == 1
    assert lib.det_set_batched_pipeline(1) == 0
    assert lib.det_set_batched_pipeline(1) == 1
