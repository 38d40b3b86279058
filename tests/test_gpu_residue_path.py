"""Parity of the tensor-core residue path against the oracle, bit for bit.

det_gemm routes tiles whose rows and columns hold few "deep" elements (more
than 18 binades below their row maximum) to the residue decomposition on the
tensor cores, and other tiles to the general Kulisch kernel.  These cases aim
at the residue path's own corners: the longest K (14 moduli, 631 exact fp32
accumulation windows reduced in TMEM), bf16 planes, deep elements handled
from the per-row lists (inside and outside the 192-bit window), non-finite
values next to deep ones, matrices whose tiles are split between the two
kernels, and the per-band moduli count at the edge of its Cauchy-Schwarz
bound.  Every expected value comes from the oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

import exact_sum_gemm_gb300 as dg
from exact_sum_gemm_gb300 import workloads as wl
from gpu_util import assert_bits_equal, bits_of, dev_bf16, dev_f32, np_bits

pytestmark = pytest.mark.gpu


def moduli_used():
    """Moduli counts (one per row band) of the last residue-path call."""
    out = (ctypes.c_int * 8)()
    n = dg.library().det_moduli_used(out, 8)
    assert n >= 0
    return list(out[:n])


def edge_rows(M, K, v, seed):
    """Rows of one element +-1 and K - 1 elements +-v, random signs.  For
    C = A A^T the diagonal outputs' exact integer dot products S equal the
    Cauchy-Schwarz bound |row|^2 from which the band's moduli count is chosen."""
    g = np.random.default_rng(seed)
    A = np.full((M, K), np.float32(v), np.float32)
    A[:, 0] = 1.0
    return A * np.where(g.random((M, K)) < 0.5, -1, 1).astype(np.float32)


@pytest.mark.parametrize("v,count", [(0.84, 12), (0.845, 13)])
def test_moduli_count_at_the_cauchy_schwarz_edge(oracle_mod, v, count):
    # K = 4096: the worst case needs 13 moduli.  |v| = 0.84 puts the diagonal
    # |S| = 2^93.497 just under the 12-moduli limit prod/(2 (1 + 2^-7)) =
    # 2^93.513; |v| = 0.845 puts it just over (2^93.514), so 13 are needed
    K = 4096
    A = edge_rows(64, K, v, 41)
    assert dg.library().det_residue_moduli(0, K) == 13
    got = bits_of(dg.det_gemm(dev_f32(A), dev_f32(A)))
    torch.cuda.synchronize()
    assert moduli_used() == [count]
    assert_bits_equal(got, np_bits(oracle_mod.gemm(A, A)), f"|x| = {v}")
    P = dg.det_gemm_partial(dev_f32(A), dev_f32(A)).cpu().numpy()
    assert moduli_used() == [count]
    np.testing.assert_array_equal(P, oracle_mod.gemm_digits(A, A))


def test_normal_data_uses_fewer_moduli_in_both_bands(oracle_mod):
    # N(0,1) at K = 4096: |S| <= |row of A| |row of B| stays below 2^93,
    # so both row bands of a 2048-row C take 12 moduli instead of 13
    K = 4096
    A = wl.normal_f32((2048, K), 47, 0)
    B = wl.normal_f32((384, K), 47, 1)
    got = bits_of(dg.det_gemm(dev_f32(A), dev_f32(B)))
    torch.cuda.synchronize()
    assert moduli_used() == [12, 12]
    rows = np.array([0, 1, 777, 1023, 1024, 1500, 2047])
    assert_bits_equal(got[rows], np_bits(oracle_mod.gemm(A[rows], B)), "N(0,1) 2048 x 384")


def test_k_limit_normal_data_takes_the_tensor_core_path(oracle_mod):
    K = 1 << 19
    A = wl.normal_f32((256, K), 13, 0)
    B = wl.normal_f32((256, K), 13, 1)
    assert dg.library().det_residue_moduli(0, K) == 14
    got = bits_of(dg.det_gemm(dev_f32(A), dev_f32(B)))
    rows, cols = np.array([0, 131, 255]), np.arange(0, 256, 5)
    want = np_bits(oracle_mod.gemm(A[rows], B[cols]))
    assert_bits_equal(got[np.ix_(rows, cols)], want, "K=2^19 N(0,1)")


def test_bf16_normal_data_takes_the_tensor_core_path(oracle_mod):
    g = np.random.default_rng(17)
    a = (g.standard_normal((300, 4096)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    b = (g.standard_normal((260, 4096)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    want = np_bits(oracle_mod.gemm(a, b, dtype="bf16"))
    assert_bits_equal(bits_of(dg.det_gemm(dev_bf16(a), dev_bf16(b))), want, "bf16 N(0,1)")
    np.testing.assert_array_equal(dg.det_gemm_partial(dev_bf16(a), dev_bf16(b)).cpu().numpy(),
                                  oracle_mod.gemm_digits(a, b, dtype="bf16"))


def test_planted_deep_elements(oracle_mod):
    g = np.random.default_rng(23)
    M, N, K = 200, 190, 3000
    A = g.standard_normal((M, K)).astype(np.float32)
    B = g.standard_normal((N, K)).astype(np.float32)
    # deep but inside the 192-bit window: ~2^-25 relative to the row max
    A[5, 100] = np.float32(3e-8)
    A[5, 2000] = np.float32(-1e-7)
    B[7, 100] = np.float32(2e-8)
    # far below the window: the digit route
    A[9, 50] = np.float32(1e-35)
    B[11, 2999] = np.float32(-3e-38)
    B[12, 17] = np.float32(1e-45)              # subnormal
    # a deep element and a non-finite one on the same row / column
    A[20, 30] = np.float32(1e-9)
    A[20, 31] = np.float32(np.inf)
    B[40, 30] = np.float32(np.nan)
    a, b = dev_f32(A), dev_f32(B)
    want = np_bits(oracle_mod.gemm(A, B))
    assert_bits_equal(bits_of(dg.det_gemm(a, b)), want, "planted deep elements")
    np.testing.assert_array_equal(dg.det_gemm_partial(a, b).cpu().numpy(), oracle_mod.gemm_digits(A, B))


def test_tiles_split_between_tensor_cores_and_general_kernel(oracle_mod):
    g = np.random.default_rng(29)
    M, N, K = 300, 280, 1024
    A = g.standard_normal((M, K)).astype(np.float32)
    B = g.standard_normal((N, K)).astype(np.float32)
    # rows 64..127 of A and columns 128..191 of C get wide exponents: those
    # tiles go to the general kernel, the rest to the residue path
    A[64:128] = wl.loguniform_f32((64, K), 29, 0, lo=-60, hi=60)
    B[128:192] = wl.loguniform_f32((64, K), 29, 1, lo=-60, hi=60)
    want = np_bits(oracle_mod.gemm(A, B))
    assert_bits_equal(bits_of(dg.det_gemm(dev_f32(A), dev_f32(B))), want, "mixed routing")


def test_transposed_operands_on_tensor_core_path(oracle_mod):
    # the DetLinear dgrad / wgrad layouts with narrow exponents
    A = wl.normal_f32((192, 700), 31, 0)
    B = wl.normal_f32((320, 700), 31, 1)
    want = np_bits(oracle_mod.gemm(A, B))
    at = dev_f32(np.ascontiguousarray(A.T)).t()
    bt = dev_f32(np.ascontiguousarray(B.T)).t()
    assert_bits_equal(bits_of(dg.det_gemm(at, bt)), want, "TT on residue path")


def test_all_zero_rows_and_exact_cancellation(oracle_mod):
    g = np.random.default_rng(37)
    A = g.standard_normal((130, 512)).astype(np.float32)
    B = g.standard_normal((140, 512)).astype(np.float32)
    A[3] = 0.0
    B[:, 256:] = B[:, :256]
    A[:, 256:] = -A[:, :256]                   # every output cancels to exactly +0
    got = bits_of(dg.det_gemm(dev_f32(A), dev_f32(B)))
    assert np.all(got == 0)
    assert_bits_equal(got, np_bits(oracle_mod.gemm(A, B)), "cancellation")


def test_many_deep_columns_and_rows(oracle_mod):
    # 100 columns of C and 40 rows of A with one deep element each: more deep
    # columns than the reconstruction buffers (64 here), so some deep-column
    # outputs take the buffered shallow sum and the rest re-read residues
    g = np.random.default_rng(41)
    M, N, K = 130, 300, 1000
    A = g.standard_normal((M, K)).astype(np.float32)
    B = g.standard_normal((N, K)).astype(np.float32)
    for i, n in enumerate(range(0, N, 3)):
        B[n, (7 * i) % K] = np.float32(3e-9) * (1 if i % 2 else -1)
    for i, m in enumerate(range(0, M, 3)[:40]):
        A[m, (11 * i + 5) % K] = np.float32(-2e-9)
    A[4, 9] = np.float32(1e-40)                  # far below the window: digit route
    want = np_bits(oracle_mod.gemm(A, B))
    a, b = dev_f32(A), dev_f32(B)
    assert_bits_equal(bits_of(dg.det_gemm(a, b)), want, "many deep rows and columns")
    np.testing.assert_array_equal(dg.det_gemm_partial(a, b).cpu().numpy(), oracle_mod.gemm_digits(A, B))


@pytest.mark.parametrize("N", [400, 512])
def test_partial_row_segments_with_deep_and_general_outputs(oracle_mod, N):
    # N a multiple of 16: det_gemm_partial writes row segments of 128 columns
    # by bulk copies.  Deep columns inside a segment get placeholders that the
    # deep kernel rewrites after it, deep rows are left to the deep kernel,
    # and a segment touching a general tile is written output by output.
    # N = 400 ends in a 16-column segment; M = 2048 makes two row bands.
    g = np.random.default_rng(43)
    M, K = 2048, 1024
    A = g.standard_normal((M, K)).astype(np.float32)
    B = g.standard_normal((N, K)).astype(np.float32)
    for i, n in enumerate(range(1, N, 37)):                 # deep columns
        B[n, (5 * i) % K] = np.float32(3e-9) * (1 if i % 2 else -1)
    for i, m in enumerate(range(2, M, 53)):                 # deep rows
        A[m, (13 * i + 1) % K] = np.float32(-2e-9)
    # general tiles: rows 64..127 of C, and columns 256..319 (half of the
    # third segment, so that segment mixes general and residue-path tiles)
    A[64:128] = wl.loguniform_f32((64, K), 43, 0, lo=-60, hi=60)
    B[256:320] = wl.loguniform_f32((64, K), 43, 1, lo=-60, hi=60)
    A[300, 10] = np.float32(np.inf)
    A[1900:1964] = wl.loguniform_f32((64, K), 44, 0, lo=-60, hi=60)   # and in the second band
    B[N - 3, 20] = np.float32(1e-40)                        # the digit route, last segment
    a, b = dev_f32(A), dev_f32(B)
    P = torch.full((20, M, N), -5, dtype=torch.int64, device="cuda")   # every plane written?
    dg.det_gemm_partial(a, b, out=P)
    np.testing.assert_array_equal(P.cpu().numpy(), oracle_mod.gemm_digits(A, B))


def test_vector_rows_with_ragged_k_tail(oracle_mod):
    # rows padded to a 16-byte multiple (the vector-load residue kernel) with
    # K = 1001, so the last run of four k crosses the end of the row
    M, N, K, ld = 70, 90, 1001, 1004
    A = wl.normal_f32((M, K), 43, 0)
    B = wl.normal_f32((N, K), 43, 1)
    A[2, 1000] = np.float32(3e-9)                # deep element in the tail
    pa = np.zeros((M, ld), np.float32)
    pb = np.zeros((N, ld), np.float32)
    pa[:, :K] = A
    pb[:, :K] = B
    pa[:, K:] = np.float32(np.nan)               # padding must never be read
    pb[:, K:] = np.float32(np.nan)
    a = dev_f32(pa)[:, :K]
    b = dev_f32(pb)[:, :K]
    want = np_bits(oracle_mod.gemm(A, B))
    assert_bits_equal(bits_of(dg.det_gemm(a, b)), want, "vector rows, ragged K")
    abf = (pa.view(np.uint32) >> 16).astype(np.uint16)     # bf16 rows: 2008-byte stride
    bbf = (pb.view(np.uint32) >> 16).astype(np.uint16)
    want16 = np_bits(oracle_mod.gemm(abf[:, :K], bbf[:, :K], dtype="bf16"))
    got16 = dg.det_gemm(dev_bf16(abf)[:, :K], dev_bf16(bbf)[:, :K])
    assert_bits_equal(bits_of(got16), want16, "bf16 vector rows, ragged K")


def test_banded_schedule_matches_single_band_calls(oracle_mod):
    # At 4096^3 f32 the rows run in two bands, each band's CUDA-core stages
    # beside the other's tensor-core GEMM.  Four 1024-row calls run the
    # one-band schedule: the two must agree on every output, and rows on both
    # sides of the band edge on the oracle.
    A = wl.normal_f32((4096, 4096), 0, 0)
    B = wl.normal_f32((4096, 4096), 0, 1)
    a, b = dev_f32(A), dev_f32(B)
    whole = bits_of(dg.det_gemm(a, b))
    parts = np.concatenate([bits_of(dg.det_gemm(a[i:i + 1024], b)) for i in range(0, 4096, 1024)])
    assert np.array_equal(whole, parts), "4096^3: banded schedule differs from single-band calls"
    rows = np.array([5, 1500, 2047, 2048, 4095])
    want = np_bits(oracle_mod.gemm(A[rows], B))
    assert_bits_equal(whole[rows], want, "4096^3 rows on both sides of the band edge")


@pytest.mark.parametrize("sa,sb", [(-120, -98), (-100, -60), (-64, -32), (-30, -2), (0, 0),
                                   (16, 48), (60, 40), (100, 30), (124, 110)])
def test_partial_digit_windows_across_scales(oracle_mod, sa, sb):
    # N(0,1) operands times 2^sa and 2^sb: the shallow sum S * 2^E lands on
    # digits (E + 298) / 32 .. + 4 with E = emaxA + emaxB - 38, so these
    # scales spread the window's first digit over 0 .. 14 (the
    # digit writer has straight-line code per start).
    A = wl.normal_f32((96, 512), 41, 0, scale_pow2=sa)
    B = wl.normal_f32((80, 512), 41, 1, scale_pow2=sb)
    a, b = dev_f32(A), dev_f32(B)
    np.testing.assert_array_equal(dg.det_gemm_partial(a, b).cpu().numpy(), oracle_mod.gemm_digits(A, B),
                                  err_msg=f"digits at 2^{sa} x 2^{sb}")
    assert_bits_equal(bits_of(dg.det_gemm(a, b)), np_bits(oracle_mod.gemm(A, B)), f"2^{sa} x 2^{sb}")


def test_fused_and_two_pass_planes_agree(oracle_mod):
    # K-contiguous operands (K <= 4096) take the fused kernel: row maxima,
    # planes, norm bounds and the band's moduli count in one launch.  The same
    # operands stored K-minor take the two-pass kernels (row maxima, plane
    # kernel, moduli kernel).  Both give the same bits and the same counts.
    K = 3000
    A = wl.normal_f32((2304, K), 53, 0)
    B = wl.normal_f32((320, K), 53, 1)
    A[7, 11] = np.float32(3e-9)                 # deep elements on both sides
    B[5, 2999] = np.float32(-2e-10)
    fused = bits_of(dg.det_gemm(dev_f32(A), dev_f32(B)))
    torch.cuda.synchronize()
    used_fused = moduli_used()
    at = dev_f32(np.ascontiguousarray(A.T)).t()      # logical [M, K], K-minor
    bt = dev_f32(np.ascontiguousarray(B.T)).t()
    two_pass = bits_of(dg.det_gemm(at, bt))
    torch.cuda.synchronize()
    assert moduli_used() == used_fused == [12, 12]
    assert_bits_equal(two_pass, fused, "K-minor operands against K-contiguous ones")
    rows = np.array([0, 7, 1279, 1280, 2303])
    assert_bits_equal(fused[rows], np_bits(oracle_mod.gemm(A[rows], B)), "fused planes")


def test_general_kernel_split_over_k(oracle_mod):
    # Wide exponents route every tile to the general kernel; with few tiles
    # (96 x 96: nine 32 x 32 tiles, some quarters of the 64 x 64 tiles outside
    # C) and a long K it splits K among CTAs and sums their digits exactly.
    # A non-finite element checks the count through the split as well.
    K = 12288
    A = wl.loguniform_f32((96, K), 59, 0, lo=-60, hi=60)
    B = wl.loguniform_f32((96, K), 59, 1, lo=-60, hi=60)
    A[5, 7000] = np.float32(np.inf)
    a, b = dev_f32(A), dev_f32(B)
    assert_bits_equal(bits_of(dg.det_gemm(a, b)), np_bits(oracle_mod.gemm(A, B)), "split K")
    np.testing.assert_array_equal(dg.det_gemm_partial(a, b).cpu().numpy(),
                                  oracle_mod.gemm_digits(A, B))
