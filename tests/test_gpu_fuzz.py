"""Seeded random cases against the oracle: every output and every digit.

Each case draws, from its own seed, a shape (M and N up to 700, K up to
2000, each possibly 1), a value distribution (N(0,1), log-uniform magnitudes over a
spread of 20 to 200 binades, or bf16 with exponents over +-60 and cancelling
pairs), an operand layout for each side (K-contiguous or K-minor), optionally
a padded leading dimension, and optionally zero rows, an Inf or a NaN.  The
same inputs are drawn on every run, so a failure replays.  Both det_gemm (the
rounded outputs) and det_gemm_partial (the canonical digits) must equal the
oracle's: whichever path the library takes for the case (narrow or wide
residue path, general kernel, mixed routing).
"""
import numpy as np
import pytest
import torch

import exact_sum_gemm_gb300 as dg
from exact_sum_gemm_gb300 import workloads as wl
from gpu_util import assert_bits_equal, bits_of, np_bits

pytestmark = pytest.mark.gpu

CASES = 36


def _operand(x, layout, pad, dtype):
    """A device operand [rows, K] stored K-contiguous ('N') or K-minor ('T'),
    with `pad` extra elements per stored row."""
    stored = x if layout == "N" else np.ascontiguousarray(x.T)
    if pad:
        wide = np.zeros((stored.shape[0], stored.shape[1] + pad), dtype=stored.dtype)
        wide[:, :stored.shape[1]] = stored
        dev = (torch.from_numpy(wide).cuda() if dtype == "f32" else wl.to_torch_bf16(wide, "cuda"))
        dev = dev[:, :stored.shape[1]]
    else:
        dev = (torch.from_numpy(np.ascontiguousarray(stored)).cuda() if dtype == "f32"
               else wl.to_torch_bf16(np.ascontiguousarray(stored), "cuda"))
    return dev if layout == "N" else dev.t()


def _draw(case):
    g = np.random.default_rng(1000 + case)
    M, N = (int(v) for v in g.integers(1, 700, size=2))
    K = int(g.choice([1, 3, 64, 129, 700, 1025, int(g.integers(1, 2000)), int(g.integers(1, 2000))]))
    kind = ["normal", "loguniform", "bf16"][case % 3]
    if kind == "bf16":
        A, B, _ = wl.bf16_wide_with_cancellation(M, N, K, seed=2000 + case)
        dtype = "bf16"
    elif kind == "normal":
        A = wl.normal_f32((M, K), 3000 + case, 0)
        B = wl.normal_f32((N, K), 3000 + case, 1)
        dtype = "f32"
    else:
        span = float(g.choice([10, 30, 44, 60, 100]))
        A = wl.loguniform_f32((M, K), 3000 + case, 0, lo=-span, hi=span)
        B = wl.loguniform_f32((N, K), 3000 + case, 1, lo=-span, hi=span)
        dtype = "f32"
    # planted specials (f32 only: the bf16 generator already mixes exponents)
    if dtype == "f32" and g.random() < 0.5:
        A[int(g.integers(0, M))] = 0.0
        if g.random() < 0.5:
            A[int(g.integers(0, M)), int(g.integers(0, K))] = np.float32(np.inf)
        if g.random() < 0.5:
            B[int(g.integers(0, N)), int(g.integers(0, K))] = np.float32(np.nan)
    la, lb = (str(c) for c in g.choice(["N", "T"], size=2))
    pa, pb = (int(g.choice([0, 0, 4, 7])) for _ in range(2))
    return A, B, dtype, la, lb, pa, pb


@pytest.mark.parametrize("case", range(CASES))
def test_random_case_against_the_oracle(oracle_mod, case):
    A, B, dtype, la, lb, pa, pb = _draw(case)
    a = _operand(A, la, pa, dtype)
    b = _operand(B, lb, pb, dtype)
    tag = f"case {case}: {A.shape[0]}x{B.shape[0]}x{A.shape[1]} {dtype} {la}{lb} pad {pa},{pb}"
    assert_bits_equal(bits_of(dg.det_gemm(a, b)), np_bits(oracle_mod.gemm(A, B, dtype=dtype)), tag)
    np.testing.assert_array_equal(dg.det_gemm_partial(a, b).cpu().numpy(),
                                  oracle_mod.gemm_digits(A, B, dtype=dtype), err_msg=tag)
