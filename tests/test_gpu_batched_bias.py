"""Batched exact GEMM and the exact bias term of DetLinear, against the oracle.

* det_gemm_strided_batched: every batch entry equals the oracle's GEMM of its
  operands and the single det_gemm of the same operands, bit for bit.
  Covered: f32 and bf16, a shared operand (stride 0), transposed views,
  attention-like small shapes, batch 0 and K = 0.
* Bias: y = RNE_f32(x W^T + b) with b one more exact product, 1 * b[o].  The
  oracle sees exactly that sum: x widened by a column of ones, W by the bias
  column.  The bias gradient is the exact column sum of dy (oracle: a GEMM of
  a row of ones with dy^T).
"""
import numpy as np
import pytest
import torch

import exact_sum_gemm_gb300 as dg
from exact_sum_gemm_gb300 import workloads as wl
from gpu_util import assert_bits_equal, bits_of, dev_bf16, dev_f32, np_bits

pytestmark = pytest.mark.gpu


def _wide(shape, seed, stream):
    """N(0,1) with a few elements far down the exponent range (deep elements)."""
    x = wl.normal_f32(shape, seed, stream)
    g = np.random.default_rng(seed * 31 + stream)
    idx = g.integers(0, x.size, size=max(1, x.size // 500))
    x.reshape(-1)[idx] *= np.float32(2.0 ** -40)
    return x


def test_batched_f32_matches_oracle_and_single_calls(oracle_mod):
    batch, M, N, K = 5, 70, 90, 300
    A = np.stack([_wide((M, K), 3, b) for b in range(batch)])
    B = np.stack([_wide((N, K), 4, b) for b in range(batch)])
    a, b = dev_f32(A), dev_f32(B)
    got = dg.det_gemm_batched(a, b)
    for i in range(batch):
        want = np_bits(oracle_mod.gemm(A[i], B[i]))
        assert_bits_equal(bits_of(got[i]), want, f"batch entry {i}")
        assert_bits_equal(bits_of(got[i]), bits_of(dg.det_gemm(a[i], b[i])), f"single call {i}")


def test_batched_bf16_shared_weight_and_transposed_views(oracle_mod):
    batch, M, N, K = 4, 33, 65, 257
    ab, _, _ = wl.bf16_wide_with_cancellation(M * batch, 8, K, seed=9)
    _, wb, _ = wl.bf16_wide_with_cancellation(8, N, K, seed=10)
    a_bits = ab.reshape(batch, M, K)
    x = dev_bf16(a_bits)
    w = dev_bf16(wb)                                   # shared [N, K]: stride 0 across the batch
    got = dg.det_gemm_batched(x, w)
    for i in range(batch):
        want = np_bits(oracle_mod.gemm(a_bits[i], wb, dtype="bf16"))
        assert_bits_equal(bits_of(got[i]), want, f"bf16 entry {i}")
    # x stored as [batch, K, M] and read through a transposed view (op = 1)
    xt = dev_bf16(np.ascontiguousarray(a_bits.transpose(0, 2, 1))).transpose(1, 2)
    assert_bits_equal(bits_of(dg.det_gemm_batched(xt, w)), bits_of(got), "transposed view")


def test_batched_attention_like_heads(oracle_mod):
    # 16 heads of Q K^T with sequence 96 and head dimension 64
    heads, S, D = 16, 96, 64
    Q = wl.normal_f32((heads, S, D), 21, 0)
    Kt = wl.normal_f32((heads, S, D), 21, 1)
    got = dg.det_gemm_batched(dev_f32(Q), dev_f32(Kt))
    for h in (0, 7, 15):
        assert_bits_equal(bits_of(got[h]), np_bits(oracle_mod.gemm(Q[h], Kt[h])), f"head {h}")


def test_batched_degenerate():
    x = torch.zeros((0, 5, 7), device="cuda")
    w = torch.zeros((0, 3, 7), device="cuda")
    assert dg.det_gemm_batched(x, w).shape == (0, 5, 3)
    x = torch.empty((3, 5, 0), device="cuda")
    w = torch.empty((3, 4, 0), device="cuda")
    y = dg.det_gemm_batched(x, w)
    assert torch.equal(y.view(torch.int32), torch.zeros((3, 5, 4), dtype=torch.int32, device="cuda"))


def _widen(x, col):
    return np.hstack([x, col.reshape(-1, 1).astype(x.dtype)])


def test_bias_forward_is_one_more_exact_product(oracle_mod):
    M, N, K = 50, 70, 300
    x = wl.normal_f32((M, K), 5, 0)
    W = wl.normal_f32((N, K), 5, 1)
    bias = wl.normal_f32((N,), 5, 2) * np.float32(8.0)
    bias[3] = np.float32(1e-30)                        # far below the products
    bias[4] = np.float32(3e30)                         # far above them
    got = dg.det_linear_forward_bias(dev_f32(x), dev_f32(W), dev_f32(bias))
    want = oracle_mod.gemm(_widen(x, np.ones(M, np.float32)), _widen(W, bias))
    assert_bits_equal(bits_of(got), np_bits(want), "x W^T + b")


def test_bias_forward_bf16(oracle_mod):
    M, N, K = 40, 60, 200
    xb, wb, _ = wl.bf16_wide_with_cancellation(M, N, K, seed=12)
    bb = wl.bf16_wide_with_cancellation(1, N, 1, seed=13)[1].reshape(-1)
    got = dg.det_linear_forward_bias(dev_bf16(xb), dev_bf16(wb), dev_bf16(bb))
    one = np.full(M, 0x3F80, np.uint16)                # bf16 1.0
    want = oracle_mod.gemm(_widen(xb, one), _widen(wb, bb), dtype="bf16")
    assert_bits_equal(bits_of(got), np_bits(want), "bf16 x W^T + b")


def test_bias_grad_is_the_exact_column_sum(oracle_mod):
    B, N = 300, 77
    dy = wl.normal_f32((B, N), 6, 0)
    dy[:, 5] = 0.0
    dy[::2, 6] = np.float32(1e8)
    dy[1::2, 6] = np.float32(-1e8)                     # cancels exactly...
    dy[7, 6] = np.float32(1e-3)                        # ...but for this term
    got = dg.det_linear_bias_grad(dev_f32(dy))
    want = oracle_mod.gemm(np.ones((1, B), np.float32), np.ascontiguousarray(dy.T)).reshape(-1)
    assert_bits_equal(bits_of(got), np_bits(want), "db")
    assert bits_of(got)[5] == 0


def test_detlinear_bias_sharded_equals_unsharded(oracle_mod):
    M, d_in, d_out = 64, 256, 96
    x0 = wl.normal_f32((M, d_in), 8, 0)
    w0 = wl.normal_f32((d_out, d_in), 8, 1) * np.float32(2.0 ** -4)
    b0 = wl.normal_f32((d_out,), 8, 2)
    outs = []
    for shards, cuts in ((1, None), (3, lambda K: wl.kshard_cuts(K, 3, seed=K)),
                         (8, lambda K: wl.kshard_cuts(K, 8, seed=K + 1))):
        layer = dg.DetLinear(d_in, d_out, device="cuda", k_shards=shards, cuts=cuts,
                             weight=torch.from_numpy(w0), bias=torch.from_numpy(b0))
        x = dev_f32(x0).requires_grad_(True)
        y = layer(x)
        y.square().mean().backward()
        outs.append((y.detach(), x.grad, layer.weight.grad, layer.bias.grad))
    for o in outs[1:]:
        for got, want in zip(o, outs[0]):
            assert torch.equal(got.view(torch.int32), want.view(torch.int32))
    want_y = oracle_mod.gemm(_widen(x0, np.ones(M, np.float32)), _widen(w0, b0))
    assert_bits_equal(bits_of(outs[0][0]), np_bits(want_y), "DetLinear(bias) forward")
