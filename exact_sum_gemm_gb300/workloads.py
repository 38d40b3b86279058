"""Seeded synthetic inputs for the exact-sum GEMM.

This module draws random operands and nothing else: it holds none of the
method's arithmetic, and both the oracle-based tests and the GPU path take
their inputs from here.  Every generator is numpy ``Generator(PCG64)`` seeded
from ``SeedSequence([seed, stream])``; arrays are produced on the host, so the
oracle and the kernels see identical bytes.  bf16 operands are returned as
uint16 arrays of raw bit patterns.

The workloads follow the det-train page: its usage section (a 4096->4096
DetLinear with ``y.square().mean().backward()``, K-sharded partials), its
"Requirements and limits" (K <= 2^19, bf16 and f32), and its 160-step
training comparison.  The value distributions are the ones named for each
workload below; the pages give no data set.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "rng",
    "normal_f32",
    "bf16_wide_with_cancellation",
    "loguniform_f32",
    "detlinear_inputs",
    "kshard_cuts",
    "equal_cuts",
    "mlp_init",
    "mlp_batch",
    "to_torch_bf16",
    "bf16_bits_to_f32",
]


def rng(seed: int, stream: int = 0) -> np.random.Generator:
    """Independent, reproducible stream ``stream`` of seed ``seed``."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))


def normal_f32(shape, seed: int, stream: int = 0, scale_pow2: int = 0) -> np.ndarray:
    """iid N(0,1) f32 samples, optionally times 2^scale_pow2 (an exact scaling)."""
    x = rng(seed, stream).standard_normal(shape, dtype=np.float32)
    if scale_pow2:
        x = np.ldexp(x, scale_pow2).astype(np.float32)
    return x


def bf16_wide_with_cancellation(M: int, N: int, K: int, seed: int,
                                e_lo: int = -60, e_hi: int = 60,
                                cancel_frac: float = 0.10):
    """bf16 operands sign * m * 2^e, m on the bf16 grid in [1,2), e ~ U{e_lo..e_hi}.

    A fraction ``cancel_frac`` of the K positions is paired off into disjoint
    pairs (k1, k2) with A[:, k2] = -A[:, k1] and B[:, k2] = B[:, k1], so that in
    every output the two products cancel exactly.  Returns (A_bits [M,K],
    B_bits [N,K], pairs [P,2]) with A_bits/B_bits uint16 bf16 patterns.
    """
    g = rng(seed, 0)

    def draw(rows):
        sign = g.integers(0, 2, size=(rows, K), dtype=np.uint16)
        expo = g.integers(e_lo, e_hi + 1, size=(rows, K)).astype(np.int32) + 127
        frac = g.integers(0, 128, size=(rows, K), dtype=np.uint16)
        return ((sign << 15) | (expo.astype(np.uint16) << 7) | frac).astype(np.uint16)

    a = draw(M)
    b = draw(N)
    n_pos = int(round(cancel_frac * K)) // 2 * 2
    pos = g.permutation(K)[:n_pos]
    pairs = pos.reshape(-1, 2)
    a[:, pairs[:, 1]] = a[:, pairs[:, 0]] ^ np.uint16(0x8000)   # flip the sign bit
    b[:, pairs[:, 1]] = b[:, pairs[:, 0]]
    return a, b, pairs


def loguniform_f32(shape, seed: int, stream: int = 0, lo: float = -100.0,
                   hi: float = 100.0) -> np.ndarray:
    """|x| = 2^u, u ~ U[lo, hi] continuous (computed in double), random signs."""
    g = rng(seed, stream)
    u = g.uniform(lo, hi, size=shape)
    s = np.where(g.integers(0, 2, size=shape) == 1, -1.0, 1.0)
    return (s * np.exp2(u)).astype(np.float32)


def detlinear_inputs(batch: int = 2048, d_in: int = 4096, d_out: int = 4096, seed: int = 2):
    """x ~ N(0,1) [batch, d_in]; W ~ N(0,1) * 2^-6 [d_out, d_in] (std 1/64 = 1/sqrt(4096))."""
    x = normal_f32((batch, d_in), seed, 0)
    w = normal_f32((d_out, d_in), seed, 1, scale_pow2=-6)
    return x, w


def kshard_cuts(K: int, n_shards: int, seed: int, stream: int = 7) -> list:
    """Arbitrary shard boundaries: n_shards-1 cut points ~ U{0..K}, sorted.

    Duplicates are allowed, so some shards may be empty.  Returns the list of
    (k0, k1) half-open ranges covering [0, K).
    """
    cuts = np.sort(rng(seed, stream).integers(0, K + 1, size=n_shards - 1))
    edges = [0] + [int(c) for c in cuts] + [K]
    return [(edges[i], edges[i + 1]) for i in range(n_shards)]


def equal_cuts(K: int, n_shards: int) -> list:
    edges = [K * i // n_shards for i in range(n_shards + 1)]
    return [(edges[i], edges[i + 1]) for i in range(n_shards)]


def mlp_init(d_in: int = 1024, d_hidden: int = 4096, d_out: int = 1024, seed: int = 7,
             stream: int = 0):
    """Bias-free 2-layer MLP weights, N(0, 1/fan_in) with power-of-two fan_in.

    W1 [d_hidden, d_in] = N(0,1) * 2^-log2(sqrt(d_in)), W2 [d_out, d_hidden]
    likewise.  ``stream`` separates the student (0) from the teacher (1).
    """
    def pow2_std(fan_in):
        e = np.log2(fan_in) / 2
        if e != int(e):
            raise ValueError("fan_in must be an even power of two")
        return -int(e)
    w1 = normal_f32((d_hidden, d_in), seed, 100 + 2 * stream, scale_pow2=pow2_std(d_in))
    w2 = normal_f32((d_out, d_hidden), seed, 101 + 2 * stream, scale_pow2=pow2_std(d_hidden))
    return w1, w2


def mlp_batch(step: int, batch: int = 256, d_in: int = 1024, seed: int = 7) -> np.ndarray:
    """Input batch of training step ``step``: x ~ N(0,1) [batch, d_in]."""
    return normal_f32((batch, d_in), seed, 1000 + step)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bit patterns to the f32 values they denote (exact)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def to_torch_bf16(bits: np.ndarray, device=None):
    """A torch.bfloat16 tensor with the given raw bit patterns."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device) if device is not None else t
