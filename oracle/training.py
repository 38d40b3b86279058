"""The det-train page's training comparison, computed with the oracle.
TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``).

det-train page, usage section: a small MLP is trained for 160 steps, once
with every GEMM unsharded and once with 4-way K-sharded GEMMs; with exact
GEMMs the per-step losses and the final weights are identical bytes.  This
module runs that training loop on the CPU with every GEMM taken from the
oracle (the exact sum of the exact products, rounded once), and the few
elementwise steps in numpy float32, whose operations round to nearest-even
like the device's elementwise kernels:

    target = GEMM(relu(GEMM(x, T1)), T2)          teacher, no gradient
    h_pre  = GEMM(x, W1)        h = relu(h_pre)    forward, layer 1
    y      = GEMM(h, W2)                           forward, layer 2
    dy     = (y - target) * 2 / numel              gradient of mean((y - target)^2)
    dh     = GEMM(dy, W2^T)                        dgrad, layer 2
    dh_pre = dh where h_pre >= 0, else +0          gradient of relu (clamp at zero)
    dW2    = GEMM(dy^T, h^T)    dW1 = GEMM(dh_pre^T, x^T)   wgrad
    W     <- W - (dW * lr)                         two roundings, no fused update

GEMM(a, b)[m, n] = RNE_f32(sum_k a[m, k] b[n, k]) exactly (``oracle.gemm``).
The workload (sizes, seeds, initialisation, teacher, learning rate) is not on
the pages; it is the reading the tests and the design notes state: a
bias-free 1024 -> 4096 (ReLU) -> 1024 student, batch 256, SGD at lr 1e-2.
"""
from __future__ import annotations

import hashlib

import numpy as np

from . import gemm

F32 = np.float32


def relu(x):
    """max(x, 0) elementwise (exact)."""
    return np.maximum(x, F32(0.0)).astype(F32)


def digest(a) -> str:
    """SHA-256 (first 32 hex digits) of an array's float32 bytes in C order."""
    return hashlib.sha256(np.ascontiguousarray(a, dtype=F32).tobytes()).hexdigest()[:32]


def train_step(x, w1, w2, t1, t2, lr, nthreads=None):
    """One step; returns (new w1, new w2, dict of every GEMM's output)."""
    x = np.ascontiguousarray(x, F32)
    target = gemm(relu(gemm(x, t1, nthreads=nthreads)), t2, nthreads=nthreads)
    h_pre = gemm(x, w1, nthreads=nthreads)
    h = relu(h_pre)
    y = gemm(h, w2, nthreads=nthreads)
    scale = F32(2.0 / y.size)                       # 2 / numel, a power of two here
    dy = ((y - target).astype(F32) * scale).astype(F32)
    dh = gemm(dy, np.ascontiguousarray(w2.T), nthreads=nthreads)
    dh_pre = np.where(h_pre >= 0, dh, F32(0.0)).astype(F32)
    dw2 = gemm(np.ascontiguousarray(dy.T), np.ascontiguousarray(h.T), nthreads=nthreads)
    dw1 = gemm(np.ascontiguousarray(dh_pre.T), np.ascontiguousarray(x.T), nthreads=nthreads)
    lr = F32(lr)
    new_w1 = (w1 - (dw1 * lr).astype(F32)).astype(F32)
    new_w2 = (w2 - (dw2 * lr).astype(F32)).astype(F32)
    outs = {"target": target, "h_pre": h_pre, "y": y, "dh": dh, "dw1": dw1, "dw2": dw2}
    return new_w1, new_w2, outs
