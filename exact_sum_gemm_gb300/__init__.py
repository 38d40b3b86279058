"""Exact-sum (Kulisch long-accumulator) GEMM for GB300, as a thin torch binding.

The call names follow the det-train page's usage section:

    y = det_gemm(a, b)                         # a [M,K], b [N,K] -> fp32 [M,N]
    lo = det_gemm_partial(a[:, :k], b[:, :k])  # int64 digit array [20,M,N]
    hi = det_gemm_partial(a[:, k:], b[:, k:])
    y2 = det_finalize(det_combine([lo, hi]))   # equal to y, bit for bit
    lin = DetLinear(1024, 512, device="cuda")

Every step runs in the sm_103a kernels of ``libdetgemm.so`` behind the C ABI of
``include/det_gemm.h``; this module only checks arguments, allocates outputs
with torch and passes pointers, strides and torch's current stream.  There is
no CPU or eager fallback: without the CUDA library every call raises.
"""
from __future__ import annotations

import ctypes

from . import _native
from ._native import (DET_BF16, DET_DIGITS, DET_F32, DET_K_MAX, DET_MAX_COMBINE, DET_PLANES,
                      DetError)

__all__ = [
    "det_gemm", "det_gemm_partial", "det_combine", "det_finalize", "det_gemm_sharded",
    "det_gemm_batched", "det_linear_forward", "det_linear_forward_bias", "det_linear_dgrad",
    "det_linear_wgrad", "det_linear_bias_grad", "DetLinear",
    "DetError", "DET_DIGITS", "DET_PLANES", "DET_K_MAX", "DET_MAX_COMBINE", "library",
    "device_status", "release_scratch", "set_scratch_retention", "scratch_stats",
]


def library():
    """The loaded C-ABI library (ctypes handle); builds it on first use."""
    return _native.lib()


def device_status(clear=False):
    """'ok', or 'timeout' if a bounded wait in one of the library's kernels ran
    out on the current device since the status was last cleared (that call's
    outputs are NaN).  Synchronises the device."""
    st = _native.lib().det_device_status(1 if clear else 0)
    if st == 9:
        return "timeout"
    _native.check("det_device_status", st)
    return "ok"


def release_scratch():
    """Synchronise the current device and return the library's unused scratch."""
    _native.check("det_release_scratch", _native.lib().det_release_scratch())


def set_scratch_retention(nbytes):
    """Bytes of freed scratch the library's pools keep reserved (default: all)."""
    _native.check("det_set_scratch_retention",
                  _native.lib().det_set_scratch_retention(int(nbytes)))


def scratch_stats():
    """(allocations so far, reserved bytes, used bytes) of the library's scratch pool."""
    return _native.scratch_stats()


def _torch():
    import torch
    return torch


def _stream(t):
    return _torch().cuda.current_stream(t.device).cuda_stream


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.float32:
        return DET_F32
    if t.dtype == torch.bfloat16:
        return DET_BF16
    raise ValueError(f"det_gemm operands must be float32 or bfloat16, got {t.dtype}")


def _operand(t, name):
    """(tensor, ld, op) for a logical [rows, K] operand with a unit stride."""
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    rows, K = t.shape
    s0, s1 = t.stride()
    if (K <= 1 or s1 == 1) and (rows <= 1 or s0 >= max(K, 1)):
        return t, (s0 if rows > 1 else max(K, 1)), 0
    if (rows <= 1 or s0 == 1) and (K <= 1 or s1 >= max(rows, 1)):
        return t, (s1 if K > 1 else max(rows, 1)), 1
    t = t.contiguous()
    return t, max(K, 1), 0


def _check_pair(x, w):
    if x.dim() != 2 or w.dim() != 2:
        raise ValueError("det_gemm takes 2-D x [M,K] and w [N,K]")
    if x.shape[1] != w.shape[1]:
        raise ValueError(f"K mismatch: x is {tuple(x.shape)}, w is {tuple(w.shape)}")
    if x.dtype != w.dtype:
        raise ValueError(f"x and w must share a dtype, got {x.dtype} and {w.dtype}")
    if x.device != w.device:
        raise ValueError("x and w must be on the same device")
    return _dtype_code(x)


def det_gemm(x, w, out=None):
    """y = RNE_f32(x @ w.T) with every product summed exactly (fp32 output)."""
    torch = _torch()
    dt = _check_pair(x, w)
    a, lda, opa = _operand(x, "x")
    b, ldb, opb = _operand(w, "w")
    M, K = x.shape
    N = w.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    elif out.shape != (M, N) or out.dtype != torch.float32 or out.stride(1) != 1:
        raise ValueError("out must be a float32 [M,N] tensor with unit column stride")
    with torch.cuda.device(x.device):
        st = _native.lib().det_gemm(dt, M, N, K, a.data_ptr(), lda, opa, b.data_ptr(), ldb, opb,
                                    out.data_ptr(), max(out.stride(0), N), _stream(x))
    _native.check("det_gemm", st)
    return out


def det_gemm_partial(x, w, out=None):
    """Unrounded exact sums of x @ w.T as a canonical int64 digit array [20, M, N]."""
    torch = _torch()
    dt = _check_pair(x, w)
    a, lda, opa = _operand(x, "x")
    b, ldb, opb = _operand(w, "w")
    M, K = x.shape
    N = w.shape[0]
    if out is None:
        out = torch.empty((DET_PLANES, M, N), dtype=torch.int64, device=x.device)
    elif out.shape != (DET_PLANES, M, N) or out.dtype != torch.int64 or not out.is_contiguous():
        raise ValueError("out must be a contiguous int64 [20,M,N] tensor")
    with torch.cuda.device(x.device):
        st = _native.lib().det_gemm_partial(dt, M, N, K, a.data_ptr(), lda, opa, b.data_ptr(), ldb,
                                            opb, out.data_ptr(), _stream(x))
    _native.check("det_gemm_partial", st)
    return out


def _check_planes(t, name):
    torch = _torch()
    if t.dim() != 3 or t.shape[0] != DET_PLANES or t.dtype != torch.int64:
        raise ValueError(f"{name} must be an int64 [20, M, N] digit array")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def det_combine(parts, out=None):
    """Sum digit arrays exactly (elementwise int64) and carry-normalise the result."""
    torch = _torch()
    parts = list(parts)
    if not parts:
        raise ValueError("det_combine needs at least one partial")
    for i, p in enumerate(parts):
        _check_planes(p, f"parts[{i}]")
        if p.shape != parts[0].shape or p.device != parts[0].device:
            raise ValueError("all partials must share shape and device")
    _, M, N = parts[0].shape
    if out is None:
        out = torch.empty_like(parts[0])
    else:
        _check_planes(out, "out")
    ptrs = (ctypes.c_void_p * len(parts))(*[p.data_ptr() for p in parts])
    with torch.cuda.device(out.device):
        st = _native.lib().det_combine(M, N, ptrs, len(parts), out.data_ptr(), _stream(out))
    _native.check("det_combine", st)
    return out


def det_finalize(acc, out=None):
    """Round a digit array [20, M, N] once to fp32 [M, N] (round to nearest even)."""
    torch = _torch()
    _check_planes(acc, "acc")
    _, M, N = acc.shape
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=acc.device)
    elif out.shape != (M, N) or out.dtype != torch.float32 or out.stride(1) != 1:
        raise ValueError("out must be a float32 [M,N] tensor with unit column stride")
    with torch.cuda.device(acc.device):
        st = _native.lib().det_finalize(M, N, acc.data_ptr(), out.data_ptr(),
                                        max(out.stride(0), N), _stream(acc))
    _native.check("det_finalize", st)
    return out


def det_gemm_sharded(x, w, cuts):
    """x @ w.T over K-shards [(k0, k1), ...]: partials, one combine, one finalize."""
    parts = [det_gemm_partial(x[:, k0:k1], w[:, k0:k1]) for k0, k1 in cuts]
    return det_finalize(det_combine(parts))


def _linear_check(t, name, shape, dtype=None):
    torch = _torch()
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}")
    return torch


def det_linear_forward(x, W):
    """y = x W^T through the C ABI's det_linear_forward (x [B,in], W [out,in])."""
    torch = _torch()
    B, d_in = x.shape
    d_out = W.shape[0]
    _linear_check(W, "W", (d_out, d_in), x.dtype)
    _linear_check(x, "x", (B, d_in))
    y = torch.empty((B, d_out), dtype=torch.float32, device=x.device)
    with torch.cuda.device(x.device):
        st = _native.lib().det_linear_forward(_dtype_code(x), B, d_in, d_out, x.data_ptr(),
                                              W.data_ptr(), y.data_ptr(), _stream(x))
    _native.check("det_linear_forward", st)
    return y


def det_linear_dgrad(dy, W):
    """dx = dy W through the C ABI (dy [B,out], W [out,in], fp32)."""
    torch = _torch()
    B, d_out = dy.shape
    d_in = W.shape[1]
    _linear_check(dy, "dy", (B, d_out), torch.float32)
    _linear_check(W, "W", (d_out, d_in), torch.float32)
    dx = torch.empty((B, d_in), dtype=torch.float32, device=dy.device)
    with torch.cuda.device(dy.device):
        st = _native.lib().det_linear_dgrad(B, d_in, d_out, dy.data_ptr(), W.data_ptr(),
                                            dx.data_ptr(), _stream(dy))
    _native.check("det_linear_dgrad", st)
    return dx


def det_linear_wgrad(dy, x):
    """dW = dy^T x through the C ABI (dy [B,out], x [B,in], fp32)."""
    torch = _torch()
    B, d_out = dy.shape
    d_in = x.shape[1]
    _linear_check(dy, "dy", (B, d_out), torch.float32)
    _linear_check(x, "x", (B, d_in), torch.float32)
    dW = torch.empty((d_out, d_in), dtype=torch.float32, device=dy.device)
    with torch.cuda.device(dy.device):
        st = _native.lib().det_linear_wgrad(B, d_in, d_out, dy.data_ptr(), x.data_ptr(),
                                            dW.data_ptr(), _stream(dy))
    _native.check("det_linear_wgrad", st)
    return dW


def det_linear_forward_bias(x, W, bias):
    """y = x W^T + bias, the bias summed exactly with the products and rounded once."""
    torch = _torch()
    B, d_in = x.shape
    d_out = W.shape[0]
    _linear_check(W, "W", (d_out, d_in), x.dtype)
    _linear_check(x, "x", (B, d_in))
    _linear_check(bias, "bias", (d_out,), x.dtype)
    y = torch.empty((B, d_out), dtype=torch.float32, device=x.device)
    with torch.cuda.device(x.device):
        st = _native.lib().det_linear_forward_bias(_dtype_code(x), B, d_in, d_out, x.data_ptr(),
                                                   W.data_ptr(), bias.data_ptr(), y.data_ptr(),
                                                   _stream(x))
    _native.check("det_linear_forward_bias", st)
    return y


def det_linear_bias_grad(dy):
    """db = column sums of dy [B, out], exact (fp32)."""
    torch = _torch()
    B, d_out = dy.shape
    _linear_check(dy, "dy", (B, d_out), torch.float32)
    db = torch.empty((d_out,), dtype=torch.float32, device=dy.device)
    with torch.cuda.device(dy.device):
        st = _native.lib().det_linear_bias_grad(B, d_out, dy.data_ptr(), db.data_ptr(), _stream(dy))
    _native.check("det_linear_bias_grad", st)
    return db


def _batch_operand(t, name, batch, K):
    """(tensor, ld, op, batch stride) for [batch, rows, K] (or a shared [rows, K])."""
    if t.dim() == 2:
        a, ld, op = _operand(t, name)
        return a, ld, op, 0
    if t.dim() != 3 or t.shape[0] != batch or t.shape[2] != K:
        raise ValueError(f"{name} must be [{batch}, rows, {K}] or [rows, {K}], got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if batch > 0:
        a, ld, op = _operand(t[0], name)
        if a.data_ptr() != t[0].data_ptr():            # unsupported inner strides: copy once
            t = t.contiguous()
            a, ld, op = _operand(t[0], name)
    else:
        ld, op = max(K, 1), 0
    return t, ld, op, t.stride(0)


def det_gemm_batched(x, w, out=None):
    """y[b] = RNE_f32(x[b] @ w[b].T) for each b; x [B,M,K], w [B,N,K] or a shared [N,K]."""
    torch = _torch()
    if x.dim() != 3:
        raise ValueError(f"x must be [batch, M, K], got {tuple(x.shape)}")
    batch, M, K = x.shape
    if w.dtype != x.dtype or w.device != x.device:
        raise ValueError("x and w must share dtype and device")
    dt = _dtype_code(x)
    a, lda, opa, sa = _batch_operand(x, "x", batch, K)
    b, ldb, opb, sb = _batch_operand(w, "w", batch, K)
    N = w.shape[-2]
    if out is None:
        out = torch.empty((batch, M, N), dtype=torch.float32, device=x.device)
    elif (out.shape != (batch, M, N) or out.dtype != torch.float32 or out.stride(2) != 1
          or (M > 1 and out.stride(1) < N)):
        raise ValueError("out must be a float32 [batch,M,N] tensor with unit column stride")
    if batch == 0 or M == 0 or N == 0:
        return out
    with torch.cuda.device(x.device):
        st = _native.lib().det_gemm_strided_batched(
            dt, batch, M, N, K, a.data_ptr(), lda, opa, sa, b.data_ptr(), ldb, opb, sb,
            out.data_ptr(), max(out.stride(1), N), out.stride(0), _stream(x))
    _native.check("det_gemm_strided_batched", st)
    return out


def __getattr__(name):
    if name == "DetLinear":
        from .linear import DetLinear
        return DetLinear
    raise AttributeError(name)
