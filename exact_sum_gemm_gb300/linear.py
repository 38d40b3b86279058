"""DetLinear: a bias-free linear layer whose forward and backward GEMMs are exact.

det-train page, usage section: a DetLinear layer is deterministic in both the
forward and the backward pass.  Forward is y = x W^T, dgrad dx = dy W, wgrad
dW = dy^T x; each is one exact GEMM with a single rounding to fp32.  With ``k_shards = s > 1`` every GEMM is
instead computed as s K-shard partials, one combine and one finalize, which the
page's "Method" section says gives identical bytes.
"""
from __future__ import annotations

import torch

from . import (det_combine, det_finalize, det_gemm_partial, det_linear_dgrad, det_linear_forward,
               det_linear_wgrad)
from .workloads import equal_cuts


def _sharded(a, b, k_shards):
    """RNE(a @ b.T) as k_shards partials over K, combined and finalized."""
    K = a.shape[1]
    parts = [det_gemm_partial(a[:, k0:k1], b[:, k0:k1]) for k0, k1 in equal_cuts(K, k_shards)]
    return det_finalize(det_combine(parts))


class _DetLinearFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, weight, k_shards):
        ctx.save_for_backward(x, weight)
        ctx.k_shards = k_shards
        if k_shards > 1:
            return _sharded(x, weight, k_shards)
        return det_linear_forward(x.contiguous(), weight.contiguous())

    @staticmethod
    def backward(ctx, dy):
        x, weight = ctx.saved_tensors
        dy = dy.contiguous().to(torch.float32)
        s = ctx.k_shards
        dx = dw = None
        if ctx.needs_input_grad[0]:
            if x.dtype != torch.float32:
                raise ValueError("DetLinear backward needs float32 activations and weights")
            dx = _sharded(dy, weight.t(), s) if s > 1 else det_linear_dgrad(dy, weight.contiguous())
        if ctx.needs_input_grad[1]:
            dw = _sharded(dy.t(), x.t(), s) if s > 1 else det_linear_wgrad(dy, x.contiguous())
        return dx, dw, None


class DetLinear(torch.nn.Module):
    """y = x W^T with exact accumulation; W is [out_features, in_features] fp32."""

    def __init__(self, in_features, out_features, device=None, dtype=torch.float32, k_shards=1,
                 weight=None):
        super().__init__()
        self.in_features = int(in_features)
        self.out_features = int(out_features)
        self.k_shards = int(k_shards)
        if weight is None:
            w = torch.empty(out_features, in_features, device=device, dtype=dtype)
            torch.nn.init.kaiming_uniform_(w, a=5 ** 0.5)
        else:
            w = weight.detach().to(device=device, dtype=dtype).clone()
            if tuple(w.shape) != (out_features, in_features):
                raise ValueError("weight must be [out_features, in_features]")
        self.weight = torch.nn.Parameter(w)

    def forward(self, x):
        if x.shape[-1] != self.in_features:
            raise ValueError(f"expected last dim {self.in_features}, got {x.shape[-1]}")
        lead = x.shape[:-1]
        y = _DetLinearFn.apply(x.reshape(-1, self.in_features), self.weight, self.k_shards)
        return y.reshape(*lead, self.out_features)

    def extra_repr(self):
        return f"in_features={self.in_features}, out_features={self.out_features}, " \
               f"k_shards={self.k_shards}"
