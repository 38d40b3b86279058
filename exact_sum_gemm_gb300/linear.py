"""DetLinear: a linear layer whose forward and backward GEMMs are exact.

det-train page, usage section: a DetLinear layer is deterministic in both the
forward and the backward pass.  Forward is y = x W^T (+ bias), dgrad dx = dy W,
wgrad dW = dy^T x, and the bias gradient db = sum of dy over rows; each is one
exact GEMM with a single rounding to fp32.  The page's layer is bias-free;
with ``bias=True`` the bias enters the forward sum as one more exact product
(1 * bias[o]) before that single rounding, so every invariance still holds.

With ``k_shards = s > 1`` every GEMM is instead computed as s K-shard
partials (``cuts`` picks the cut points, equal shards by default), one combine
and one finalize; the page's "Method" section says this gives identical
bytes, and with ``bias=True`` the bias is one more partial of K = 1.
"""
from __future__ import annotations

import torch

from . import (det_combine, det_finalize, det_gemm_partial, det_linear_bias_grad,
               det_linear_dgrad, det_linear_forward, det_linear_forward_bias, det_linear_wgrad)


def even_cuts(K, shards):
    """Cut points of `shards` K-shards of (nearly) equal size."""
    edges = [K * i // shards for i in range(shards + 1)]
    return [(edges[i], edges[i + 1]) for i in range(shards)]


def _sharded(a, b, cuts, extra=None):
    """RNE(a @ b.T [+ the sum in `extra`]) from K-shard partials, combined and finalized."""
    parts = [det_gemm_partial(a[:, k0:k1], b[:, k0:k1]) for k0, k1 in cuts]
    if extra is not None:
        parts.append(extra)
    return det_finalize(det_combine(parts))


def _bias_partial(rows, bias):
    """The digit array of the bias term: 1 * bias[o] for every row (K = 1)."""
    ones = torch.ones((rows, 1), dtype=bias.dtype, device=bias.device)
    return det_gemm_partial(ones, bias.reshape(-1, 1))


class _DetLinearFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, weight, bias, cuts_fn):
        ctx.save_for_backward(x, weight)
        ctx.cuts_fn = cuts_fn
        ctx.has_bias = bias is not None
        if cuts_fn is not None:
            extra = _bias_partial(x.shape[0], bias) if bias is not None else None
            return _sharded(x, weight, cuts_fn(x.shape[1]), extra)
        if bias is not None:
            return det_linear_forward_bias(x.contiguous(), weight.contiguous(), bias.contiguous())
        return det_linear_forward(x.contiguous(), weight.contiguous())

    @staticmethod
    def backward(ctx, dy):
        x, weight = ctx.saved_tensors
        dy = dy.contiguous().to(torch.float32)
        cuts_fn = ctx.cuts_fn
        dx = dw = db = None
        if ctx.needs_input_grad[0]:
            if x.dtype != torch.float32:
                raise ValueError("DetLinear backward needs float32 activations and weights")
            dx = (_sharded(dy, weight.t(), cuts_fn(dy.shape[1])) if cuts_fn is not None
                  else det_linear_dgrad(dy, weight.contiguous()))
        if ctx.needs_input_grad[1]:
            dw = (_sharded(dy.t(), x.t(), cuts_fn(dy.shape[0])) if cuts_fn is not None
                  else det_linear_wgrad(dy, x.contiguous()))
        if ctx.has_bias and ctx.needs_input_grad[2]:
            if cuts_fn is not None:
                ones = torch.ones((1, dy.shape[0]), dtype=torch.float32, device=dy.device)
                db = _sharded(ones, dy.t(), cuts_fn(dy.shape[0])).reshape(-1)
            else:
                db = det_linear_bias_grad(dy)
        return dx, dw, db, None


class DetLinear(torch.nn.Module):
    """y = x W^T (+ bias) with exact accumulation; W is [out_features, in_features].

    k_shards > 1 computes every GEMM as that many K-shard partials; ``cuts``
    (a function K -> [(k0, k1), ...]) overrides the equal cut points.
    """

    def __init__(self, in_features, out_features, device=None, dtype=torch.float32, k_shards=1,
                 weight=None, bias=False, cuts=None):
        super().__init__()
        self.in_features = int(in_features)
        self.out_features = int(out_features)
        self.k_shards = int(k_shards)
        if cuts is not None:
            self._cuts_fn = cuts
        elif self.k_shards > 1:
            self._cuts_fn = lambda K, s=self.k_shards: even_cuts(K, s)
        else:
            self._cuts_fn = None
        if weight is None:
            w = torch.empty(out_features, in_features, device=device, dtype=dtype)
            torch.nn.init.kaiming_uniform_(w, a=5 ** 0.5)
        else:
            w = weight.detach().to(device=device, dtype=dtype).clone()
            if tuple(w.shape) != (out_features, in_features):
                raise ValueError("weight must be [out_features, in_features]")
        self.weight = torch.nn.Parameter(w)
        if bias is True:
            bound = 1.0 / max(self.in_features, 1) ** 0.5
            b = torch.empty(out_features, device=device, dtype=dtype).uniform_(-bound, bound)
            self.bias = torch.nn.Parameter(b)
        elif bias is not False and bias is not None:
            b = bias.detach().to(device=device, dtype=dtype).clone()
            if tuple(b.shape) != (out_features,):
                raise ValueError("bias must be [out_features]")
            self.bias = torch.nn.Parameter(b)
        else:
            self.register_parameter("bias", None)

    def forward(self, x):
        if x.shape[-1] != self.in_features:
            raise ValueError(f"expected last dim {self.in_features}, got {x.shape[-1]}")
        lead = x.shape[:-1]
        y = _DetLinearFn.apply(x.reshape(-1, self.in_features), self.weight, self.bias,
                               self._cuts_fn)
        return y.reshape(*lead, self.out_features)

    def extra_repr(self):
        return f"in_features={self.in_features}, out_features={self.out_features}, " \
               f"bias={self.bias is not None}, k_shards={self.k_shards}"
