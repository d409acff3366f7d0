"""Autograd wrappers over the C ABI: first-order gradients, like the
``once_differentiable`` backward of the fused-RMSNorm page (DeepSpeed PR 8645
quoted in PR 8664, "Where the kernels run").  Double backward raises.
"""
from __future__ import annotations

import torch
from torch.autograd.function import once_differentiable

from . import _lib


class _DyT(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, alpha, gamma, beta):
        ctx.save_for_backward(x, alpha, gamma)
        return _lib.dyt_fwd(x, alpha, gamma, beta).view(x.shape)

    @staticmethod
    @once_differentiable
    def backward(ctx, dy):
        x, alpha, gamma = ctx.saved_tensors
        dx, da, dg, db = _lib.dyt_bwd(x, dy, alpha, gamma, *ctx.needs_input_grad[1:4])
        return dx.view(x.shape), da, dg, db


class _LayerNorm(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, gamma, beta, eps):
        y, mean, rstd = _lib.layernorm_fwd(x, gamma, beta, eps)
        ctx.save_for_backward(x, gamma, mean, rstd)
        ctx.param_dtype = (gamma if gamma is not None else beta).dtype if (
            gamma is not None or beta is not None) else torch.float32
        return y.view(x.shape)

    @staticmethod
    @once_differentiable
    def backward(ctx, dy):
        x, gamma, mean, rstd = ctx.saved_tensors
        dx, dg, db = _lib.layernorm_bwd(x, dy, mean, rstd, gamma, ctx.needs_input_grad[1],
                                        ctx.needs_input_grad[2], ctx.param_dtype)
        return dx.view(x.shape), dg, db, None


class _RMSNorm(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, w, eps, variant):
        y, rstd = _lib.rmsnorm_fwd(x, w, eps, variant=variant)
        ctx.save_for_backward(x, w, rstd)
        ctx.eps, ctx.variant = eps, variant
        return y.view(x.shape)

    @staticmethod
    @once_differentiable
    def backward(ctx, dy):
        x, w, rstd = ctx.saved_tensors
        dx, dw = _lib.rmsnorm_bwd(x, dy, w, rstd, ctx.eps, ctx.needs_input_grad[1],
                                  variant=ctx.variant)
        return dx.view(x.shape), dw, None, None


def dyt(x, alpha, gamma, beta):
    """Dynamic Tanh: gamma * tanh(alpha * x) + beta over the last dimension."""
    return _DyT.apply(x, alpha, gamma, beta)


def layer_norm(x, gamma=None, beta=None, eps=1e-5):
    """LayerNorm over the last dimension (biased variance)."""
    return _LayerNorm.apply(x, gamma, beta, eps)


def rms_norm(x, weight, eps=1e-6, variant=_lib.GBN_RMS_CAST_FIRST):
    """RMSNorm over the last dimension.  variant 0 (default) is the Llama
    expression weight * (x.float() * rsqrt(mean(x^2) + eps)).to(x.dtype);
    1 multiplies by the weight before the cast; 2 is Gemma's (1 + weight)
    before the cast."""
    return _RMSNorm.apply(x, weight, eps, variant)
