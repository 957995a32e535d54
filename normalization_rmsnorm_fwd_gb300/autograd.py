"""PyTorch autograd for the RMSNorm forward / backward kernels.

Source: "FlashInfer normalization operator guide" 6.2 and 6.4, and the
flashinfer.norm API index entries for cake_rmsnorm and CakeRMSNormFunction:
the function keeps only three tensors for the backward -- the tensor that was
normalised (x, or h_new = bf16(x + residual) on the residual route), the
weight and the FP32 rstd per row -- and returns the weight gradient, which
the kernel accumulates in FP32, in the weight's dtype.  On the residual route
the forward also returns h_new, and the gradient of x and of the residual is
the same tensor: the normalisation gradient plus the gradient flowing
straight into h_new.

Layouts: a tensor whose rows the kernels can read in place (row-collapsible,
contiguous features, ld >= H, 4-byte aligned, even stride) is passed as is;
any other layout (an expanded gradient, a transposed view, an odd offset) is
copied to a contiguous tensor once.
"""
from __future__ import annotations

import torch

from . import binding
from .binding import rmsnorm_bwd, rmsnorm_fwd


def _readable(t: torch.Tensor) -> torch.Tensor:
    """t itself when the kernels can read its rows in place, else a
    contiguous copy."""
    try:
        rows, H, ld = binding.as_rows(t, "tensor")
    except ValueError:
        return t.contiguous()
    if (rows > 1 and (ld < H or ld % 2)) or t.data_ptr() % 4:
        # A fresh allocation (contiguous() would return a misaligned but
        # contiguous tensor unchanged).
        return t.clone(memory_format=torch.contiguous_format)
    return t


class RMSNormFunction(torch.autograd.Function):
    """y = RMSNorm(x) * (w + weight_bias), or (y, h_new) with a residual."""

    @staticmethod
    def forward(ctx, x, w, residual, eps, weight_bias):
        x = _readable(x)
        if residual is not None:
            residual = _readable(residual)
        y, rstd, h_new = rmsnorm_fwd(x, w, eps, residual=residual, weight_bias=weight_bias)
        ctx.save_for_backward(h_new if residual is not None else x, w, rstd)
        ctx.weight_bias = float(weight_bias)
        ctx.has_residual = residual is not None
        ctx.set_materialize_grads(False)
        if residual is not None:
            return y, h_new
        return y

    @staticmethod
    def backward(ctx, gy, gh=None):
        xn, w, rstd = ctx.saved_tensors
        if gy is None:
            gy = torch.zeros_like(xn)
        gy = _readable(gy)
        g_res = _readable(gh) if gh is not None else None
        dx, dw = rmsnorm_bwd(gy, xn, w, rstd.reshape(-1), weight_bias=ctx.weight_bias,
                             g_residual=g_res)
        dw = dw.to(w.dtype)
        if ctx.has_residual:
            return dx, dw, dx, None, None
        return dx, dw, None, None, None


def rmsnorm(x: torch.Tensor, w: torch.Tensor, eps: float = 1e-6, residual=None,
            weight_bias: float = 0.0):
    """Autograd-enabled RMSNorm: y (BF16, x's shape), or (y, h_new) when a
    residual is given (h_new = bf16(x + residual), the updated residual
    stream).  w is BF16 (weight_bias 1 for Gemma) or FP32 (weight_bias 1 for
    the zero-centred form)."""
    return RMSNormFunction.apply(x, w, residual, eps, weight_bias)
