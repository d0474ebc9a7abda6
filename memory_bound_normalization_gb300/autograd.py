"""PyTorch autograd wrappers around the C ABI, for use inside models.

``rms_norm(x, weight, eps)`` and ``fused_add_rms_norm(x, residual, weight,
eps)`` run the library's forward on the call and its backward (with the fp32
rstd saved by the forward) when autograd asks; every step of both runs in the
CUDA library. ``RMSNorm`` is the module form. The weight gradient comes back
in fp32, as the library computes it; autograd casts it to the weight's dtype
(an fp32 master weight needs no cast). Inputs must be contiguous CUDA
tensors; rows are the last dimension.
"""
from __future__ import annotations

import torch

from . import _lib
from . import dtype_code


def _rows(t: torch.Tensor):
    n = t.shape[-1]
    return (t.numel() // n if n else 0), n


class _RMSNormFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, weight, eps):
        M, N = _rows(x)
        code = dtype_code(x.dtype, weight.dtype)
        y = torch.empty_like(x)
        rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
        _lib.check(_lib.rmsnorm_fwd(x, weight, y, rstd, M, N, eps, code), "rmsnorm_fwd")
        ctx.save_for_backward(x, weight, rstd)
        return y

    @staticmethod
    def backward(ctx, dy):
        x, weight, rstd = ctx.saved_tensors
        M, N = _rows(x)
        dy = dy.contiguous()
        dx = torch.empty_like(x)
        dw = torch.empty(N, dtype=torch.float32, device=x.device)
        _lib.check(_lib.rmsnorm_bwd(x, weight, dy, rstd, dx, dw, M, N,
                                    dtype_code(x.dtype, weight.dtype)), "rmsnorm_bwd")
        return dx, dw, None


class _AddRMSNormFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, residual, weight, eps):
        M, N = _rows(x)
        code = dtype_code(x.dtype, weight.dtype)
        h = torch.empty_like(x)
        y = torch.empty_like(x)
        rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
        _lib.check(_lib.rmsnorm_add_fwd(x, residual, weight, h, y, rstd, M, N, eps, code),
                   "rmsnorm_add_fwd")
        ctx.save_for_backward(h, weight, rstd)
        return y, h

    @staticmethod
    def backward(ctx, dy, dh):
        h, weight, rstd = ctx.saved_tensors
        M, N = _rows(h)
        dy = dy.contiguous() if dy is not None else torch.zeros_like(h)
        dres = dh.contiguous() if dh is not None else None
        dx = torch.empty_like(h)
        dw = torch.empty(N, dtype=torch.float32, device=h.device)
        _lib.check(_lib.rmsnorm_add_bwd(h, weight, dy, rstd, dres, dx, dw, M, N,
                                        dtype_code(h.dtype, weight.dtype)), "rmsnorm_add_bwd")
        # h = x + residual: both receive the same gradient
        return dx, dx, dw, None


def rms_norm(x: torch.Tensor, weight: torch.Tensor, eps: float = 1e-6) -> torch.Tensor:
    """y = x * rstd * weight over the last dimension, differentiable."""
    return _RMSNormFn.apply(x.contiguous(), weight.contiguous(), float(eps))


def fused_add_rms_norm(x: torch.Tensor, residual: torch.Tensor, weight: torch.Tensor,
                       eps: float = 1e-6):
    """(y, h): h = x + residual rounded into x's dtype, y = rms_norm(h),
    differentiable in x, residual and weight (h's own gradient, from its
    later uses, flows back through the same call)."""
    return _AddRMSNormFn.apply(x.contiguous(), residual.contiguous(), weight.contiguous(),
                               float(eps))


class RMSNorm(torch.nn.Module):
    """``torch.nn.RMSNorm``-like module over the last dimension, backed by
    the CUDA library. ``weight_dtype`` lets an fp32 master weight serve 16-bit
    activations."""

    def __init__(self, dim: int, eps: float = 1e-6, device=None,
                 weight_dtype: torch.dtype = torch.float32):
        super().__init__()
        self.eps = eps
        self.weight = torch.nn.Parameter(torch.ones(dim, device=device, dtype=weight_dtype))

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        w = self.weight
        if w.dtype != x.dtype and not (w.dtype == torch.float32 and x.dtype in
                                       (torch.bfloat16, torch.float16)):
            raise TypeError(f"weight {w.dtype} cannot serve activations {x.dtype}")
        return rms_norm(x, w, self.eps)
