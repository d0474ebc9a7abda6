"""Fused RMSNorm forward and deterministic backward for NVIDIA GB300.

The computation lives in the CUDA library ``librmsnorm.so`` (C ABI in
``include/rmsnorm.h``); this package is its Python binding. The ``rmsnorm_*``
functions mirror the C entry points one for one. ``forward`` and ``backward``
are conveniences that allocate outputs with PyTorch (device memory only) and
raise ``RMSNormError`` on a non-OK status; ``add_forward`` and
``add_backward`` do the same for the residual add. ``autograd`` holds
differentiable wrappers (``rms_norm``, ``fused_add_rms_norm``, ``RMSNorm``).
"""
from __future__ import annotations

from ._lib import (  # noqa: F401
    BF16,
    BF16_W_F32,
    ERR_CUDA,
    ERR_DEVICE_TIMEOUT,
    ERR_INVALID_ARG,
    ERR_MISALIGNED,
    ERR_NOMEM,
    ERR_OUT_OF_BOUNDS,
    ERR_UNSUPPORTED,
    EXPORTS,
    F16,
    F16_W_F32,
    F32,
    OK,
    PASS_BWD,
    PASS_BWD_RES,
    PASS_FWD,
    PASS_FWD_ADD,
    PROBE_2R1W,
    PROBE_COPY,
    PROBE_WRITE,
    VARIANTS,
    Plan,
    RMSNormError,
    check,
    checked_variant,
    library_path,
    load_library,
    rmsnorm_add_bwd,
    rmsnorm_add_fwd,
    rmsnorm_bwd,
    rmsnorm_bwd_naive,
    rmsnorm_bwd_noalloc,
    rmsnorm_bwd_workspace_size,
    rmsnorm_bwd_ws,
    rmsnorm_fwd,
    rmsnorm_get_last_device_error,
    rmsnorm_noalloc_scratch_bytes,
    rmsnorm_plan,
    rmsnorm_probe,
    rmsnorm_set_wait_limit_ns,
    rmsnorm_status_string,
    rmsnorm_test_drop_copy,
    rmsnorm_version,
)

__version__ = "0.2.0"


def dtype_code(torch_dtype, w_dtype=None) -> int:
    """C-ABI dtype code of an activation dtype (float32, bfloat16 or float16)
    and a weight dtype (None or the same dtype, or float32 with 16-bit
    activations)."""
    import torch

    same = w_dtype is None or w_dtype == torch_dtype
    codes = {torch.float32: F32, torch.bfloat16: BF16, torch.float16: F16}
    if torch_dtype in codes and same:
        return codes[torch_dtype]
    if w_dtype == torch.float32 and torch_dtype == torch.bfloat16:
        return BF16_W_F32
    if w_dtype == torch.float32 and torch_dtype == torch.float16:
        return F16_W_F32
    raise RMSNormError(ERR_INVALID_ARG, f"unsupported dtypes x={torch_dtype} w={w_dtype}")


def forward(x, w, eps: float = 1e-6, stream=None):
    """y, rstd = RMSNorm(x) over the last dimension (x contiguous, on a GPU)."""
    import torch

    N = x.shape[-1]
    M = x.numel() // N if N else 0
    y = torch.empty_like(x)
    rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    check(rmsnorm_fwd(x, w, y, rstd, M, N, eps, dtype_code(x.dtype, w.dtype), stream),
          "rmsnorm_fwd")
    return y, rstd


def backward(x, w, dy, rstd, stream=None):
    """dx, dw = RMSNorm backward from the forward's rstd."""
    import torch

    N = x.shape[-1]
    M = x.numel() // N if N else 0
    dx = torch.empty_like(x)
    dw = torch.empty((N,), dtype=torch.float32, device=x.device)
    check(rmsnorm_bwd(x, w, dy, rstd, dx, dw, M, N, dtype_code(x.dtype, w.dtype), stream),
          "rmsnorm_bwd")
    return dx, dw


def add_forward(x, residual, w, eps: float = 1e-6, stream=None, inplace: bool = False):
    """h, y, rstd = (x + residual, RMSNorm(x + residual), rstd); with
    inplace=True the sum is written into `residual` and returned as h."""
    import torch

    N = x.shape[-1]
    M = x.numel() // N if N else 0
    h = residual if inplace else torch.empty_like(x)
    y = torch.empty_like(x)
    rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    check(rmsnorm_add_fwd(x, residual, w, h, y, rstd, M, N, eps, dtype_code(x.dtype, w.dtype),
                          stream), "rmsnorm_add_fwd")
    return h, y, rstd


def add_backward(h, w, dy, rstd, dres=None, stream=None):
    """dx, dw of the residual add + RMSNorm: dx (the gradient of x and of the
    residual) = RMSNorm's input gradient at h plus dres."""
    import torch

    N = h.shape[-1]
    M = h.numel() // N if N else 0
    dx = torch.empty_like(h)
    dw = torch.empty((N,), dtype=torch.float32, device=h.device)
    check(rmsnorm_add_bwd(h, w, dy, rstd, dres, dx, dw, M, N, dtype_code(h.dtype, w.dtype),
                          stream), "rmsnorm_add_bwd")
    return dx, dw
