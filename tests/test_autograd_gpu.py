"""The autograd wrappers run the library's kernels: their outputs and
gradients equal the direct C-ABI calls bit for bit, match the fp64 oracle
within the parity tolerances, and agree with PyTorch's own rms_norm autograd
(fp32) within the bf16 rule."""
from __future__ import annotations

import pytest
import torch
import torch.nn.functional as F

import oracle
from parity_util import check_dw, check_rows

pytestmark = pytest.mark.gpu

pkg = pytest.importorskip("memory_bound_normalization_gb300")
from memory_bound_normalization_gb300 import synth  # noqa: E402

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.set_device(0)
    pkg.load_library(build_if_missing=True)
    oracle.build()
    yield


def _inputs(M, N, dtype, w_dtype=None, seed=0):
    wl = synth.Workload("ag", M, N, dtype, 1e-6, 81 + seed, 82 + seed, 83 + seed, w_dtype=w_dtype)
    return synth.make_inputs(wl, device=DEV)


def _close_bf16(got, ref):
    err = (got.float() - ref.float()).abs()
    assert (err <= 1e-2 * ref.float().abs() + 1e-3).all(), err.max()


@pytest.mark.parametrize("shape,dtype,w_dtype", [((4, 64, 4096), torch.bfloat16, None),
                                                 ((300, 128), torch.bfloat16, torch.float32),
                                                 ((7, 2880), torch.float32, None)])
def test_rms_norm_autograd(shape, dtype, w_dtype):
    from memory_bound_normalization_gb300.autograd import rms_norm

    M, N = int(torch.tensor(shape[:-1]).prod()), shape[-1]
    inp = _inputs(M, N, dtype, w_dtype)
    x = inp["x"].view(*shape).requires_grad_(True)
    w = inp["w"].clone().requires_grad_(True)
    g = inp["dy"].view(*shape)
    y = rms_norm(x, w, 1e-6)
    y.backward(g)
    # the direct calls
    y2, rstd = pkg.forward(inp["x"], inp["w"], 1e-6)
    dx2, dw2 = pkg.backward(inp["x"], inp["w"], inp["dy"], rstd)
    assert torch.equal(y.detach().view(M, N), y2)
    assert torch.equal(x.grad.view(M, N), dx2)
    assert torch.equal(w.grad.float(), dw2.to(w.dtype).float())
    # the oracle
    xc, wc, dyc = inp["x"].cpu(), inp["w"].cpu(), inp["dy"].cpu()
    check_rows(y.detach().view(M, N), oracle.fwd(xc, wc, 1e-6)[0], dtype, "autograd y")
    check_rows(x.grad.view(M, N), oracle.bwd_dx(xc, wc, dyc, 1e-6), dtype, "autograd dx")
    check_dw(dw2, oracle.bwd_dw(xc, dyc, 1e-6), "autograd dw (fp32)")
    # PyTorch's own, in fp32
    x32 = inp["x"].float().requires_grad_(True)
    w32 = inp["w"].float().requires_grad_(True)
    y32 = F.rms_norm(x32, (N,), w32, 1e-6)
    y32.backward(inp["dy"].float())
    if dtype == torch.bfloat16:
        _close_bf16(y.detach().view(M, N), y32)
        _close_bf16(x.grad.view(M, N), x32.grad)
    rel = (w.grad.float() - w32.grad).norm() / w32.grad.norm()
    assert rel < 1e-2


def test_fused_add_rms_norm_autograd():
    from memory_bound_normalization_gb300.autograd import fused_add_rms_norm

    M, N = 96, 4096
    a = _inputs(M, N, torch.bfloat16, seed=1)
    b = _inputs(M, N, torch.bfloat16, seed=2)
    x = a["x"].clone().requires_grad_(True)
    res = b["x"].clone().requires_grad_(True)
    w = a["w"].clone().requires_grad_(True)
    y, h = fused_add_rms_norm(x, res, w, 1e-6)
    loss = (y.float() * a["dy"].float()).sum() + (h.float() * b["dy"].float()).sum()
    loss.backward()
    assert torch.equal(x.grad, res.grad)  # h = x + residual
    # the direct calls: dres is the gradient reaching h from its other use
    hh = torch.empty_like(a["x"])
    yy = torch.empty_like(a["x"])
    rstd = torch.empty(M, dtype=torch.float32, device=DEV)
    code = pkg.dtype_code(torch.bfloat16)
    pkg.check(pkg.rmsnorm_add_fwd(a["x"], b["x"], a["w"], hh, yy, rstd, M, N, 1e-6, code))
    assert torch.equal(h.detach(), hh) and torch.equal(y.detach(), yy)
    dx = torch.empty_like(hh)
    dw = torch.empty(N, dtype=torch.float32, device=DEV)
    pkg.check(pkg.rmsnorm_add_bwd(hh, a["w"], a["dy"], rstd, b["dy"], dx, dw, M, N, code))
    torch.cuda.synchronize()
    assert torch.equal(x.grad, dx)
    assert torch.equal(w.grad, dw.to(torch.bfloat16))


def test_module_with_fp32_master_weight():
    from memory_bound_normalization_gb300.autograd import RMSNorm

    M, N = 64, 1024
    inp = _inputs(M, N, torch.bfloat16, torch.float32, seed=3)
    mod = RMSNorm(N, eps=1e-6, device=DEV)
    with torch.no_grad():
        mod.weight.copy_(inp["w"])
    x = inp["x"].clone().requires_grad_(True)
    y = mod(x)
    y.backward(inp["dy"])
    assert mod.weight.grad.dtype == torch.float32
    y2, rstd = pkg.forward(inp["x"], inp["w"], 1e-6)
    dx2, dw2 = pkg.backward(inp["x"], inp["w"], inp["dy"], rstd)
    assert torch.equal(y.detach(), y2) and torch.equal(x.grad, dx2)
    assert torch.equal(mod.weight.grad, dw2)
