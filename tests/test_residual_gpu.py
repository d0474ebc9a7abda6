"""Residual add fused into the norm, CUDA library vs fp64 oracle, through the
C ABI (rmsnorm_add_fwd / rmsnorm_add_bwd).

The stored sum h = x + res is a rounding of an exact sum into the activation
type: both sides take that decision once, to nearest even, so h must match
the oracle bit for bit. y, rstd, dx and dw use the tolerances of the plain
norm. The backward is checked with and without dres (the gradient reaching
h from its other uses) and in place (h written over the residual, dx over
dres).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from parity_util import check_dw, check_rows, check_rstd

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


TYPES = [(torch.bfloat16, None), (torch.float32, None), (torch.float16, None),
         (torch.bfloat16, torch.float32), (torch.float16, torch.float32)]
TYPE_IDS = ["bf16", "f32", "f16", "bf16_wf32", "f16_wf32"]


def inputs(M, N, dtype, w_dtype=None, seed=0):
    """x, res, w, dy, dres: x and dy from the workload recipe, the residual
    and dres drawn the same way from their own seeds."""
    wl = synth.Workload(f"r{M}x{N}", M, N, dtype, 1e-5, 400 + seed, 500 + seed, 600 + seed,
                        w_dtype=w_dtype)
    a = synth.make_inputs(wl, device=DEV)
    wl2 = synth.Workload(f"r{M}x{N}b", M, N, dtype, 1e-5, 700 + seed, 800 + seed, 900 + seed,
                         dy_scale=0.5, w_dtype=w_dtype)
    b = synth.make_inputs(wl2, device=DEV)
    return a["x"], b["x"], a["w"], a["dy"], b["dy"], wl.eps


def run_fwd(x, res, w, eps, h=None):
    M, N = x.shape
    code = pkg.dtype_code(x.dtype, w.dtype)
    h = torch.empty_like(x) if h is None else h
    y = torch.empty_like(x)
    rstd = torch.empty(M, dtype=torch.float32, device=DEV)
    pkg.check(pkg.rmsnorm_add_fwd(x, res, w, h, y, rstd, M, N, eps, code), "add_fwd")
    return h, y, rstd


def run_bwd(h, w, dy, rstd, dres, dx=None):
    M, N = h.shape
    code = pkg.dtype_code(h.dtype, w.dtype)
    dx = torch.empty_like(h) if dx is None else dx
    dw = torch.empty(N, dtype=torch.float32, device=DEV)
    pkg.check(pkg.rmsnorm_add_bwd(h, w, dy, rstd, dres, dx, dw, M, N, code), "add_bwd")
    st = pkg.rmsnorm_get_last_device_error()
    assert st == pkg.OK, pkg.rmsnorm_status_string(st)
    return dx, dw


def check_fwd(x, res, w, eps, h, y, rstd, rows=None):
    h_ref, y_ref, r_ref = oracle.add_fwd(x.cpu(), res.cpu(), w.cpu(), eps, rows=rows)
    sel = slice(None) if rows is None else torch.as_tensor(rows)
    got_h = h[sel].double().cpu().numpy()
    same = (got_h == h_ref) | (np.isnan(got_h) & np.isnan(h_ref))
    assert same.all(), f"h differs from the oracle's stored sum at {np.argwhere(~same)[:5]}"
    check_rows(y[sel], y_ref, x.dtype, "y")
    check_rstd(rstd[sel], r_ref)


def check_bwd(h, w, dy, dres, eps, dx, dw, rows=None):
    hc, wc, dyc = h.cpu(), w.cpu(), dy.cpu()
    dx_ref = oracle.add_bwd_dx(hc, wc, dyc, None if dres is None else dres.cpu(), eps, rows=rows)
    sel = slice(None) if rows is None else torch.as_tensor(rows)
    check_rows(dx[sel], dx_ref, h.dtype, "dx")
    check_dw(dw, oracle.bwd_dw(hc, dyc, eps))


SHAPES = [(1, 8), (3, 13), (33, 257), (7, 32), (100, 64), (130, 128), (19, 512), (256, 1024),
          (40, 1032), (21, 1536), (5, 2048), (9, 2880), (6, 4096), (4, 8192), (3, 16384),
          (2, 65536), (1000, 40)]


@pytest.mark.parametrize("dtype,w_dtype", TYPES, ids=TYPE_IDS)
@pytest.mark.parametrize("M,N", SHAPES, ids=[f"{m}x{n}" for m, n in SHAPES])
def test_residual_shapes(M, N, dtype, w_dtype):
    x, res, w, dy, dres, eps = inputs(M, N, dtype, w_dtype)
    h, y, rstd = run_fwd(x, res, w, eps)
    check_fwd(x, res, w, eps, h, y, rstd)
    for g in (dres, None):
        dx, dw = run_bwd(h, w, dy, rstd, g)
        check_bwd(h, w, dy, g, eps, dx, dw)


@pytest.mark.parametrize("dtype,w_dtype", TYPES[:3], ids=TYPE_IDS[:3])
@pytest.mark.parametrize("N", [128, 4096, 65536])
def test_in_place(N, dtype, w_dtype):
    """h written over the residual buffer (and over x), dx over dres: the
    same results as with separate outputs."""
    M = 37
    x, res, w, dy, dres, eps = inputs(M, N, dtype, w_dtype, seed=1)
    h0, y0, r0 = run_fwd(x, res, w, eps)
    res_buf = res.clone()
    h1, y1, r1 = run_fwd(x, res_buf, w, eps, h=res_buf)
    assert h1.data_ptr() == res_buf.data_ptr()
    assert torch.equal(h1, h0) and torch.equal(y1, y0) and torch.equal(r1, r0)
    x_buf = x.clone()
    h2, y2, r2 = run_fwd(x_buf, res, w, eps, h=x_buf)
    assert torch.equal(h2, h0) and torch.equal(y2, y0) and torch.equal(r2, r0)
    dx0, dw0 = run_bwd(h0, w, dy, r0, dres)
    g_buf = dres.clone()
    dx1, dw1 = run_bwd(h0, w, dy, r0, g_buf, dx=g_buf)
    assert torch.equal(dx1, dx0) and torch.equal(dw1, dw0)


@pytest.mark.parametrize("dtype,w_dtype", TYPES, ids=TYPE_IDS)
@pytest.mark.parametrize("N", [128, 4096, 16384])
def test_rows_around_residual_grid(N, dtype, w_dtype):
    """M around the persistent grid of the backward with dres, whose kernels
    (and so resident blocks) differ from the plain backward's."""
    code = pkg.dtype_code(dtype, w_dtype)
    plan = pkg.rmsnorm_plan(1 << 20, N, code, pkg.PASS_BWD_RES, 0)
    per_unit, P = plan.rows_per_unit, plan.partial_rows
    for M in sorted({max(1, (P - 1) * per_unit), P * per_unit + 1}):
        x, res, w, dy, dres, eps = inputs(M, N, dtype, w_dtype, seed=M % 5)
        h, y, rstd = run_fwd(x, res, w, eps)
        dx, dw = run_bwd(h, w, dy, rstd, dres)
        rows = np.unique(np.concatenate([[0, M - 1], np.arange(0, M, max(1, M // 300))]))
        check_fwd(x, res, w, eps, h, y, rstd, rows=rows)
        check_bwd(h, w, dy, dres, eps, dx, dw, rows=rows)


@pytest.mark.parametrize("N,dtype", [(262144, torch.bfloat16), (131072, torch.float32)],
                         ids=["262144-bf16", "131072-f32"])
def test_residual_backward_cluster_of_16(N, dtype):
    """The residual backward over rows a cluster of 8 cannot hold: 16 blocks
    with dres as a third tensor in a two-deep ring, M around the number of
    resident clusters."""
    code = pkg.dtype_code(dtype, None)
    plan = pkg.rmsnorm_plan(1 << 20, N, code, pkg.PASS_BWD_RES, 0)
    assert pkg.VARIANTS[plan.variant] == "cluster_row" and plan.cluster in (8, 16)
    P = plan.partial_rows
    for M in sorted({max(1, P - 1), 3 * P + 2}):
        x, res, w, dy, dres, eps = inputs(M, N, dtype, None, seed=M % 5)
        h, y, rstd = run_fwd(x, res, w, eps)
        check_fwd(x, res, w, eps, h, y, rstd)
        for g in (dres, None):
            dx, dw = run_bwd(h, w, dy, rstd, g)
            check_bwd(h, w, dy, g, eps, dx, dw)


@pytest.mark.parametrize("dtype,w_dtype", TYPES, ids=TYPE_IDS)
@pytest.mark.parametrize("N", [128, 4104])
def test_residual_unaligned(N, dtype, w_dtype):
    """The residual or dres one element past a 16-byte boundary sends both
    passes to the scalar kernels."""
    M = 40
    x, res, w, dy, dres, eps = inputs(M, N, dtype, w_dtype, seed=2)
    views = {}
    for name, t in (("res", res), ("dres", dres)):
        buf = torch.empty(M * N + 1, dtype=dtype, device=DEV)
        buf[1:].copy_(t.view(-1))
        views[name] = buf[1:].view(M, N)
    h, y, rstd = run_fwd(x, views["res"], w, eps)
    check_fwd(x, views["res"], w, eps, h, y, rstd)
    dx, dw = run_bwd(h, w, dy, rstd, views["dres"])
    check_bwd(h, w, dy, views["dres"], eps, dx, dw)


@pytest.mark.parametrize("N", [128, 4096, 65536])
def test_residual_special_rows(N):
    """A NaN in the residual makes that row's h, y and dx NaN and leaves the
    other rows alone; x = -res gives a zero row (y = 0, rstd = eps^-1/2)."""
    M, dtype = 5, torch.bfloat16
    x, res, w, dy, dres, eps = inputs(M, N, dtype, seed=3)
    res = res.clone()
    res[2, N // 2] = float("nan")
    res[4] = -x[4]
    h, y, rstd = run_fwd(x, res, w, eps)
    assert torch.isnan(y[2].float()).all() and not torch.isnan(y[1].float()).any()
    assert torch.all(h[4] == 0) and torch.all(y[4] == 0)
    assert abs(rstd[4].item() - eps ** -0.5) / eps ** -0.5 < 1e-5
    keep = [0, 1, 3, 4]
    check_fwd(x, res, w, eps, h, y, rstd, rows=keep)
    dx, dw = run_bwd(h, w, dy, rstd, dres)
    assert torch.isnan(dx[2].float()).all()
    dx_ref = oracle.add_bwd_dx(h.cpu(), w.cpu(), dy.cpu(), dres.cpu(), eps, rows=keep)
    check_rows(dx[keep], dx_ref, dtype, "dx")


def test_residual_arguments():
    x = torch.zeros(4, 64, dtype=torch.bfloat16, device=DEV)
    w = torch.ones(64, dtype=torch.bfloat16, device=DEV)
    y, h = torch.empty_like(x), torch.empty_like(x)
    rstd = torch.empty(4, dtype=torch.float32, device=DEV)
    B = pkg.BF16
    assert pkg.rmsnorm_add_fwd(x, None, w, h, y, rstd, 4, 64, 1e-6, B) == pkg.ERR_INVALID_ARG
    assert pkg.rmsnorm_add_fwd(x, x, w, None, y, rstd, 4, 64, 1e-6, B) == pkg.ERR_INVALID_ARG
    assert pkg.rmsnorm_add_fwd(x, x.data_ptr() + 1, w, h, y, rstd, 4, 64, 1e-6, B) == \
        pkg.ERR_MISALIGNED
    assert pkg.rmsnorm_add_fwd(x, x, w, h, y, rstd, 0, 64, 1e-6, B) == pkg.OK
    dw = torch.full((64,), 3.0, device=DEV)
    assert pkg.rmsnorm_add_bwd(x, w, x, rstd, None, y, dw, 0, 64, B) == pkg.OK
    torch.cuda.synchronize()
    assert torch.all(dw == 0)
    assert pkg.rmsnorm_add_bwd(x, w, x, rstd, x.data_ptr() + 1, y, dw, 4, 64, B) == \
        pkg.ERR_MISALIGNED


@pytest.mark.parametrize("dtype,w_dtype", [(torch.bfloat16, None), (torch.float32, None)],
                         ids=["bf16", "f32"])
def test_residual_bitwise_repeatable(dtype, w_dtype):
    M, N = 3000, 4096
    x, res, w, dy, dres, eps = inputs(M, N, dtype, w_dtype, seed=4)
    h, y, rstd = run_fwd(x, res, w, eps)
    dx0, dw0 = run_bwd(h, w, dy, rstd, dres)
    for _ in range(4):
        dx, dw = run_bwd(h, w, dy, rstd, dres)
        assert torch.equal(dw.view(torch.int32), dw0.view(torch.int32))
        bits = torch.int32 if dtype == torch.float32 else torch.int16
        assert torch.equal(dx.view(bits), dx0.view(bits))


@pytest.mark.parametrize("wl_name", ["hidden4096_16384x4096", "qknorm_1048576x128",
                                     "sweep_f32_N16384"])
def test_residual_full_size_sampled(wl_name):
    """Full workload sizes with a residual of the same recipe: h, y, rstd and
    dx on >= 2048 sampled rows plus the first and last, and all of dw."""
    wl = synth.WORKLOADS[wl_name]
    a = synth.make_inputs(wl, device=DEV)
    import dataclasses
    b = synth.make_inputs(dataclasses.replace(wl, seed_x=wl.seed_x + 1000,
                                              seed_dy=wl.seed_dy + 1000), device=DEV)
    x, res, w, dy, dres = a["x"], b["x"], a["w"], a["dy"], b["dy"]
    h, y, rstd = run_fwd(x, res, w, wl.eps)
    dx, dw = run_bwd(h, w, dy, rstd, dres)
    M = wl.M
    rng = np.random.default_rng(54321)
    rows = np.unique(np.concatenate([[0, M - 1], rng.choice(M, size=min(M, 2048), replace=False)]))
    check_fwd(x, res, w, wl.eps, h, y, rstd, rows=rows)
    check_bwd(h, w, dy, dres, wl.eps, dx, dw, rows=rows)
