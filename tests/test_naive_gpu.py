"""The naive three-kernel backward (rmsnorm_bwd_naive, kept as an ablation)
against the fp64 oracle, through the C ABI.

dx follows the tolerances of the plain backward. dw is looser by
construction: every contribution dy*x*rstd is rounded into the activation
type before the fp32 column sums, so column j can be off by up to one
rounding of each term. The bound used is
    |dw_j - ref_j| <= (2u + 1e-4) * sum_i |dy_ij * x_ij * r_i| + M * s
with u the unit roundoff of the activation type (2^-9 bf16, 2^-11 fp16,
2^-24 fp32; doubled for the fp32 result each contribution starts from),
1e-4 for the fp32 sums of up to M/64 terms, and s half the smallest
subnormal spacing (fp16 contributions can be subnormal).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

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


TYPES = [(torch.bfloat16, None), (torch.float32, None), (torch.float16, None),
         (torch.bfloat16, torch.float32), (torch.float16, torch.float32)]
TYPE_IDS = ["bf16", "f32", "f16", "bf16_wf32", "f16_wf32"]
UNIT = {torch.bfloat16: 2.0 ** -9, torch.float16: 2.0 ** -11, torch.float32: 2.0 ** -24}
SUBNORMAL_HALF = {torch.bfloat16: 2.0 ** -134, torch.float16: 2.0 ** -25, torch.float32: 2.0 ** -150}


def run_naive(x, w, dy, eps):
    M, N = x.shape
    dx = torch.empty_like(x)
    dw = torch.empty(N, dtype=torch.float32, device=DEV)
    st = pkg.rmsnorm_bwd_naive(x, w, dy, dx, dw, M, N, eps, pkg.dtype_code(x.dtype, w.dtype))
    pkg.check(st, "bwd_naive")
    torch.cuda.synchronize()
    return dx, dw


def check_naive_dw(x, dy, eps, dw):
    xc, dyc = x.cpu(), dy.cpu()
    ref = oracle.bwd_dw(xc, dyc, eps)
    if x.dtype == torch.float32:
        check_dw(dw, ref)
        return
    _, r = oracle.fwd(xc, torch.ones(x.shape[1], dtype=torch.float64), eps)
    mag = np.sum(np.abs(dyc.double().numpy() * xc.double().numpy() * r[:, None]), axis=0)
    bound = (2 * UNIT[x.dtype] + 1e-4) * mag + x.shape[0] * SUBNORMAL_HALF[x.dtype]
    err = np.abs(dw.cpu().double().numpy() - ref)
    assert (err <= bound).all(), f"dw: worst err/bound {np.max(err / np.maximum(bound, 1e-300)):.3g}"


SHAPES = [(1, 8), (3, 16), (33, 256), (100, 64), (257, 1024), (64, 2880), (17, 4096),
          (9, 8192), (1000, 40)]


@pytest.mark.parametrize("dtype,w_dtype", TYPES, ids=TYPE_IDS)
@pytest.mark.parametrize("M,N", SHAPES, ids=[f"{m}x{n}" for m, n in SHAPES])
def test_naive_shapes(M, N, dtype, w_dtype):
    if dtype == torch.float32 and N > 4096:
        pytest.skip("fp32 rows over 4096 exceed one block of 1024 vectors")
    wl = synth.Workload(f"n{M}x{N}", M, N, dtype, 1e-5, 31 + M, 32 + M, 33 + M, w_dtype=w_dtype)
    inp = synth.make_inputs(wl, device=DEV)
    x, w, dy = inp["x"], inp["w"], inp["dy"]
    dx, dw = run_naive(x, w, dy, wl.eps)
    check_rows(dx, oracle.bwd_dx(x.cpu(), w.cpu(), dy.cpu(), wl.eps), dtype, "dx")
    check_naive_dw(x, dy, wl.eps, dw)


def test_naive_repeatable_and_limits():
    wl = synth.WORKLOADS["small_256x1024"]
    inp = synth.make_inputs(wl, device=DEV)
    x, w, dy = inp["x"], inp["w"], inp["dy"]
    dx0, dw0 = run_naive(x, w, dy, wl.eps)
    for _ in range(3):
        dx, dw = run_naive(x, w, dy, wl.eps)
        assert torch.equal(dw.view(torch.int32), dw0.view(torch.int32))
        assert torch.equal(dx.view(torch.int16), dx0.view(torch.int16))
    big = torch.zeros(2, 16384, dtype=torch.bfloat16, device=DEV)
    wb = torch.ones(16384, dtype=torch.bfloat16, device=DEV)
    out = torch.empty_like(big)
    dwb = torch.empty(16384, dtype=torch.float32, device=DEV)
    assert pkg.rmsnorm_bwd_naive(big, wb, big, out, dwb, 2, 16384, 1e-6, pkg.BF16) == \
        pkg.ERR_UNSUPPORTED


def test_naive_full_size_sampled():
    """The 16384 x 4096 bf16 workload: dx on sampled rows, all of dw."""
    wl = synth.WORKLOADS["hidden4096_16384x4096"]
    inp = synth.make_inputs(wl, device=DEV)
    x, w, dy = inp["x"], inp["w"], inp["dy"]
    dx, dw = run_naive(x, w, dy, wl.eps)
    rows = np.unique(np.concatenate([[0, wl.M - 1],
                                     np.random.default_rng(7).choice(wl.M, 1024, replace=False)]))
    check_rows(dx[torch.as_tensor(rows)], oracle.bwd_dx(x.cpu(), w.cpu(), dy.cpu(), wl.eps,
                                                        rows=rows), x.dtype, "dx")
    check_naive_dw(x, dy, wl.eps, dw)
