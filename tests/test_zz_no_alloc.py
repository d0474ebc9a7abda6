"""rmsnorm_bwd_noalloc: the backward for callers that cannot allocate device
memory (a custom allocator owns all of it, a real-time loop may not allocate
after start-up, or a host runtime forbids allocator calls from libraries).

It is called through the C ABI and must give what rmsnorm_bwd gives, within
the parity tolerances of the other tests (and in fact bit for bit, since the
same kernels run with the same plan), on two calls in a row: the second call
reuses the scratch array the first one left behind. At the size limit, a
shape whose partial rows just fit in the fixed scratch runs, and one whose
partial rows just do not fit is refused before anything runs.

Kept in a file of its own that pytest collects last; it runs the same alone
in a fresh process or after the rest of the suite.
"""
from __future__ import annotations

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


CASES = [(16384, 4096, torch.bfloat16), (4096, 128, torch.bfloat16), (64, 65536, torch.bfloat16),
         (300, 2880, torch.float32), (50, 4104, torch.bfloat16)]


@pytest.mark.parametrize("M,N,dtype", CASES, ids=[f"{m}x{n}-{str(d)[6:]}" for m, n, d in CASES])
def test_matches_allocating_backward_twice(M, N, dtype):
    wl = synth.Workload(f"noalloc{M}x{N}", M, N, dtype, 1e-6, 51, 52, 53)
    inp = synth.make_inputs(wl, device=DEV)
    x, w, dy = inp["x"], inp["w"], inp["dy"]
    code = pkg.dtype_code(dtype)
    y, rstd = pkg.forward(x, w, wl.eps)
    dx_ref, dw_ref = pkg.backward(x, w, dy, rstd)
    # the allocating backward against the fp64 oracle on sampled rows and all
    # of dw, so the bit equality below ties the no-alloc results to it too
    rows = sorted({0, M - 1, *range(0, M, max(1, M // 64))})
    sel = torch.as_tensor(rows, device=DEV)
    xc, wc, dyc = x.cpu(), w.cpu(), dy.cpu()
    dx_oracle = oracle.bwd_dx(xc, wc, dyc, wl.eps, rows=rows)
    dw_oracle = oracle.bwd_dw(xc, dyc, wl.eps)
    check_rows(dx_ref[sel], dx_oracle, dtype, "rmsnorm_bwd dx")
    check_dw(dw_ref, dw_oracle, "rmsnorm_bwd dw")
    for call in range(2):
        dx = torch.full_like(x, float("nan"))
        dw = torch.full((N,), float("nan"), dtype=torch.float32, device=DEV)
        st = pkg.rmsnorm_bwd_noalloc(x, w, dy, rstd, dx, dw, M, N, code)
        assert st == pkg.OK, pkg.rmsnorm_status_string(st)
        assert pkg.rmsnorm_get_last_device_error() == pkg.OK
        check_rows(dx[sel], dx_oracle, dtype, f"dx (call {call})")
        check_dw(dw, dw_oracle, f"dw (call {call})")
        assert torch.equal(dx, dx_ref) and torch.equal(dw, dw_ref), f"call {call} differs in bits"


def bwd_need(M, N, code):
    """Workspace bytes of the plan rmsnorm_bwd_noalloc runs for 16-byte
    aligned tensors (the vector plan), on this device."""
    return pkg.rmsnorm_plan(M, N, code, pkg.PASS_BWD, 0).workspace_bytes


def full_grid_rows(N, code):
    """Rows that give the plan its full persistent grid (every partial row)."""
    p = pkg.rmsnorm_plan(1 << 22, N, code, pkg.PASS_BWD, 0)
    return p.partial_rows * (p.rows_per_unit if p.variant in (1, 2) else 1)


def widths_around_the_limit(code=pkg.F32):
    """fp32 widths whose full-grid workspace is the largest at or under the
    scratch size and the smallest over it: coarse steps, then 16-column
    steps inside the bracket."""
    limit = pkg.rmsnorm_noalloc_scratch_bytes()

    def need(n):
        return bwd_need(1 << 22, n, code)

    under = over = None
    for n in range(1024, 262145, 1024):
        if need(n) <= limit:
            under = n
        elif under is not None:
            over = n
            break
    assert under is not None and over is not None, "no width crosses the scratch size"
    best_under, best_over = under, over
    for n in range(under, over + 1, 16):
        if need(n) <= limit:
            if need(n) >= need(best_under):
                best_under = n
        elif need(n) < need(best_over):
            best_over = n
    return best_under, best_over


def test_scratch_limit_from_both_sides():
    """A shape whose partial rows just fit runs and matches rmsnorm_bwd bit
    for bit (twice); one whose partial rows just do not fit is refused before
    anything is launched."""
    limit = pkg.rmsnorm_noalloc_scratch_bytes()
    n_under, n_over = widths_around_the_limit()
    for N, fits in ((n_under, True), (n_over, False)):
        M = full_grid_rows(N, pkg.F32)
        need = bwd_need(M, N, pkg.F32)
        assert (need <= limit) == fits, (N, M, need, limit)
        wl = synth.Workload(f"limit{M}x{N}", M, N, torch.float32, 1e-6, 81, 82, 83)
        inp = synth.make_inputs(wl, device=DEV)
        x, w, dy = inp["x"], inp["w"], inp["dy"]
        y, rstd = pkg.forward(x, w, wl.eps)
        dx = torch.full_like(x, 7.0)
        dw = torch.full((N,), 3.0, dtype=torch.float32, device=DEV)
        if fits:
            dx_ref, dw_ref = pkg.backward(x, w, dy, rstd)
            for call in range(2):
                st = pkg.rmsnorm_bwd_noalloc(x, w, dy, rstd, dx, dw, M, N, pkg.F32)
                assert st == pkg.OK, pkg.rmsnorm_status_string(st)
                assert pkg.rmsnorm_get_last_device_error() == pkg.OK
                assert torch.equal(dx, dx_ref) and torch.equal(dw, dw_ref), f"call {call}"
        else:
            st = pkg.rmsnorm_bwd_noalloc(x, w, dy, rstd, dx, dw, M, N, pkg.F32)
            assert st == pkg.ERR_UNSUPPORTED
            torch.cuda.synchronize()
            assert torch.all(dw == 3.0) and torch.all(dx == 7.0), \
                "a refused call must not launch anything"


def test_empty_and_invalid():
    dw = torch.full((8,), 5.0, device=DEV)
    assert pkg.rmsnorm_bwd_noalloc(0, 0, 0, 0, 0, dw, 0, 8, pkg.F32) == pkg.OK
    torch.cuda.synchronize()
    assert torch.all(dw == 0)
    assert pkg.rmsnorm_bwd_noalloc(0, 0, 0, 0, 0, dw, 4, 0, pkg.F32) == pkg.ERR_INVALID_ARG
    assert pkg.rmsnorm_bwd_noalloc(None, dw, dw, dw, dw, dw, 1, 8, pkg.F32) == pkg.ERR_INVALID_ARG
