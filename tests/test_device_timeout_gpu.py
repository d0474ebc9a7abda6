"""Every wait on a bulk copy, in the backward and in the ring forward, is
bounded in time.

The library's failure-injection hook makes the next launch that stages rows
skip one bulk copy, so the wait for it can never complete (a flag that
nothing sets). The wait must give up after the configured limit, the kernel
must return, the device status word must read RMSNORM_ERR_DEVICE_TIMEOUT,
and the context must stay usable: the next, normal call matches the oracle.
No GPU fault is involved.
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
    pkg.load_library(build_if_missing=True)
    yield
    pkg.rmsnorm_test_drop_copy(-1)
    pkg.rmsnorm_set_wait_limit_ns(0)


CASES = [(64, 4096, torch.bfloat16), (4096, 128, torch.bfloat16), (8, 65536, torch.bfloat16),
         (32, 2880, torch.float32)]


@pytest.mark.parametrize("M,N,dtype", CASES, ids=[f"{m}x{n}-{d}".replace("torch.", "")
                                                  for m, n, d in CASES])
def test_dropped_copy_times_out_and_recovers(M, N, dtype):
    wl = synth.Workload(f"timeout{M}x{N}", M, N, dtype, 1e-5, 7, 8, 9)
    inp = synth.make_inputs(wl, device=DEV)
    x, w, dy = inp["x"], inp["w"], inp["dy"]
    y, rstd = pkg.forward(x, w, wl.eps)
    assert pkg.rmsnorm_get_last_device_error() == pkg.OK
    code = pkg.dtype_code(dtype)
    plan = pkg.rmsnorm_plan(M, N, code, pkg.PASS_BWD, 0)
    assert pkg.VARIANTS[plan.variant] != "scalar"
    dx = torch.empty_like(x)
    dw = torch.empty(N, dtype=torch.float32, device=DEV)
    pkg.rmsnorm_set_wait_limit_ns(50_000_000)  # 50 ms
    try:
        pkg.rmsnorm_test_drop_copy(0)
        assert pkg.rmsnorm_bwd(x, w, dy, rstd, dx, dw, M, N, code) == pkg.OK
        assert pkg.rmsnorm_get_last_device_error() == pkg.ERR_DEVICE_TIMEOUT
        # the status word is cleared by reading it
        assert pkg.rmsnorm_get_last_device_error() == pkg.OK
    finally:
        pkg.rmsnorm_test_drop_copy(-1)
        pkg.rmsnorm_set_wait_limit_ns(0)
    dx, dw = pkg.backward(x, w, dy, rstd)
    assert pkg.rmsnorm_get_last_device_error() == pkg.OK
    xc, wc, dyc = x.cpu(), w.cpu(), dy.cpu()
    check_rows(dx, oracle.bwd_dx(xc, wc, dyc, wl.eps), dtype, "dx")
    check_dw(dw, oracle.bwd_dw(xc, dyc, wl.eps))


FWD_CASES = [(64, 65536, torch.bfloat16), (256, 16384, torch.bfloat16), (64, 32768, torch.float32)]


@pytest.mark.parametrize("M,N,dtype", FWD_CASES, ids=[f"{m}x{n}-{d}".replace("torch.", "")
                                                      for m, n, d in FWD_CASES])
def test_dropped_copy_in_ring_forward_times_out_and_recovers(M, N, dtype):
    """The persistent ring forward (one block, or a cluster that exchanges its
    row sums) stages rows through bulk copies as well; a dropped copy must
    end in a bounded wait, a reported timeout and a usable context."""
    wl = synth.Workload(f"fwdtimeout{M}x{N}", M, N, dtype, 1e-5, 17, 18, 19)
    inp = synth.make_inputs(wl, device=DEV)
    x, w = inp["x"], inp["w"]
    code = pkg.dtype_code(dtype)
    plan = pkg.rmsnorm_plan(M, N, code, pkg.PASS_FWD, 0)
    assert pkg.VARIANTS[plan.variant] == "ring"
    y = torch.empty_like(x)
    rstd = torch.empty(M, dtype=torch.float32, device=DEV)
    assert pkg.rmsnorm_get_last_device_error() == pkg.OK
    pkg.rmsnorm_set_wait_limit_ns(50_000_000)  # 50 ms
    try:
        pkg.rmsnorm_test_drop_copy(0)
        assert pkg.rmsnorm_fwd(x, w, y, rstd, M, N, wl.eps, code) == pkg.OK
        assert pkg.rmsnorm_get_last_device_error() == pkg.ERR_DEVICE_TIMEOUT
        assert pkg.rmsnorm_get_last_device_error() == pkg.OK
    finally:
        pkg.rmsnorm_test_drop_copy(-1)
        pkg.rmsnorm_set_wait_limit_ns(0)
    y, rstd = pkg.forward(x, w, wl.eps)
    assert pkg.rmsnorm_get_last_device_error() == pkg.OK
    y_ref, r_ref = oracle.fwd(x.cpu(), w.cpu(), wl.eps)
    check_rows(y, y_ref, dtype, "y")
