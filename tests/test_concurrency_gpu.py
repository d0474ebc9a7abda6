"""Calls in flight on several streams from several host threads at once: each
backward takes its workspace from the stream-ordered pool on its own stream,
and the plan caches (the device's cluster-shape choice included) are shared.
Every thread's results equal the same calls made one after another, bit for
bit, and those results match the fp64 oracle."""
from __future__ import annotations

import threading

import pytest
import torch

import oracle
from parity_util import check_dw, check_rows, check_rstd

pytestmark = pytest.mark.gpu

pkg = pytest.importorskip("memory_bound_normalization_gb300")
from memory_bound_normalization_gb300 import synth  # noqa: E402

DEV = "cuda:0"

CASES = [(512, 4096, torch.bfloat16), (64, 40960, torch.bfloat16), (96, 24576, torch.float32),
         (2048, 128, torch.bfloat16), (33, 257, torch.float32), (40, 53248, torch.float16),
         (16, 4096, torch.bfloat16), (40, 1024, torch.bfloat16)]  # the last two: one cluster


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.set_device(0)
    pkg.load_library(build_if_missing=True)
    oracle.build()
    yield


def _step(inp, out, M, N, code, eps, stream):
    x, w, dy = inp["x"], inp["w"], inp["dy"]
    y, rstd, dx, dw = out
    pkg.check(pkg.rmsnorm_fwd(x, w, y, rstd, M, N, eps, code, stream))
    pkg.check(pkg.rmsnorm_bwd(x, w, dy, rstd, dx, dw, M, N, code, stream))


def test_threads_and_streams_match_sequential_calls():
    work = []
    for i, (M, N, dt) in enumerate(CASES):
        wl = synth.Workload(f"conc{i}", M, N, dt, 1e-6, 91 + i, 191 + i, 291 + i)
        inp = synth.make_inputs(wl, device=DEV)
        code = pkg.dtype_code(dt)
        x = inp["x"]
        ref = (torch.empty_like(x), torch.empty(M, device=DEV), torch.empty_like(x),
               torch.empty(N, device=DEV))
        _step(inp, ref, M, N, code, wl.eps, torch.cuda.current_stream())
        work.append((inp, ref, M, N, code, wl.eps))
    torch.cuda.synchronize()
    # the sequential results against the oracle (so the threads below are
    # checked against it too, through bit equality)
    for inp, (y, rstd, dx, dw), M, N, code, eps in work:
        xc, wc, dyc = inp["x"].cpu(), inp["w"].cpu(), inp["dy"].cpu()
        y_ref, r_ref = oracle.fwd(xc, wc, eps)
        check_rows(y, y_ref, inp["x"].dtype, f"{M}x{N} y")
        check_rstd(rstd, r_ref, f"{M}x{N} rstd")
        check_rows(dx, oracle.bwd_dx(xc, wc, dyc, eps), inp["x"].dtype, f"{M}x{N} dx")
        check_dw(dw, oracle.bwd_dw(xc, dyc, eps), f"{M}x{N} dw")

    errors = []

    def run(item):
        inp, ref, M, N, code, eps = item
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            x = inp["x"]
            out = (torch.empty_like(x), torch.empty(M, device=DEV), torch.empty_like(x),
                   torch.empty(N, device=DEV))
            with torch.cuda.stream(s):
                for _ in range(5):
                    for t in out:
                        t.fill_(float("nan"))
                    _step(inp, out, M, N, code, eps, s)
            s.synchronize()
            for got, want in zip(out, ref):
                if not torch.equal(got, want):
                    errors.append(f"{M}x{N}: results differ from the sequential calls")
        except Exception as e:  # reported below, on the main thread
            errors.append(f"{M}x{N}: {e!r}")

    threads = [threading.Thread(target=run, args=(item,)) for item in work]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads)
    assert not errors, errors
    assert pkg.rmsnorm_get_last_device_error() == pkg.OK
