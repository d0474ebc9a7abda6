"""Forward and backward captured into a CUDA graph replay bit for bit like the
eager calls, and the replayed outputs match the fp64 oracle within the
parity tolerances. Small-M shapes are launch-bound (a 256 x 1024 step moves
2.6 MB), so a caller replays the pair as one graph; the backward's workspace
comes from the stream-ordered allocator, which capture turns into graph
memory nodes. Every kernel family is covered: short rows, one block per row,
row groups, clusters (fp32 wide rows), two-pass forward, scalar (ragged N)."""
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


def check_against_oracle(x, w, dy, eps, y, rstd, dx, dw):
    """Replayed outputs against the fp64 oracle (the definition), element by
    element."""
    xc, wc, dyc = x.cpu(), w.cpu(), dy.cpu()
    y_ref, r_ref = oracle.fwd(xc, wc, eps)
    check_rows(y, y_ref, x.dtype, "replayed y")
    check_rstd(rstd, r_ref, "replayed rstd")
    check_rows(dx, oracle.bwd_dx(xc, wc, dyc, eps), x.dtype, "replayed dx")
    check_dw(dw, oracle.bwd_dw(xc, dyc, eps), "replayed dw")


F32 = torch.float32
CASES = [(1, 4096, torch.bfloat16, None), (16, 4096, torch.bfloat16, None),
         (256, 1024, torch.bfloat16, None), (300, 128, torch.bfloat16, None),
         (64, 16384, F32, None), (8, 65536, torch.bfloat16, None), (33, 257, F32, None),
         (64, 4096, torch.float16, None), (16, 8192, torch.bfloat16, F32),
         (100, 128, torch.float16, F32)]


@pytest.mark.parametrize("M,N,dtype,w_dtype", CASES,
                         ids=[f"{m}x{n}-{str(d)[6:]}" + (f"-w{str(wd)[6:]}" if wd else "")
                              for m, n, d, wd in CASES])
def test_graph_replay_matches_eager(M, N, dtype, w_dtype):
    wl = synth.Workload(f"graph{M}x{N}", M, N, dtype, 1e-6, 61, 62, 63, w_dtype=w_dtype)
    inp = synth.make_inputs(wl, device=DEV)
    x, w, dy = inp["x"], inp["w"], inp["dy"]
    code = pkg.dtype_code(dtype, w_dtype)
    y = torch.empty_like(x)
    rstd = torch.empty(M, dtype=torch.float32, device=DEV)
    dx = torch.empty_like(x)
    dw = torch.empty(N, dtype=torch.float32, device=DEV)

    def step(stream):
        pkg.check(pkg.rmsnorm_fwd(x, w, y, rstd, M, N, wl.eps, code, stream))
        pkg.check(pkg.rmsnorm_bwd(x, w, dy, rstd, dx, dw, M, N, code, stream))

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(side)  # eager: plans, device properties and attributes cached
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    ref = [t.clone() for t in (y, rstd, dx, dw)]
    for t in (y, rstd, dx, dw):
        t.fill_(float("nan"))

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(torch.cuda.current_stream())
    for _ in range(3):
        for t in (y, rstd, dx, dw):
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        for got, want in zip((y, rstd, dx, dw), ref):
            assert torch.equal(got, want)
    assert pkg.rmsnorm_get_last_device_error() == pkg.OK
    check_against_oracle(x, w, dy, wl.eps, y, rstd, dx, dw)


RES_CASES = [(1, 4096, torch.bfloat16), (256, 1024, torch.bfloat16), (300, 128, torch.float16),
             (8, 65536, torch.bfloat16)]


@pytest.mark.parametrize("M,N,dtype", RES_CASES,
                         ids=[f"{m}x{n}-{str(d)[6:]}" for m, n, d in RES_CASES])
def test_graph_replay_residual_in_place(M, N, dtype):
    """The residual pair captured with the sum written over the residual and
    dx over dres (as a serving step would) replays like the eager calls."""
    wl = synth.Workload(f"graphres{M}x{N}", M, N, dtype, 1e-6, 64, 65, 66)
    a = synth.make_inputs(wl, device=DEV)
    b = synth.make_inputs(synth.Workload("r", M, N, dtype, 1e-6, 67, 68, 69), device=DEV)
    x, w, dy = a["x"], a["w"], a["dy"]
    res0, dres0 = b["x"].clone(), b["dy"].clone()
    code = pkg.dtype_code(dtype)
    res, dres = torch.empty_like(res0), torch.empty_like(dres0)
    y = torch.empty_like(x)
    rstd = torch.empty(M, dtype=torch.float32, device=DEV)
    dw = torch.empty(N, dtype=torch.float32, device=DEV)

    def step(stream):
        res.copy_(res0)
        dres.copy_(dres0)
        pkg.check(pkg.rmsnorm_add_fwd(x, res, w, res, y, rstd, M, N, wl.eps, code, stream))
        pkg.check(pkg.rmsnorm_add_bwd(res, w, dy, rstd, dres, dres, dw, M, N, code, stream))

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    ref = [t.clone() for t in (res, y, rstd, dres, dw)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(torch.cuda.current_stream())
    for _ in range(3):
        for t in (y, rstd, dw):
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        for got, want in zip((res, y, rstd, dres, dw), ref):
            assert torch.equal(got, want)
    assert pkg.rmsnorm_get_last_device_error() == pkg.OK
    # the replayed outputs against the oracle: the stored sum bit for bit,
    # the rest within the parity tolerances
    h_ref, y_ref, r_ref = oracle.add_fwd(x.cpu(), res0.cpu(), w.cpu(), wl.eps)
    assert np.array_equal(res.float().cpu().numpy().astype(np.float64), h_ref), "replayed h"
    check_rows(y, y_ref, dtype, "replayed y")
    check_rstd(rstd, r_ref, "replayed rstd")
    hc, wc, dyc = res.cpu(), w.cpu(), dy.cpu()
    check_rows(dres, oracle.add_bwd_dx(hc, wc, dyc, dres0.cpu(), wl.eps), dtype, "replayed dx")
    check_dw(dw, oracle.bwd_dw(hc, dyc, wl.eps), "replayed dw")


@pytest.mark.parametrize("M,N,dtype", [(48, 45056, torch.bfloat16), (8, 28672, F32),
                                       (40, 1000, torch.bfloat16)])
def test_first_call_inside_capture(M, N, dtype):
    """A width's first call may come inside stream capture: its plan (the
    device's cluster-shape choice included) is made there, and the replay
    matches eager calls bit for bit. The widths are used by no other test."""
    wl = synth.Workload(f"cap{M}x{N}", M, N, dtype, 1e-6, 71, 72, 73)
    inp = synth.make_inputs(wl, device=DEV)
    x, w, dy = inp["x"], inp["w"], inp["dy"]
    code = pkg.dtype_code(dtype)
    y = torch.empty_like(x)
    rstd = torch.empty(M, dtype=torch.float32, device=DEV)
    dx = torch.empty_like(x)
    dw = torch.empty(N, dtype=torch.float32, device=DEV)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        s = torch.cuda.current_stream()
        pkg.check(pkg.rmsnorm_fwd(x, w, y, rstd, M, N, wl.eps, code, s))
        pkg.check(pkg.rmsnorm_bwd(x, w, dy, rstd, dx, dw, M, N, code, s))
    graph.replay()
    torch.cuda.synchronize()
    y2, r2 = pkg.forward(x, w, wl.eps)
    dx2, dw2 = pkg.backward(x, w, dy, r2)
    torch.cuda.synchronize()
    assert torch.equal(y, y2) and torch.equal(rstd, r2)
    assert torch.equal(dx, dx2) and torch.equal(dw, dw2)
    assert pkg.rmsnorm_get_last_device_error() == pkg.OK
    check_against_oracle(x, w, dy, wl.eps, y, rstd, dx, dw)
