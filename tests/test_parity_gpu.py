"""CUDA library vs fp64 oracle, element by element, through the C ABI.

Small shapes (the oracle finishes in seconds) cover every kernel family and
every dtype code (fp32, bf16, fp16, and bf16/fp16 activations with an fp32
weight) with several tiles and a ragged tail; the full workload sizes are
checked on sampled rows (every column of >= 4096 random rows plus the first
and last) and on the whole of dw, in the same launch configuration the
benchmark times.
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


def run(x, w, dy, eps):
    """fwd + bwd on the GPU through the C ABI; returns host tensors."""
    M, N = x.shape
    code = pkg.dtype_code(x.dtype, w.dtype)
    y = torch.empty_like(x)
    rstd = torch.empty(M, dtype=torch.float32, device=x.device)
    dx = torch.empty_like(x)
    dw = torch.empty(N, dtype=torch.float32, device=x.device)
    pkg.check(pkg.rmsnorm_fwd(x, w, y, rstd, M, N, eps, code), "fwd")
    pkg.check(pkg.rmsnorm_bwd(x, w, dy, rstd, dx, dw, M, N, code), "bwd")
    st = pkg.rmsnorm_get_last_device_error()
    assert st == pkg.OK, pkg.rmsnorm_status_string(st)
    return y, rstd, dx, dw


def check_all(x, w, dy, eps, y, rstd, dx, dw, rows=None):
    xc, wc, dyc = x.cpu(), w.cpu(), dy.cpu()
    y_ref, r_ref = oracle.fwd(xc, wc, eps, rows=rows)
    dx_ref = oracle.bwd_dx(xc, wc, dyc, eps, rows=rows)
    dw_ref = oracle.bwd_dw(xc, dyc, eps)
    sel = slice(None) if rows is None else torch.as_tensor(rows)
    check_rows(y[sel], y_ref, x.dtype, "y")
    check_rows(dx[sel], dx_ref, x.dtype, "dx")
    check_rstd(rstd[sel], r_ref)
    check_dw(dw, dw_ref)


def inputs(M, N, dtype, seed=0, dy_scale=1.0, w_dtype=None):
    wl = synth.Workload(f"t{M}x{N}", M, N, dtype, 1e-5, 100 + seed, 200 + seed, 300 + seed,
                        dy_scale=dy_scale, w_dtype=w_dtype)
    return synth.make_inputs(wl, device=DEV), wl.eps


# (activation dtype, weight dtype) for every dtype code
TYPES = [(torch.bfloat16, None), (torch.float32, None), (torch.float16, None),
         (torch.bfloat16, torch.float32), (torch.float16, torch.float32)]
TYPE_IDS = ["bf16", "f32", "f16", "bf16_wf32", "f16_wf32"]


SHAPES = [(1, 8), (3, 13), (33, 257), (5, 16), (7, 32), (100, 64), (130, 128), (37, 256),
          (19, 512), (256, 1024), (11, 2048), (9, 2880), (6, 4096), (3, 5120), (5, 6144),
          (2, 7168), (4, 8192),
          (3, 16384), (3, 20480), (5, 24576), (2, 32768), (3, 40960), (4, 49152), (3, 57344),
          (2, 65536), (1, 65536), (2, 98304), (3, 131072), (2, 196608), (1, 524288),
          (1000, 40), (777, 96)]


@pytest.mark.parametrize("dtype,w_dtype", TYPES, ids=TYPE_IDS)
@pytest.mark.parametrize("M,N", SHAPES, ids=[f"{m}x{n}" for m, n in SHAPES])
def test_small_shapes(M, N, dtype, w_dtype):
    inp, eps = inputs(M, N, dtype, w_dtype=w_dtype)
    out = run(inp["x"], inp["w"], inp["dy"], eps)
    check_all(inp["x"], inp["w"], inp["dy"], eps, *out)


@pytest.mark.parametrize("dtype,w_dtype", TYPES, ids=TYPE_IDS)
@pytest.mark.parametrize("N", [128, 1024, 4096, 16384])
def test_rows_around_persistent_grid(N, dtype, w_dtype):
    """M just below, at and above the persistent grid size, and a few rows
    per block, so that some blocks get one row (or tile) more than others."""
    code = pkg.dtype_code(dtype, w_dtype)
    plan = pkg.rmsnorm_plan(1 << 20, N, code, pkg.PASS_BWD, 0)
    per_unit = plan.rows_per_unit
    P = plan.partial_rows
    for M in sorted({max(1, (P - 1) * per_unit), P * per_unit, P * per_unit + 1,
                     3 * P * per_unit + per_unit // 2 + 1}):
        inp, eps = inputs(M, N, dtype, seed=M % 7, w_dtype=w_dtype)
        out = run(inp["x"], inp["w"], inp["dy"], eps)
        check_all(inp["x"], inp["w"], inp["dy"], eps, *out)


@pytest.mark.parametrize("dtype,w_dtype", TYPES, ids=TYPE_IDS)
@pytest.mark.parametrize("N", [16384, 20480, 24576, 32768, 40960, 49152, 57344, 65536, 98304,
                               131072])
def test_device_chosen_wide_shapes(N, dtype, w_dtype):
    """Wide rows take a cluster shape chosen with the occupancy API: every
    pass's plan covers the row with a legal block, cluster and ring, and
    asking again gives the same plan (so dw keeps its bits)."""
    code = pkg.dtype_code(dtype, w_dtype)
    vec = 4 if dtype == torch.float32 else 8
    for pass_ in (pkg.PASS_FWD, pkg.PASS_FWD_ADD, pkg.PASS_BWD, pkg.PASS_BWD_RES):
        p = pkg.rmsnorm_plan(1 << 20, N, code, pass_, 0)
        q = pkg.rmsnorm_plan(1 << 20, N, code, pass_, 0)
        fields = ("variant", "cluster", "threads", "vectors_per_thread", "stages", "smem_bytes",
                  "grid")
        assert all(getattr(p, f) == getattr(q, f) for f in fields)
        name = pkg.VARIANTS[p.variant]
        if name not in ("ring", "cluster_row"):
            continue
        assert p.cluster in (1, 2, 4, 5, 6, 8, 16) and 32 <= p.threads <= 512
        if p.cluster == 16:  # backward rows that 8 blocks cannot hold
            assert pass_ in (pkg.PASS_BWD, pkg.PASS_BWD_RES) and N * (16 // vec) > 256 * 1024
        assert p.threads * p.vectors_per_thread * p.cluster * vec >= N
        assert p.vectors_per_thread in (4, 8)
        if dtype != torch.float32 and p.vectors_per_thread == 8:
            # 16-bit rows: 8 vectors a thread (the slice re-read from its
            # stage) only in the forward ring, in one block for 2048-3072
            # vectors a row and past 8192 vectors
            nvec = N // 8
            assert name == "ring" and pass_ == pkg.PASS_FWD
            assert (p.cluster == 1 and 2048 <= nvec <= 3072) or nvec > 8192
        assert p.smem_bytes <= 227 * 1024
        assert p.grid % p.cluster == 0 and p.grid > 0
        if name == "ring" or pass_ in (pkg.PASS_BWD, pkg.PASS_BWD_RES):
            assert 2 <= p.stages <= 6  # the forward's one-shot cluster kernel has no ring


WIDE_GRID = [(N, dt) for N in (24576, 40960, 49152, 65536, 98304)
             for dt in (torch.bfloat16, torch.float32)] + [(131072, torch.bfloat16)]


@pytest.mark.parametrize("N,dtype", WIDE_GRID,
                         ids=[f"{n}-{str(d)[6:]}" for n, d in WIDE_GRID])
def test_wide_rows_around_cluster_grid(N, dtype, w_dtype=None):
    """Rows split over a cluster of the shape chosen on the device: M just
    below, at and above the number of co-resident clusters, and a ragged
    multiple of it."""
    code = pkg.dtype_code(dtype, w_dtype)
    plan = pkg.rmsnorm_plan(1 << 20, N, code, pkg.PASS_BWD, 0)
    P = plan.partial_rows
    assert plan.grid == P * plan.cluster
    for M in sorted({max(1, P - 1), P, P + 1, 2 * P + 3}):
        inp, eps = inputs(M, N, dtype, seed=M % 5, w_dtype=w_dtype)
        out = run(inp["x"], inp["w"], inp["dy"], eps)
        check_all(inp["x"], inp["w"], inp["dy"], eps, *out)


RING_GRID = [(N, dt, wdt) for N in (16384, 24576, 98304, 131072)
             for dt, wdt in ((torch.bfloat16, None), (torch.float16, None),
                             (torch.bfloat16, torch.float32), (torch.float32, None))
             if N > 65536 or dt != torch.float32] + [(262144, torch.bfloat16, None)]


@pytest.mark.parametrize("N,dtype,w_dtype", RING_GRID,
                         ids=[f"{n}-{str(d)[6:]}" + ("-wf32" if w else "") for n, d, w in RING_GRID])
def test_forward_ring_rows_around_grid(N, dtype, w_dtype):
    """The persistent forward at 8 vectors a thread: 16-bit rows of 2048-3072
    vectors in one block and rows wider than 8192 vectors in clusters (16-bit
    slices are read from the ring stage twice and their stage is refilled one
    row late; fp32 slices are held in registers). M around the number of
    resident blocks or clusters and several rows each (more than the ring's
    stages), so that every stage is refilled and reused."""
    code = pkg.dtype_code(dtype, w_dtype)
    plan = pkg.rmsnorm_plan(1 << 20, N, code, pkg.PASS_FWD, 0)
    assert pkg.VARIANTS[plan.variant] == "ring" and plan.vectors_per_thread == 8
    units = plan.grid // plan.cluster
    for M in sorted({max(1, units - 1), units + 1, (plan.stages + 1) * units + 3}):
        inp, eps = inputs(M, N, dtype, seed=M % 3, w_dtype=w_dtype)
        out = run(inp["x"], inp["w"], inp["dy"], eps)
        check_all(inp["x"], inp["w"], inp["dy"], eps, *out)


WIDEST = [(196608, torch.bfloat16, None), (262144, torch.bfloat16, None),
          (262144, torch.float16, torch.float32), (98304, torch.float32, None),
          (131072, torch.float32, None), (196608, torch.float32, None)]


@pytest.mark.parametrize("N,dtype,w_dtype", WIDEST,
                         ids=[f"{n}-{str(d)[6:]}" + ("-wf32" if w else "") for n, d, w in WIDEST])
def test_backward_cluster_of_16(N, dtype, w_dtype):
    """Rows of 256..512 KiB in the backward: a cluster of 16 blocks (the
    exchange of row sums over 16 peers), or for fp32 rows the 8 blocks of 8
    vectors with a two-deep ring that the device's choice may prefer. M
    around the number of resident clusters and several rows per cluster."""
    code = pkg.dtype_code(dtype, w_dtype)
    plan = pkg.rmsnorm_plan(1 << 20, N, code, pkg.PASS_BWD, 0)
    assert pkg.VARIANTS[plan.variant] == "cluster_row"
    assert plan.cluster == 16 or (dtype == torch.float32 and plan.cluster == 8)
    units = plan.grid // plan.cluster
    assert plan.partial_rows == units
    for M in sorted({max(1, units - 1), units + 1, (plan.stages + 1) * units + 3}):
        inp, eps = inputs(M, N, dtype, seed=M % 3, w_dtype=w_dtype)
        out = run(inp["x"], inp["w"], inp["dy"], eps)
        check_all(inp["x"], inp["w"], inp["dy"], eps, *out)


@pytest.mark.parametrize("dtype,w_dtype", TYPES, ids=TYPE_IDS)
@pytest.mark.parametrize("N", [128, 4096, 4104])
def test_unaligned_pointers(N, dtype, w_dtype):
    """Tensors starting one element past a 16-byte boundary take the scalar
    kernels and still match."""
    M = 50
    inp, eps = inputs(M, N, dtype, w_dtype=w_dtype)
    views = {}
    for k in ("x", "dy"):
        buf = torch.empty(M * N + 1, dtype=dtype, device=DEV)
        buf[1:].copy_(inp[k].view(-1))
        views[k] = buf[1:].view(M, N)
    wbuf = torch.empty(N + 1, dtype=inp["w"].dtype, device=DEV)
    wbuf[1:].copy_(inp["w"])
    w = wbuf[1:]
    assert views["x"].data_ptr() % 16 != 0
    out = run(views["x"], w, views["dy"], eps)
    check_all(views["x"], w, views["dy"], eps, *out)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32, torch.float16],
                         ids=["bf16", "f32", "f16"])
def test_worked_examples(dtype):
    """The printed examples of the hello-gpu Fused RMSNorm chapter, section
    13.1 and Figure 13.1, on the GPU (values are exact in bf16)."""
    x = torch.tensor([[3.0, 4.0]], dtype=dtype, device=DEV)
    w = torch.tensor([1.0, 1.0], dtype=dtype, device=DEV)
    y, rstd = pkg.forward(x, w, 1e-5)
    tol = {torch.float32: 5e-5, torch.float16: 5e-4, torch.bfloat16: 4e-3}[dtype]
    assert np.allclose(y.float().cpu().numpy()[0], [0.8485, 1.1314], atol=tol)
    assert abs(rstd.item() - 0.2828) < 5e-5
    x = torch.tensor([[3.0, 4.0, -3.0, -4.0]], dtype=dtype, device=DEV)
    w = torch.tensor([1.0, 0.5, 2.0, 1.0], dtype=dtype, device=DEV)
    y, rstd = pkg.forward(x, w, 1e-5)
    assert abs(y.float()[0, 1].item() - 0.5657) < tol
    assert abs(rstd.item() - 0.2828) < 5e-5


@pytest.mark.parametrize("dtype,w_dtype", TYPES, ids=TYPE_IDS)
@pytest.mark.parametrize("N", [128, 4096, 65536])
def test_special_rows(N, dtype, w_dtype):
    """Zero rows (y = 0, rstd = eps^-1/2), a row with a NaN (propagates to
    that row only), huge values, and zero weights in some columns."""
    M = 6
    inp, eps = inputs(M, N, dtype, w_dtype=w_dtype)
    x, w, dy = inp["x"].clone(), inp["w"].clone(), inp["dy"]
    x[1].zero_()
    x[3, N // 3] = float("nan")
    x[4] *= 1e4 if dtype == torch.float32 else 1e3
    w[: N // 8] = 0
    out = run(x, w, dy, eps)
    y, rstd, dx, dw = out
    assert torch.all(y[1] == 0)
    assert abs(rstd[1].item() - eps ** -0.5) / eps ** -0.5 < 1e-5
    assert torch.isnan(y[3].float()).all() and not torch.isnan(y[2].float()).any()
    keep = [0, 1, 2, 4, 5]
    xc, wc, dyc = x.cpu(), w.cpu(), dy.cpu()
    y_ref, r_ref = oracle.fwd(xc, wc, eps, rows=keep)
    dx_ref = oracle.bwd_dx(xc, wc, dyc, eps, rows=keep)
    check_rows(y[keep], y_ref, dtype, "y")
    check_rows(dx[keep], dx_ref, dtype, "dx")
    check_rstd(rstd[keep], r_ref)
    assert torch.all(y[keep][:, : N // 8] == 0)
    # dw has NaN exactly in the columns the NaN row touches: every column
    assert torch.isnan(dw).all()


def test_empty_and_degenerate():
    x = torch.empty(0, 64, dtype=torch.bfloat16, device=DEV)
    w = torch.ones(64, dtype=torch.bfloat16, device=DEV)
    y = torch.empty_like(x)
    rstd = torch.empty(0, dtype=torch.float32, device=DEV)
    dw = torch.full((64,), 7.0, device=DEV)
    assert pkg.rmsnorm_fwd(x, w, y, rstd, 0, 64, 1e-6, pkg.BF16) == pkg.OK
    assert pkg.rmsnorm_bwd(x, w, x, rstd, y, dw, 0, 64, pkg.BF16) == pkg.OK
    torch.cuda.synchronize()
    assert torch.all(dw == 0), "empty backward must give dw = 0 (the empty sum)"
    # invalid arguments are rejected before anything runs
    assert pkg.rmsnorm_fwd(x, w, y, rstd, 4, 0, 1e-6, pkg.BF16) == pkg.ERR_INVALID_ARG
    assert pkg.rmsnorm_fwd(x, w, y, rstd, 4, 64, -1.0, pkg.BF16) == pkg.ERR_INVALID_ARG
    assert pkg.rmsnorm_fwd(x, w, y, rstd, 4, 64, 1e-6, 9) == pkg.ERR_INVALID_ARG
    assert pkg.rmsnorm_fwd(0, w, y, rstd, 4, 64, 1e-6, pkg.BF16) == pkg.ERR_INVALID_ARG


def test_strided_and_host_tensors_are_refused():
    """The kernels read dense row-major device memory: a transposed view or a
    host tensor raises in the binding and nothing is launched."""
    x = torch.randn(64, 128, device=DEV, dtype=torch.bfloat16)
    w = torch.ones(64, device=DEV, dtype=torch.bfloat16)
    y = torch.full((128, 64), 7.0, device=DEV, dtype=torch.bfloat16)
    rstd = torch.zeros(128, device=DEV)
    with pytest.raises(ValueError, match="contiguous"):
        pkg.rmsnorm_fwd(x.t(), w, y, rstd, 128, 64, 1e-6, pkg.BF16)
    with pytest.raises(ValueError, match="CUDA tensors"):
        pkg.rmsnorm_fwd(x.t().contiguous().cpu(), w, y, rstd, 128, 64, 1e-6, pkg.BF16)
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)


def test_workspace_entry_point():
    M, N = 300, 4096
    inp, eps = inputs(M, N, torch.bfloat16)
    x, w, dy = inp["x"], inp["w"], inp["dy"]
    y, rstd = pkg.forward(x, w, eps)
    need = pkg.rmsnorm_bwd_workspace_size(M, N, pkg.BF16, 0)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    dx = torch.empty_like(x)
    dw = torch.empty(N, dtype=torch.float32, device=DEV)
    # the query covers every alignment class; this call needs the vector plan's
    vec_need = pkg.rmsnorm_plan(M, N, pkg.BF16, pkg.PASS_BWD, 0).workspace_bytes
    assert 0 < vec_need <= need
    assert pkg.rmsnorm_bwd_ws(x, w, dy, rstd, dx, dw, M, N, pkg.BF16, ws, vec_need - 16) == \
        pkg.ERR_INVALID_ARG
    assert pkg.rmsnorm_bwd_ws(x, w, dy, rstd, dx, dw, M, N, pkg.BF16, ws.data_ptr() + 4, need) == \
        pkg.ERR_MISALIGNED
    pkg.check(pkg.rmsnorm_bwd_ws(x, w, dy, rstd, dx, dw, M, N, pkg.BF16, ws, need))
    dx2, dw2 = pkg.backward(x, w, dy, rstd)
    torch.cuda.synchronize()
    assert torch.equal(dx, dx2) and torch.equal(dw, dw2)
    check_all(x, w, dy, eps, y, rstd, dx, dw)


@pytest.mark.parametrize("M,N,dtype", [(1, 4096, torch.bfloat16), (4, 4096, torch.bfloat16),
                                     (2, 128, torch.bfloat16), (1, 13, torch.bfloat16),
                                     (1, 65536, torch.float32), (1, 40960, torch.bfloat16)],
                         ids=["1x4096", "4x4096", "2x128", "1x13", "1x65536f32", "1x40960"])
def test_single_partial_row_is_dw(M, N, dtype):
    """Rows few enough for one block (or one cluster) of the persistent
    backward: its partial row is written to dw directly, with no workspace
    and no column sum; every entry point agrees bit for bit."""
    code = pkg.dtype_code(dtype)
    plan = pkg.rmsnorm_plan(M, N, code, pkg.PASS_BWD, 0)
    if plan.partial_rows != 1:
        # several clusters can be resident; one row per cluster then
        assert M > 1 and plan.partial_rows == min(M, plan.grid // plan.cluster)
        pytest.skip("more than one partial row on this device")
    assert plan.workspace_bytes == 0
    # the size query covers the scalar plan too, which has one partial row
    # per row here: none at M = 1
    assert (pkg.rmsnorm_bwd_workspace_size(M, N, code, 0) == 0) == (M == 1)
    inp, eps = inputs(M, N, dtype, seed=M)
    x, w, dy = inp["x"], inp["w"], inp["dy"]
    y, rstd = pkg.forward(x, w, eps)
    dx = torch.empty_like(x)
    dw = torch.full((N,), float("nan"), dtype=torch.float32, device=DEV)
    pkg.check(pkg.rmsnorm_bwd_ws(x, w, dy, rstd, dx, dw, M, N, code, 0, 0))
    dx2, dw2 = pkg.backward(x, w, dy, rstd)
    torch.cuda.synchronize()
    assert torch.equal(dx, dx2) and torch.equal(dw.view(torch.int32), dw2.view(torch.int32))
    check_all(x, w, dy, eps, y, rstd, dx, dw)
    # the residual backward takes the same path
    dres = inputs(M, N, dtype, seed=M + 50)[0]["dy"]
    dxr = torch.empty_like(x)
    dwr = torch.full((N,), float("nan"), dtype=torch.float32, device=DEV)
    pkg.check(pkg.rmsnorm_add_bwd(x, w, dy, rstd, dres, dxr, dwr, M, N, code))
    torch.cuda.synchronize()
    assert torch.equal(dwr, dw)  # dres does not enter dw
    check_rows(dxr, oracle.add_bwd_dx(x.cpu(), w.cpu(), dy.cpu(), dres.cpu(), eps), dtype, "dx")


FEW = [(16, 4096, torch.bfloat16), (64, 4096, torch.bfloat16), (40, 1024, torch.bfloat16),
       (300, 128, torch.float16), (20, 2880, torch.float32), (9, 257, torch.float32)]


@pytest.mark.parametrize("M,N,dtype", FEW, ids=[f"{m}x{n}-{str(d)[6:]}" for m, n, d in FEW])
def test_few_rows_one_cluster(M, N, dtype):
    """Rows for 2 to 16 blocks run as one thread-block cluster whose blocks add
    their dw rows in rank order through distributed shared memory: no
    workspace, no column sum, dw bit for bit the same on every call, and the
    same results through every backward entry point."""
    code = pkg.dtype_code(dtype)
    plan = pkg.rmsnorm_plan(M, N, code, pkg.PASS_BWD, 0)
    inp, eps = inputs(M, N, dtype, seed=M % 11)
    x, w, dy = inp["x"], inp["w"], inp["dy"]
    vector = pkg.VARIANTS[plan.variant] in ("rowgroup", "cta_row")
    if vector and plan.cluster > 1:
        assert plan.partial_rows == 1 and plan.workspace_bytes == 0
        assert plan.grid == plan.cluster and 2 <= plan.cluster <= 16
    y, rstd, dx, dw = run(x, w, dy, eps)
    check_all(x, w, dy, eps, y, rstd, dx, dw)
    for _ in range(3):
        dx2, dw2 = pkg.backward(x, w, dy, rstd)
        torch.cuda.synchronize()
        assert torch.equal(dx2, dx) and torch.equal(dw2.view(torch.int32), dw.view(torch.int32))
    dx3 = torch.empty_like(x)
    dw3 = torch.full((N,), float("nan"), dtype=torch.float32, device=DEV)
    need = pkg.rmsnorm_bwd_workspace_size(M, N, code, 0)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=DEV)
    pkg.check(pkg.rmsnorm_bwd_ws(x, w, dy, rstd, dx3, dw3, M, N, code, ws, need))
    torch.cuda.synchronize()
    assert torch.equal(dx3, dx) and torch.equal(dw3, dw)


@pytest.mark.parametrize("wl_name", ["hidden4096_16384x4096", "qknorm_1048576x128",
                                     "sweep_bf16_N65536", "sweep_f32_N2880",
                                     "hidden4096_16384x4096_f16",
                                     "hidden4096_16384x4096_bf16_wf32"])
def test_dw_bitwise_repeatable(wl_name):
    """Ten backward calls give bitwise-identical dw and dx."""
    wl = synth.WORKLOADS[wl_name]
    inp = synth.make_inputs(wl, device=DEV)
    y, rstd = pkg.forward(inp["x"], inp["w"], wl.eps)
    dx0, dw0 = pkg.backward(inp["x"], inp["w"], inp["dy"], rstd)
    for _ in range(9):
        dx, dw = pkg.backward(inp["x"], inp["w"], inp["dy"], rstd)
        assert torch.equal(dw.view(torch.int32), dw0.view(torch.int32))
        bits = torch.int32 if wl.dtype == torch.float32 else torch.int16
        assert torch.equal(dx.view(bits), dx0.view(bits))


FULL = ["small_256x1024", "hidden4096_16384x4096", "hidden4096_16384x4096_f16",
        "hidden4096_16384x4096_bf16_wf32", "hidden8192_32768x8192_outliers",
        "qknorm_1048576x128"] + [w.name for w in synth.width_sweep(torch.bfloat16)] + \
       [w.name for w in synth.width_sweep(torch.float32)]


@pytest.mark.parametrize("wl_name", FULL)
def test_full_size_sampled(wl_name):
    """Full workload sizes: every column of >= 4096 random rows (plus the
    first and last) for y, rstd and dx; all of dw."""
    wl = synth.WORKLOADS[wl_name]
    inp = synth.make_inputs(wl, device=DEV)
    x, w, dy = inp["x"], inp["w"], inp["dy"]
    if wl.outlier_frac:
        big = (x.float().abs() > 20).sum().item()
        assert big >= 0.8 * synth.outlier_count(wl)
    out = run(x, w, dy, wl.eps)
    M = wl.M
    rng = np.random.default_rng(12345)
    rows = np.unique(np.concatenate([[0, M - 1], rng.choice(M, size=min(M, 4096), replace=False)]))
    check_all(x, w, dy, wl.eps, *out, rows=rows)


RING = [(16384, torch.bfloat16, None), (65536, torch.bfloat16, None), (65536, torch.float32, None),
        (8192, torch.bfloat16, torch.float32), (32768, torch.float16, None)]


@pytest.mark.parametrize("N,dtype,w_dtype", RING,
                         ids=[f"{n}-{str(d)[6:]}" + ("-wf32" if wd else "") for n, d, wd in RING])
def test_ring_forward_around_its_grid(N, dtype, w_dtype):
    """The persistent ring forward with M just below, at and above the number
    of co-resident clusters, and a few rows per cluster: some clusters walk
    one row more than others. Sampled rows plus the first and last."""
    code = pkg.dtype_code(dtype, w_dtype)
    plan = pkg.rmsnorm_plan(1 << 20, N, code, pkg.PASS_FWD, 0)
    assert pkg.VARIANTS[plan.variant] == "ring", pkg.VARIANTS[plan.variant]
    P = plan.grid // plan.cluster
    for M in sorted({max(1, P - 1), P, P + 1, 3 * P + 2}):
        inp, eps = inputs(M, N, dtype, seed=M % 3, w_dtype=w_dtype)
        out = run(inp["x"], inp["w"], inp["dy"], eps)
        rows = np.unique(np.concatenate([[0, M - 1], np.arange(0, M, max(1, M // 40))]))
        check_all(inp["x"], inp["w"], inp["dy"], eps, *out, rows=rows)
