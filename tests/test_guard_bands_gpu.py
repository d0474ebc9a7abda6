"""Guard bands around every output: a write outside a tensor shows.

Each output (y, rstd, dx, dw, h, and the caller's workspace of rmsnorm_bwd_ws)
is carved out of a larger buffer with 4 KiB of a fixed byte pattern before
and after it; after the call both bands must be unchanged, and the inputs
must be unchanged too. The shapes are the ones where a stray write would
land: ragged row tails, rows around the persistent grid and the cluster grid,
unaligned pointers (scalar kernels), single partial rows (dw written
directly), every kernel family and dtype code. The outputs are also checked
against the fp64 oracle, so the bands cannot pass on a call that wrote
nothing. Run against the checked debug build too (test_checked_build_gpu).
"""
from __future__ import annotations

import pytest
import torch

import oracle
from parity_util import check_dw, check_rows, check_rstd

pytestmark = pytest.mark.gpu

pkg = pytest.importorskip("memory_bound_normalization_gb300")
from memory_bound_normalization_gb300 import synth  # noqa: E402

DEV = "cuda:0"
BAND = 4096  # bytes of pattern on each side of an output
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.set_device(0)
    pkg.load_library(build_if_missing=True)
    oracle.build()
    yield


class Guarded:
    """An output tensor with BAND bytes of PATTERN on both sides; `shift`
    moves its start by that many bytes off 16-byte alignment."""

    def __init__(self, shape, dtype, shift: int = 0, fill=float("nan")):
        elem = torch.empty(0, dtype=dtype).element_size()
        n = 1
        for d in shape:
            n *= d
        self.nbytes = n * elem
        self.raw = torch.full((BAND + shift + self.nbytes + BAND,), PATTERN, dtype=torch.uint8,
                              device=DEV)
        lo = BAND + shift
        self.lo, self.hi = lo, lo + self.nbytes
        self.t = self.raw[lo:self.hi].view(dtype).view(*shape)
        if self.nbytes:
            self.t.fill_(fill)

    def bands_intact(self) -> bool:
        return bool(torch.all(self.raw[:self.lo] == PATTERN)) and \
            bool(torch.all(self.raw[self.hi:] == PATTERN))


def make(M, N, dtype, w_dtype=None, seed=0):
    wl = synth.Workload(f"g{M}x{N}", M, N, dtype, 1e-5, 400 + seed, 500 + seed, 600 + seed,
                        w_dtype=w_dtype)
    return synth.make_inputs(wl, device=DEV), wl.eps


def check_oracle(x, w, dy, eps, y, rstd, dx, dw):
    xc, wc, dyc = x.cpu(), w.cpu(), dy.cpu()
    y_ref, r_ref = oracle.fwd(xc, wc, eps)
    check_rows(y, y_ref, x.dtype, "y")
    check_rstd(rstd, r_ref)
    check_rows(dx, oracle.bwd_dx(xc, wc, dyc, eps), x.dtype, "dx")
    check_dw(dw, oracle.bwd_dw(xc, dyc, eps))


def run_guarded(M, N, dtype, w_dtype=None, shift=0, workspace=False, seed=0):
    inp, eps = make(M, N, dtype, w_dtype, seed)
    x, w, dy = inp["x"], inp["w"], inp["dy"]
    if shift:
        # inputs moved off 16-byte alignment as well: the scalar kernels
        def moved(t):
            g = Guarded(tuple(t.shape), t.dtype, shift)
            g.t.copy_(t)
            return g.t
        x, dy = moved(x), moved(dy)
    keep = [t.clone() for t in (x, w, dy)]
    code = pkg.dtype_code(dtype, w_dtype)
    y = Guarded((M, N), dtype, shift)
    dx = Guarded((M, N), dtype, shift)
    rstd = Guarded((M,), torch.float32)
    dw = Guarded((N,), torch.float32)
    pkg.check(pkg.rmsnorm_fwd(x, w, y.t, rstd.t, M, N, eps, code), "fwd")
    if workspace:
        need = pkg.rmsnorm_bwd_workspace_size(M, N, code, 0)
        ws = Guarded((max(need, 16),), torch.uint8, fill=0)
        pkg.check(pkg.rmsnorm_bwd_ws(x, w, dy, rstd.t, dx.t, dw.t, M, N, code, ws.t, need),
                  "bwd_ws")
    else:
        ws = None
        pkg.check(pkg.rmsnorm_bwd(x, w, dy, rstd.t, dx.t, dw.t, M, N, code), "bwd")
    st = pkg.rmsnorm_get_last_device_error()
    assert st == pkg.OK, pkg.rmsnorm_status_string(st)
    for name, g in (("y", y), ("dx", dx), ("rstd", rstd), ("dw", dw), ("workspace", ws)):
        if g is not None:
            assert g.bands_intact(), f"a write landed outside {name}"
    for a, b in zip((x, w, dy), keep):
        assert torch.equal(a, b), "an input changed"
    check_oracle(x, w, dy, eps, y.t, rstd.t, dx.t, dw.t)


TYPES = [(torch.bfloat16, None), (torch.float32, None), (torch.float16, None),
         (torch.bfloat16, torch.float32), (torch.float16, torch.float32)]
TYPE_IDS = ["bf16", "f32", "f16", "bf16_wf32", "f16_wf32"]
SHAPES = [(1, 8), (3, 13), (33, 257), (100, 64), (130, 128), (37, 256), (19, 512), (256, 1024),
          (9, 2880), (6, 4096), (5, 6144), (3, 16384), (5, 24576), (3, 40960), (2, 65536),
          (3, 131072), (1000, 40), (777, 96)]


@pytest.mark.parametrize("dtype,w_dtype", TYPES, ids=TYPE_IDS)
@pytest.mark.parametrize("M,N", SHAPES, ids=[f"{m}x{n}" for m, n in SHAPES])
def test_bands_small_shapes(M, N, dtype, w_dtype):
    run_guarded(M, N, dtype, w_dtype)


def grid_rows(N, dtype, w_dtype=None):
    """Row counts just around the backward's persistent grid (rows a full
    grid takes in one pass), and around the forward's when it persists."""
    code = pkg.dtype_code(dtype, w_dtype)
    p = pkg.rmsnorm_plan(1 << 22, N, code, pkg.PASS_BWD, 0)
    full = p.partial_rows * max(1, p.rows_per_unit if p.variant in (1, 2) else 1)
    return sorted({max(1, full - 1), full, full + 1})


@pytest.mark.parametrize("dtype,w_dtype", TYPES, ids=TYPE_IDS)
@pytest.mark.parametrize("N", [128, 1024, 4096, 16384, 65536])
def test_bands_around_persistent_grid(N, dtype, w_dtype):
    for M in grid_rows(N, dtype, w_dtype):
        if M * N > (1 << 26):
            continue
        run_guarded(M, N, dtype, w_dtype, seed=M % 7)


@pytest.mark.parametrize("dtype,w_dtype", TYPES[:3], ids=TYPE_IDS[:3])
@pytest.mark.parametrize("N", [128, 4104, 4096])
def test_bands_unaligned(N, dtype, w_dtype):
    elem = torch.empty(0, dtype=dtype).element_size()
    run_guarded(37, N, dtype, w_dtype, shift=elem)


@pytest.mark.parametrize("M,N,dtype", [(300, 4096, torch.bfloat16), (4096, 128, torch.bfloat16),
                                       (64, 65536, torch.float32), (1, 4096, torch.bfloat16)])
def test_bands_caller_workspace(M, N, dtype):
    run_guarded(M, N, dtype, workspace=True)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M,N", [(130, 128), (37, 4096), (3, 65536), (33, 257)])
def test_bands_residual(M, N, dtype):
    inp, eps = make(M, N, dtype, seed=3)
    more, _ = make(M, N, dtype, seed=4)
    x, w, dy, res, dres = inp["x"], inp["w"], inp["dy"], more["x"], more["dy"]
    keep = [t.clone() for t in (x, w, dy, res, dres)]
    code = pkg.dtype_code(dtype)
    h, y, dx = (Guarded((M, N), dtype) for _ in range(3))
    rstd, dw = Guarded((M,), torch.float32), Guarded((N,), torch.float32)
    pkg.check(pkg.rmsnorm_add_fwd(x, res, w, h.t, y.t, rstd.t, M, N, eps, code), "add_fwd")
    pkg.check(pkg.rmsnorm_add_bwd(h.t, w, dy, rstd.t, dres, dx.t, dw.t, M, N, code), "add_bwd")
    assert pkg.rmsnorm_get_last_device_error() == pkg.OK
    for name, g in (("h", h), ("y", y), ("dx", dx), ("rstd", rstd), ("dw", dw)):
        assert g.bands_intact(), f"a write landed outside {name}"
    for a, b in zip((x, w, dy, res, dres), keep):
        assert torch.equal(a, b), "an input changed"
    h_ref, y_ref, r_ref = oracle.add_fwd(x.cpu(), res.cpu(), w.cpu(), eps)
    check_rows(y.t, y_ref, dtype, "y")
    check_rstd(rstd.t, r_ref)
    hc = h.t.cpu()
    check_rows(dx.t, oracle.add_bwd_dx(hc, w.cpu(), dy.cpu(), dres.cpu(), eps), dtype, "dx")
    check_dw(dw.t, oracle.bwd_dw(hc, dy.cpu(), eps))
