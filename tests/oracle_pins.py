"""Pins for the fp64 oracle: checks against facts that do not come from the
oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with what the pages or the mathematics fix:

* values the pages print for worked examples (``tests/golden``);
* closed forms derived by hand from the definitions (identities that hold for
  any input, special inputs with a known answer);
* central finite differences of the forward, which pin the backward to the
  forward without restating the backward formula;
* an independent library implementation (PyTorch's ``rms_norm`` with autograd
  in float64 on the CPU).

The same functions run against deliberately broken copies of the oracle in
``test_oracle_mutants.py``; every plausible mistake must trip at least one.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_examples.json")


def _golden():
    with open(GOLDEN) as f:
        return {c["name"]: c for c in json.load(f)["cases"]}


def _rng(seed):
    return np.random.default_rng(seed)


def _rows(M, N, seed, scale=1.0):
    return _rng(seed).standard_normal((M, N)) * scale


# ---------------------------------------------------------------- printed values

def pin_printed_two_columns(o):
    """hello-gpu ch. 13 section 13.1: x=[3,4], w=[1,1], eps=1e-5 -> r~0.2828,
    y~[0.8485, 1.1314]; the sum of squares is 25 and its mean 12.5."""
    c = _golden()["two_columns"]
    p = c["printed"]
    y, r = o.fwd(np.array([c["x"]]), np.array(c["w"]), c["eps"])
    d = c["decimals"]
    assert np.allclose(np.round(y[0], d), p["y"], atol=0, rtol=0), y
    assert round(float(r[0]), d) == p["r"], r
    mean_square = 1.0 / float(r[0]) ** 2 - c["eps"]
    assert abs(mean_square - p["mean_square"]) < 1e-9, mean_square
    assert abs(mean_square * len(c["x"]) - p["sum_of_squares"]) < 1e-9


def pin_printed_four_columns(o):
    """hello-gpu ch. 13 Figure 13.1: x=[3,4,-3,-4], w=[1,.5,2,1], eps=1e-5 ->
    sum of squares 50, mean over the 4 valid columns 12.5, r~0.2828,
    second output 4 * 0.2828 * 0.5 ~ 0.5657; every output shares r and keeps
    its input's sign."""
    c = _golden()["four_columns_with_weights"]
    p = c["printed"]
    x, w = np.array([c["x"]]), np.array(c["w"])
    y, r = o.fwd(x, w, c["eps"])
    d = c["decimals"]
    assert round(float(y[0, p["y_index"]]), d) == p["y_at_index"], y
    assert round(float(r[0]), d) == p["r"], r
    mean_square = 1.0 / float(r[0]) ** 2 - c["eps"]
    assert abs(mean_square - p["mean_square"]) < 1e-9, mean_square
    assert abs(mean_square * 4 - p["sum_of_squares"]) < 1e-9
    assert np.all(np.sign(y[0]) == np.sign(x[0])), y
    # one shared scale: y_j / (x_j w_j) is the same r for every column
    assert np.allclose(y[0] / (x[0] * w), r[0], rtol=1e-14, atol=0)


# ---------------------------------------------------------------- closed forms

def pin_zero_input(o):
    """All-zero rows give all-zero outputs and r = eps^(-1/2) (hello-gpu 13.4)."""
    eps = 1e-5
    x = np.zeros((3, 7))
    w = _rng(1).standard_normal(7)
    y, r = o.fwd(x, w, eps)
    assert np.all(y == 0.0)
    assert np.allclose(r, 1.0 / math.sqrt(eps), rtol=1e-15, atol=0), r


def pin_zero_weight(o):
    """All-zero weights give y = 0 (hello-gpu 13.4) and, since g = dy*w = 0,
    dx = 0."""
    x = _rows(4, 9, 2)
    w = np.zeros(9)
    dy = _rows(4, 9, 3)
    y, _ = o.fwd(x, w, 1e-5)
    dx = o.bwd_dx(x, w, dy, 1e-5)
    assert np.all(y == 0.0)
    assert np.all(dx == 0.0)


def pin_constant_row(o):
    """x = a*1 gives r = 1/sqrt(a^2 + eps), so y = a*w/sqrt(a^2 + eps)."""
    for a, eps in ((2.5, 1e-5), (-0.75, 1e-2), (1e-3, 1e-6)):
        N = 11
        x = np.full((1, N), a)
        w = _rng(4).standard_normal(N)
        y, r = o.fwd(x, w, eps)
        assert math.isclose(r[0], 1.0 / math.sqrt(a * a + eps), rel_tol=1e-14)
        assert np.allclose(y[0], a * w / math.sqrt(a * a + eps), rtol=1e-13, atol=0)


def pin_scale_invariance(o):
    """With eps = 0, y(alpha*x) = y(x) for alpha > 0; with eps != 0 it is not
    exactly invariant (hello-gpu 13.4)."""
    x = _rows(3, 17, 5)
    w = _rng(6).standard_normal(17)
    y1, _ = o.fwd(x, w, 0.0)
    y2, _ = o.fwd(3.7 * x, w, 0.0)
    assert np.allclose(y1, y2, rtol=1e-13, atol=1e-15)
    small = x * 1e-3  # mean square ~1e-6, comparable with eps
    y3, _ = o.fwd(small, w, 1e-6)
    y4, _ = o.fwd(2.0 * small, w, 1e-6)
    assert not np.allclose(y3, y4, rtol=1e-3, atol=0)


def pin_backward_two_columns(o):
    """Derived by hand from the definitions: x=[3,4], w=[1,1], dy=[1,0], eps=0.
    r = 1/sqrt(12.5), xhat = [0.8485281, 1.1313708], mean(g*xhat) = 0.4242641,
    dx = r*([1,0] - xhat*0.4242641) = r*[0.64, -0.48], dw = [0.8485281, 0]."""
    x = np.array([[3.0, 4.0]])
    w = np.array([1.0, 1.0])
    dy = np.array([[1.0, 0.0]])
    r = 1.0 / math.sqrt(12.5)
    dx = o.bwd_dx(x, w, dy, 0.0)
    dw = o.bwd_dw(x, dy, 0.0)
    assert np.allclose(dx[0], [0.64 * r, -0.48 * r], rtol=1e-13, atol=1e-16), dx
    assert np.allclose(dw, [3.0 * r, 0.0], rtol=1e-13, atol=1e-16), dw


def pin_dx_orthogonal_to_x(o):
    """sum_j dx_ij x_ij = eps * r_i^3 * sum_j g_ij x_ij (derived from the
    definitions); exactly zero when eps = 0."""
    M, N = 5, 23
    x = _rows(M, N, 7)
    w = 1.0 + 0.1 * _rng(8).standard_normal(N)
    dy = _rows(M, N, 9)
    for eps in (0.0, 1e-6, 0.25):
        dx = o.bwd_dx(x, w, dy, eps)
        _, r = o.fwd(x, w, eps)
        lhs = np.sum(dx * x, axis=1)
        rhs = eps * r ** 3 * np.sum(dy * w * x, axis=1)
        scale = np.sum(np.abs(dy * w * x), axis=1) * r
        assert np.all(np.abs(lhs - rhs) <= 1e-12 * scale), (eps, lhs, rhs)


def pin_dy_equal_y(o):
    """dy = y, w = 1, eps = 0 gives dx = 0 (g = xhat and mean(xhat^2) = 1)."""
    M, N = 3, 19
    x = _rows(M, N, 10)
    w = np.ones(N)
    y, _ = o.fwd(x, w, 0.0)
    dx = o.bwd_dx(x, w, y, 0.0)
    assert np.max(np.abs(dx)) < 1e-14, np.max(np.abs(dx))


def pin_single_row_dw(o):
    """One row: dw_j = dy_j * xhat_j = dy_j * y_j / w_j, tying dw to the
    forward output."""
    N = 13
    x = _rows(1, N, 11)
    w = 1.0 + 0.1 * _rng(12).standard_normal(N)
    dy = _rows(1, N, 13)
    y, _ = o.fwd(x, w, 1e-5)
    dw = o.bwd_dw(x, dy, 1e-5)
    assert np.allclose(dw, dy[0] * y[0] / w, rtol=1e-13, atol=0)


def pin_dw_sums_rows(o):
    """dw over M rows is the sum of the single-row weight gradients."""
    M, N = 6, 10
    x = _rows(M, N, 14)
    dy = _rows(M, N, 15)
    total = o.bwd_dw(x, dy, 1e-5)
    parts = sum(o.bwd_dw(x[i:i + 1], dy[i:i + 1], 1e-5) for i in range(M))
    assert np.allclose(total, parts, rtol=1e-13, atol=1e-15)


# ------------------------------------------------------- finite differences

def pin_finite_differences(o):
    """dx and dw equal the central differences of L = sum(dy * y) (forward
    only), h = 1e-6, in float64."""
    h = 1e-6
    for (M, N, eps, seed) in ((1, 3, 1e-5, 20), (3, 8, 1e-6, 21), (4, 16, 0.5, 22), (2, 5, 0.0, 23)):
        x = _rows(M, N, seed)
        w = 1.0 + 0.3 * _rng(seed + 100).standard_normal(N)
        dy = _rows(M, N, seed + 200)

        def loss(xx, ww):
            y, _ = o.fwd(xx, ww, eps)
            return float(np.sum(dy * y))

        fd_x = np.zeros_like(x)
        for i in range(M):
            for j in range(N):
                xp, xm = x.copy(), x.copy()
                xp[i, j] += h
                xm[i, j] -= h
                fd_x[i, j] = (loss(xp, w) - loss(xm, w)) / (2 * h)
        fd_w = np.zeros(N)
        for j in range(N):
            wp, wm = w.copy(), w.copy()
            wp[j] += h
            wm[j] -= h
            fd_w[j] = (loss(x, wp) - loss(x, wm)) / (2 * h)
        dx = o.bwd_dx(x, w, dy, eps)
        dw = o.bwd_dw(x, dy, eps)
        tol_x = 1e-7 * max(1.0, np.max(np.abs(fd_x)))
        tol_w = 1e-7 * max(1.0, np.max(np.abs(fd_w)))
        assert np.max(np.abs(dx - fd_x)) < tol_x, (M, N, np.max(np.abs(dx - fd_x)))
        assert np.max(np.abs(dw - fd_w)) < tol_w, (M, N, np.max(np.abs(dw - fd_w)))


# ------------------------------------------------ independent library routine

def pin_torch_rms_norm(o):
    """PyTorch's CPU float64 rms_norm with autograd agrees to ~1e-12."""
    import torch
    import torch.nn.functional as F

    for (M, N, eps, seed) in ((7, 33, 1e-6, 30), (2, 128, 1e-5, 31), (5, 4, 1e-2, 32)):
        g = torch.Generator().manual_seed(seed)
        x = torch.randn(M, N, dtype=torch.float64, generator=g)
        w = 1.0 + 0.1 * torch.randn(N, dtype=torch.float64, generator=g)
        dy = torch.randn(M, N, dtype=torch.float64, generator=g)
        xt, wt = x.clone().requires_grad_(True), w.clone().requires_grad_(True)
        yt = F.rms_norm(xt, (N,), wt, eps)
        yt.backward(dy)
        y, _ = o.fwd(x, w, eps)
        dx = o.bwd_dx(x, w, dy, eps)
        dw = o.bwd_dw(x, dy, eps)
        assert np.allclose(y, yt.detach().numpy(), rtol=1e-12, atol=1e-14)
        assert np.allclose(dx, xt.grad.numpy(), rtol=1e-10, atol=1e-13)
        assert np.allclose(dw, wt.grad.numpy(), rtol=1e-10, atol=1e-13)


# ------------------------------------------------------ input decoding, rows

def pin_bf16_decoding(o):
    """bf16 bit patterns decode exactly: 0x3F80 = 1, 0xC040 = -3,
    0x4049 = 3.140625, 0x0001 = 2^-133 (a subnormal); the oracle sees the same
    values whether they arrive as bf16 bits, fp32 or fp64."""
    bits = np.array([[0x3F80, 0xC040, 0x4049, 0x0001]], dtype=np.uint16)
    vals = np.array([[1.0, -3.0, 3.140625, 2.0 ** -133]])
    wb = np.array([0x3F80, 0x3F80, 0x3F80, 0x3F80], dtype=np.uint16)
    y_b, r_b = o.fwd(bits, wb, 1e-5, dtype="bf16")
    y_d, r_d = o.fwd(vals, np.ones(4), 1e-5)
    y_f, r_f = o.fwd(vals.astype(np.float32), np.ones(4, dtype=np.float32), 1e-5)
    assert np.array_equal(y_b, y_d) and np.array_equal(r_b, r_d), (y_b, y_d)
    assert np.array_equal(y_f, y_d) and np.array_equal(r_f, r_d)


def pin_f16_decoding(o):
    """binary16 bit patterns decode exactly: 0x3C00 = 1, 0xC000 = -2,
    0x0001 = 2^-24 (smallest subnormal), 0x0400 = 2^-14 (smallest normal),
    0x7BFF = 65504 (largest finite); every pattern agrees with numpy's
    float16 conversion, and fp16 input gives the same outputs as the same
    values in fp64."""
    bits = np.array([[0x3C00, 0xC000, 0x3555, 0x0001, 0x7BFF, 0x0400, 0x8001, 0x3FFF]],
                    dtype=np.uint16)
    vals = bits.view(np.float16).astype(np.float64)
    assert vals[0, 0] == 1.0 and vals[0, 1] == -2.0 and vals[0, 3] == 2.0 ** -24
    assert vals[0, 4] == 65504.0 and vals[0, 5] == 2.0 ** -14 and vals[0, 6] == -(2.0 ** -24)
    w = np.ones(8)
    y_h, r_h = o.fwd(bits.view(np.float16), w, 1e-5)
    y_d, r_d = o.fwd(vals, w, 1e-5)
    assert np.array_equal(y_h, y_d) and np.array_equal(r_h, r_d), (y_h, y_d)
    every = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16).reshape(256, 256)
    finite = np.isfinite(every.view(np.float16))
    y_all, r_all = o.fwd(every.view(np.float16), np.ones(256), 1.0)
    x_all = every.view(np.float16).astype(np.float64)
    rows_ok = finite.all(axis=1)
    y_ref = x_all[rows_ok] * r_all[rows_ok][:, None]
    assert np.array_equal(y_all[rows_ok], y_ref)


def pin_mixed_weight_dtype(o):
    """A weight stored in its own type (an fp32 master weight with bf16 or
    fp16 activations, "What a tuned RMSNorm kernel actually costs on Hopper",
    section 07) gives exactly what the same values give in fp64."""
    import torch

    g = torch.Generator().manual_seed(50)
    for act in (torch.bfloat16, torch.float16):
        x = torch.randn(3, 16, generator=g).to(act)
        dy = torch.randn(3, 16, generator=g).to(act)
        w = (1.0 + 0.1 * torch.randn(16, generator=g)).float()
        y1, r1 = o.fwd(x, w, 1e-5)
        y2, r2 = o.fwd(x.double(), w.double(), 1e-5)
        assert np.array_equal(y1, y2) and np.array_equal(r1, r2)
        dx1 = o.bwd_dx(x, w, dy, 1e-5)
        dx2 = o.bwd_dx(x.double(), w.double(), dy.double(), 1e-5)
        assert np.array_equal(dx1, dx2)


def pin_row_selection(o):
    """A requested row list returns exactly those rows, in the order given."""
    x = _rows(6, 5, 40)
    w = _rng(41).standard_normal(5)
    dy = _rows(6, 5, 42)
    y_all, r_all = o.fwd(x, w, 1e-5)
    dx_all = o.bwd_dx(x, w, dy, 1e-5)
    rows = [5, 0, 3]
    y, r = o.fwd(x, w, 1e-5, rows=rows)
    dx = o.bwd_dx(x, w, dy, 1e-5, rows=rows)
    assert np.array_equal(y, y_all[rows]) and np.array_equal(r, r_all[rows])
    assert np.array_equal(dx, dx_all[rows])
    # each row is computed from itself only
    y_last, _ = o.fwd(x[5:6], w, 1e-5)
    assert np.array_equal(y_last[0], y_all[5])


def pin_nan_and_inf_rows(o):
    """IEEE 754 semantics of the definition on non-finite input: a NaN in a
    row makes that row's sum of squares NaN, so its r, y and dx are NaN in
    every column and every column of dw is NaN; an infinity makes the sum
    infinite, so r = 1/sqrt(inf) = 0, y is 0 except NaN (inf * 0) where the
    infinity sits, and dx is NaN across the row (its dot with g is NaN).
    Rows without such values are computed as if the others were absent."""
    x = _rows(4, 7, 50)
    w = _rng(51).standard_normal(7)
    dy = _rows(4, 7, 52)
    x[1, 3] = math.nan
    x[2, 5] = math.inf
    y, r = o.fwd(x, w, 1e-5)
    dx = o.bwd_dx(x, w, dy, 1e-5)
    dw = o.bwd_dw(x, dy, 1e-5)
    assert np.isnan(r[1]) and np.isnan(y[1]).all() and np.isnan(dx[1]).all()
    assert r[2] == 0.0
    assert np.isnan(y[2, 5]) and np.all(y[2, np.arange(7) != 5] == 0.0)
    assert np.isnan(dx[2]).all()
    assert np.isnan(dw).all()
    clean = [0, 3]
    y_c, r_c = o.fwd(x[clean], w, 1e-5)
    dx_c = o.bwd_dx(x[clean], w, dy[clean], 1e-5)
    assert np.array_equal(y[clean], y_c) and np.array_equal(r[clean], r_c)
    assert np.array_equal(dx[clean], dx_c)


# ------------------------------------------------- rounding and residual add

def _f16_ties(rng, n):
    """Doubles exactly halfway between adjacent finite fp16 values (both
    signs), with the expected round-to-nearest-even result."""
    bits = rng.integers(0, 0x7BFF, size=n, dtype=np.uint16)  # a, a+1 both finite
    lo = bits.view(np.float16).astype(np.float64)
    hi = (bits + 1).view(np.float16).astype(np.float64)
    mid = (lo + hi) / 2
    want = np.where(bits % 2 == 0, lo, hi)
    return np.concatenate([mid, -mid]), np.concatenate([want, -want])


def pin_rounding_matches_numpy(o):
    """Rounding a double into fp16 or fp32 agrees with numpy's conversions
    (IEEE 754 round to nearest even) on normal, subnormal, overflow and
    signed-zero inputs, and every exact fp16 tie goes to the even neighbour."""
    rng = _rng(60)
    v = rng.standard_normal(6000) * 10.0 ** rng.uniform(-10, 6, 6000)
    v = np.concatenate([v, [0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 1e6, 2.0 ** -25,
                            -(2.0 ** -25), 3 * 2.0 ** -26, 2.0 ** -24, 1e-30, 3.4e38, 3.5e38,
                            -3.5e38, 1e-46, 2.0 ** -150, 3 * 2.0 ** -151]])
    with np.errstate(over="ignore"):
        want16 = v.astype(np.float16).astype(np.float64)
        want32 = v.astype(np.float32).astype(np.float64)
    got16, got32 = o.round_to(v, "f16"), o.round_to(v, "f32")
    assert np.array_equal(got16, want16), v[got16 != want16][:5]
    assert np.array_equal(np.signbit(got16), np.signbit(want16))
    assert np.array_equal(got32, want32), v[got32 != want32][:5]
    ties, want = _f16_ties(rng, 3000)
    assert np.array_equal(o.round_to(ties, "f16"), want)


def pin_bf16_rounding(o):
    """bf16 rounding: float32 inputs round as torch's float32 -> bfloat16
    conversion (nearest even); exact ties between adjacent bf16 values go to
    the even bit pattern and a nudge either side goes to the nearer one;
    rounding up past the largest finite bf16 gives an infinity."""
    import torch

    rng = _rng(61)
    v32 = (rng.standard_normal(6000) * 10.0 ** rng.uniform(-30, 30, 6000)).astype(np.float32)
    want = torch.from_numpy(v32).to(torch.bfloat16).double().numpy()
    assert np.array_equal(o.round_to(v32.astype(np.float64), "bf16"), want)
    bits = rng.integers(0, 0x7F7F, size=3000).astype(np.int16)  # a, a+1 both finite
    lo = torch.from_numpy(bits).view(torch.bfloat16).double().numpy()
    hi = torch.from_numpy(bits + 1).view(torch.bfloat16).double().numpy()
    mid, gap = (lo + hi) / 2, hi - lo
    assert np.array_equal(o.round_to(mid, "bf16"), np.where(bits % 2 == 0, lo, hi))
    assert np.array_equal(o.round_to(mid + gap / 8, "bf16"), hi)
    assert np.array_equal(o.round_to(mid - gap / 8, "bf16"), lo)
    assert np.array_equal(o.round_to(-mid - gap / 8, "bf16"), -hi)
    big = float(torch.finfo(torch.bfloat16).max)
    half_ulp = 2.0 ** (127 - 8)
    r = o.round_to([big, big + half_ulp * 0.99, big + half_ulp, -(big + half_ulp)], "bf16")
    assert r[0] == big and r[1] == big and r[2] == math.inf and r[3] == -math.inf


def pin_add_printed_example(o):
    """hello-gpu ch. 13 section 13.1 values through the residual path: x = [1, 1]
    plus residual [2, 3] is the printed row [3, 4], so h = [3, 4], r ~ 0.2828
    and y ~ [0.8485, 1.1314]."""
    c = _golden()["two_columns"]
    p = c["printed"]
    d = c["decimals"]
    xr = np.array([c["x"]])
    res = np.array([[2.0, 3.0]])
    h, y, r = o.add_fwd(xr - res, res, np.array(c["w"]), c["eps"])
    assert np.array_equal(h, xr)
    assert np.allclose(np.round(y[0], d), p["y"], atol=0, rtol=0), y
    assert round(float(r[0]), d) == p["r"], r


def pin_add_stored_sum(o):
    """The stored sum h equals the addition done in the stored type by numpy
    (fp32, fp16) and torch (bf16), and y, r equal the forward of that stored
    h: adding in the type, then normalising."""
    import torch

    rng = _rng(62)
    M, N = 7, 33
    a = rng.standard_normal((M, N)) * 10.0 ** rng.uniform(-3, 3, (M, N))
    b = rng.standard_normal((M, N)) * 10.0 ** rng.uniform(-3, 3, (M, N))
    w = 1.0 + 0.1 * rng.standard_normal(N)
    cases = []
    a32, b32 = a.astype(np.float32), b.astype(np.float32)
    cases.append((a32, b32, a32 + b32))
    with np.errstate(over="ignore"):
        a16, b16 = a.astype(np.float16), b.astype(np.float16)
    cases.append((a16, b16, a16 + b16))
    ab, bb = torch.from_numpy(a32).bfloat16(), torch.from_numpy(b32).bfloat16()
    cases.append((ab, bb, ab + bb))
    for xx, rr, hh in cases:
        h, y, r = o.add_fwd(xx, rr, w, 1e-5)
        want_h = hh.double().numpy() if isinstance(hh, torch.Tensor) else hh.astype(np.float64)
        assert np.array_equal(h, want_h)
        y2, r2 = o.fwd(hh, w, 1e-5)
        assert np.array_equal(y, y2) and np.array_equal(r, r2)


def pin_add_finite_differences(o):
    """The residual backward is the gradient of L = sum(dy * y(x + res)) +
    sum(dres * (x + res)) with respect to x and to res (central differences
    in float64, h = 1e-6); without dres it is the norm's gradient alone."""
    hstep = 1e-6
    M, N, eps = 2, 6, 1e-4
    x, res = _rows(M, N, 63), _rows(M, N, 64)
    w = 1.0 + 0.3 * _rng(65).standard_normal(N)
    dy, dres = _rows(M, N, 66), _rows(M, N, 67)
    for g_extra in (dres, None):
        def loss(xx, rr):
            hh, y, _ = o.add_fwd(xx, rr, w, eps)
            extra = 0.0 if g_extra is None else float(np.sum(g_extra * hh))
            return float(np.sum(dy * y)) + extra

        h, _, _ = o.add_fwd(x, res, w, eps)
        got = o.add_bwd_dx(h, w, dy, g_extra, eps)
        for which in (0, 1):
            fd = np.zeros_like(x)
            for i in range(M):
                for j in range(N):
                    args_p, args_m = [x.copy(), res.copy()], [x.copy(), res.copy()]
                    args_p[which][i, j] += hstep
                    args_m[which][i, j] -= hstep
                    fd[i, j] = (loss(*args_p) - loss(*args_m)) / (2 * hstep)
            assert np.allclose(got, fd, rtol=1e-6, atol=1e-8), (which, got - fd)
        # a row subset gives the same rows
        sub = o.add_bwd_dx(h, w, dy, g_extra, eps, rows=[1, 0])
        assert np.array_equal(sub, got[[1, 0]])


ALL_PINS = [
    pin_printed_two_columns,
    pin_printed_four_columns,
    pin_zero_input,
    pin_zero_weight,
    pin_constant_row,
    pin_scale_invariance,
    pin_backward_two_columns,
    pin_dx_orthogonal_to_x,
    pin_dy_equal_y,
    pin_single_row_dw,
    pin_dw_sums_rows,
    pin_finite_differences,
    pin_torch_rms_norm,
    pin_bf16_decoding,
    pin_f16_decoding,
    pin_mixed_weight_dtype,
    pin_row_selection,
    pin_nan_and_inf_rows,
    pin_rounding_matches_numpy,
    pin_bf16_rounding,
    pin_add_printed_example,
    pin_add_stored_sum,
    pin_add_finite_differences,
]
