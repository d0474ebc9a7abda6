"""Tolerances and comparison helpers for CUDA-vs-oracle parity tests.

bf16 (y, dx): elementwise |err| <= 1e-2*|ref| + 1e-3.
fp16 (y, dx): elementwise |err| <= 2^-10*|ref| + 1e-5*rms_row(ref) + 2^-24:
    one rounding to fp16 costs at most 2^-11 relative (half an ulp, normal
    range) plus 2^-25 absolute (subnormal range), applied to an fp32 result
    whose own error is ~1e-6 relative to the row's terms; the bound doubles
    the rounding terms and gives the fp32 error the fp32 margin below.
fp32 (y, dx): 1e-5 relative, read as a per-row normwise bound
    ||err||_2 <= 1e-5 * ||ref||_2 together with an elementwise bound
    |err| <= 1e-5*|ref| + 1e-5*rms_row(ref); elementwise relative error alone
    is unbounded where dx cancels (sum_j dx_j x_j = 0 at eps = 0).
rstd: relative 1e-5 (fp32 accumulation of the squares plus one rsqrt).
dw: relative L2 <= 1e-4 over the whole vector.
NaN must appear exactly where the oracle has NaN.
"""
from __future__ import annotations

import numpy as np
import torch


def to_np(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


def _nan_match(got, ref, what):
    gn, rn = np.isnan(got), np.isnan(ref)
    assert np.array_equal(gn, rn), f"{what}: NaN positions differ ({gn.sum()} vs {rn.sum()})"
    return ~rn


def check_rows(got, ref, dtype: torch.dtype, what: str) -> None:
    got, ref = to_np(got), np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    ok = _nan_match(got, ref, what)
    g, r = np.where(ok, got, 0.0), np.where(ok, ref, 0.0)
    err = np.abs(g - r)
    if dtype == torch.bfloat16:
        bound = 1e-2 * np.abs(r) + 1e-3
        bad = err > bound
        assert not bad.any(), (
            f"{what}: {bad.sum()} of {bad.size} elements out of bf16 tolerance; "
            f"worst err {err.max():.3g} at ref {r.flat[np.argmax(err - bound)]:.3g}")
    elif dtype == torch.float16:
        rms = np.sqrt(np.mean(r ** 2, axis=-1, keepdims=True))
        bound = 2.0 ** -10 * np.abs(r) + 1e-5 * rms + 2.0 ** -24
        bad = err > bound
        assert not bad.any(), (
            f"{what}: {bad.sum()} of {bad.size} elements out of fp16 tolerance; "
            f"worst err {err.max():.3g} at ref {r.flat[np.argmax(err - bound)]:.3g}")
    else:
        rms = np.sqrt(np.mean(r ** 2, axis=-1, keepdims=True))
        bound = 1e-5 * np.abs(r) + 1e-5 * rms
        bad = err > bound
        assert not bad.any(), (
            f"{what}: {bad.sum()} of {bad.size} elements out of fp32 tolerance; "
            f"worst err {err.max():.3g}")
        num = np.sqrt(np.sum(err ** 2, axis=-1))
        den = np.sqrt(np.sum(r ** 2, axis=-1))
        rel = np.where(den > 0, num / np.where(den > 0, den, 1.0), num)
        assert rel.max() <= 1e-5, f"{what}: per-row normwise error {rel.max():.3g} > 1e-5"


def check_rstd(got, ref, what: str = "rstd") -> None:
    got, ref = to_np(got), np.asarray(ref, dtype=np.float64)
    ok = _nan_match(got, ref, what)
    rel = np.abs(got[ok] - ref[ok]) / np.abs(ref[ok])
    assert rel.size == 0 or rel.max() <= 1e-5, f"{what}: relative error {rel.max():.3g}"


def check_dw(got, ref, what: str = "dw") -> None:
    got, ref = to_np(got), np.asarray(ref, dtype=np.float64)
    ok = _nan_match(got, ref, what)
    den = np.linalg.norm(ref[ok])
    num = np.linalg.norm(got[ok] - ref[ok])
    rel = num / den if den > 0 else num
    assert rel <= 1e-4, f"{what}: relative L2 error {rel:.3g} > 1e-4"
