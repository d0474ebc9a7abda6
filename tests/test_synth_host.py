"""The seeded input generators on the CPU: the recipe's readings (exact
outlier count, ×100 at distinct positions, the weight distribution, rounding
into the working dtype), determinism, and the logical byte counts the bench
divides by."""
from __future__ import annotations

import dataclasses

import torch

from memory_bound_normalization_gb300 import synth


def test_outliers_are_exact_count_at_distinct_positions():
    wl = dataclasses.replace(synth.WORKLOADS["hidden8192_32768x8192_outliers"], M=64, N=1000,
                             dtype=torch.float32)
    plain = dataclasses.replace(wl, outlier_frac=0.0)
    a = synth.make_inputs(wl, device="cpu")["x"]
    b = synth.make_inputs(plain, device="cpu")["x"]
    changed = (a != b).view(-1)
    k = synth.outlier_count(wl)
    assert k == round(1e-3 * 64 * 1000) == 64
    assert int(changed.sum()) == k  # distinct positions, every one scaled
    assert torch.equal(a.view(-1)[changed], b.view(-1)[changed] * 100.0)


def test_same_seeds_same_tensors_and_dtype_rounding():
    wl = dataclasses.replace(synth.WORKLOADS["small_256x1024"], M=8)
    a = synth.make_inputs(wl, device="cpu")
    b = synth.make_inputs(wl, device="cpu")
    for k in ("x", "w", "dy"):
        assert a[k].dtype == torch.bfloat16 and torch.equal(a[k], b[k])
    # the bf16 tensors are the fp32 draws rounded once to nearest even
    wl32 = dataclasses.replace(wl, dtype=torch.float32)
    c = synth.make_inputs(wl32, device="cpu")
    assert torch.equal(a["x"], c["x"].to(torch.bfloat16))
    assert torch.equal(a["w"], c["w"].to(torch.bfloat16))


def test_weight_distribution_and_dy_scale():
    wl = dataclasses.replace(synth.WORKLOADS["hidden4096_16384x4096"], M=256,
                             dtype=torch.float32)
    inp = synth.make_inputs(wl, device="cpu")
    w = inp["w"].double()
    assert abs(w.mean().item() - 1.0) < 0.01 and abs(w.std().item() - 0.1) < 0.01
    dy = inp["dy"].double()
    assert abs(dy.std().item() - 1e-2) < 1e-3  # N(0,1) * 1e-2
    mixed = synth.make_inputs(synth.WORKLOADS["hidden4096_16384x4096_bf16_wf32"], device="cpu",
                              M=4)
    assert mixed["w"].dtype == torch.float32 and mixed["x"].dtype == torch.bfloat16


def test_logical_bytes_match_the_published_count():
    """32768 x 8192 bf16: the backward moves 1536.2 MiB (x, dy read, dx
    written, w and rstd read, dw written)."""
    fwd, bwd = synth.logical_bytes(32768, 8192, 2)
    assert bwd == 1_610_792_960 and round(bwd / 2**20, 1) == 1536.2
    assert fwd == 2 * 32768 * 8192 * 2 + 8192 * 2 + 4 * 32768
    f2, b2 = synth.logical_bytes(16384, 4096, 2, 4)  # fp32 weight
    assert f2 - synth.logical_bytes(16384, 4096, 2)[0] == 4096 * 2
    assert b2 - synth.logical_bytes(16384, 4096, 2)[1] == 4096 * 2


def test_sweep_rows_follow_the_reading():
    sweep = synth.width_sweep(torch.bfloat16)
    assert [w.N for w in sweep] == [256, 768, 2880, 6144, 16384, 65536]
    assert all(w.M == (1 << 27) // w.N for w in sweep)
