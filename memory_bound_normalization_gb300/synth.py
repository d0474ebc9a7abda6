"""Seeded synthetic inputs for the RMSNorm workloads.

Draws random numbers and nothing else: no RMSNorm arithmetic lives here. The
tests, the benchmark and the smoke check use it to feed both the CUDA library
and the CPU oracle the same arrays.

Recipe (all values drawn in fp32 from a seeded torch.Generator on the target
device, then rounded to nearest-even into the working dtype):
  x  ~ N(0, 1); optionally a fraction of entries, chosen as exactly
       round(frac * M * N) distinct positions, multiplied by 100 (outliers);
  dy ~ N(0, 1) * dy_scale;
  w  = 1 + 0.1 * N(0, 1), rounded into the weight dtype (the working dtype
       unless the workload names another, e.g. an fp32 master weight).
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    dtype: torch.dtype
    eps: float
    seed_x: int
    seed_dy: int
    seed_w: int
    dy_scale: float = 1.0
    outlier_frac: float = 0.0
    seed_outliers: int = 0
    about: str = ""
    w_dtype: torch.dtype | None = None  # None: the working dtype

    @property
    def weight_dtype(self) -> torch.dtype:
        return self.dtype if self.w_dtype is None else self.w_dtype

    @property
    def dtype_name(self) -> str:
        names = {torch.bfloat16: "bf16", torch.float32: "f32", torch.float16: "f16"}
        name = names[self.dtype]
        if self.weight_dtype != self.dtype:
            name += "_w" + names[self.weight_dtype]
        return name


def width_sweep(dtype: torch.dtype) -> list[Workload]:
    """Fixed M*N = 2^27 elements over non-power-of-two and cluster-sized rows;
    M = floor(2^27 / N)."""
    out = []
    for k, n in enumerate((256, 768, 2880, 6144, 16384, 65536)):
        tag = "bf16" if dtype == torch.bfloat16 else "f32"
        out.append(Workload(f"sweep_{tag}_N{n}", (1 << 27) // n, n, dtype, 1e-5,
                            41 + k, 141 + k, 241 + k, about="width sweep, M*N ~ 2^27"))
    return out


SMALL = Workload("small_256x1024", 256, 1024, torch.bfloat16, 1e-6, 1, 2, 3,
                 about="256 x 1024 bf16, fits in L2")
HIDDEN_4096 = Workload("hidden4096_16384x4096", 16384, 4096, torch.bfloat16, 1e-6, 11, 12, 13,
                       dy_scale=1e-2, about="7B-class hidden size, 4 x 4096 tokens")
HIDDEN_4096_F16 = Workload("hidden4096_16384x4096_f16", 16384, 4096, torch.float16, 1e-6, 11, 12,
                           13, dy_scale=1e-2, about="hidden 4096 workload in fp16")
HIDDEN_4096_W_F32 = Workload("hidden4096_16384x4096_bf16_wf32", 16384, 4096, torch.bfloat16, 1e-6,
                             11, 12, 13, dy_scale=1e-2, w_dtype=torch.float32,
                             about="hidden 4096 workload, bf16 activations, fp32 weight")
HIDDEN_8192 = Workload("hidden8192_32768x8192_outliers", 32768, 8192, torch.bfloat16, 1e-6,
                       21, 22, 23, dy_scale=1e-2, outlier_frac=1e-3, seed_outliers=24,
                       about="70B-class hidden size, 0.1% of x scaled by 100")
QK_NORM = Workload("qknorm_1048576x128", 1048576, 128, torch.bfloat16, 1e-6, 31, 32, 33,
                   about="per-head QK norm: 8 x 4096 x 32 rows of head_dim 128")

WORKLOADS = {w.name: w for w in
             [SMALL, HIDDEN_4096, HIDDEN_4096_F16, HIDDEN_4096_W_F32, HIDDEN_8192, QK_NORM, *width_sweep(torch.bfloat16),
              *width_sweep(torch.float32)]}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_inputs(wl: Workload, device="cuda", M: int | None = None):
    """Returns dict(x=[M,N], w=[N], dy=[M,N]) in wl.dtype on `device`.
    M defaults to wl.M (a smaller M keeps the same recipe for the first rows'
    distribution, not the same values)."""
    M = wl.M if M is None else M
    N = wl.N
    x = torch.randn(M, N, generator=_gen(device, wl.seed_x), device=device, dtype=torch.float32)
    if wl.outlier_frac > 0 and M * N > 0:
        k = int(round(wl.outlier_frac * M * N))
        idx = torch.randperm(M * N, generator=_gen(device, wl.seed_outliers), device=device)[:k]
        x.view(-1)[idx] *= 100.0
    dy = torch.randn(M, N, generator=_gen(device, wl.seed_dy), device=device, dtype=torch.float32)
    if wl.dy_scale != 1.0:
        dy *= wl.dy_scale
    w = 1.0 + 0.1 * torch.randn(N, generator=_gen(device, wl.seed_w), device=device,
                                dtype=torch.float32)
    return {"x": x.to(wl.dtype), "w": w.to(wl.weight_dtype), "dy": dy.to(wl.dtype)}


def random_rows(wl: Workload, count: int, device="cuda", M: int | None = None,
                x=None, dy=None):
    """Inputs of `count` rows, for tests that need arbitrary shapes:
    same distributions as `wl`, N columns."""
    return make_inputs(dataclasses.replace(wl, M=count), device=device)


def logical_bytes(M: int, N: int, elem: int, w_elem: int | None = None) -> tuple[int, int]:
    """Bytes the method must move: forward = x read + y write + w read + rstd
    write; backward = x, dy read + dx write + w, rstd read + dw write.
    `elem` is the activation element size, `w_elem` the weight's (default
    `elem`)."""
    w_elem = elem if w_elem is None else w_elem
    fwd = 2 * M * N * elem + N * w_elem + 4 * M
    bwd = 3 * M * N * elem + N * w_elem + 4 * M + 4 * N
    return fwd, bwd


def outlier_count(wl: Workload, M: int | None = None) -> int:
    M = wl.M if M is None else M
    return int(round(wl.outlier_frac * M * wl.N)) if wl.outlier_frac > 0 else 0


assert math.isclose(logical_bytes(32768, 8192, 2)[1] / 2**20, 1536.2, abs_tol=0.05)
