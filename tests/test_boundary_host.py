"""The C-ABI library without a GPU: it loads, exports every symbol the header
declares, rejects bad arguments before touching CUDA, and its width ladder
makes consistent choices. No kernel is launched here."""
from __future__ import annotations

import ctypes
import json
import math
import os
import re
import subprocess
import sys

import pytest

import memory_bound_normalization_gb300 as pkg
from memory_bound_normalization_gb300 import build as libbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "rmsnorm.h")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return pkg.load_library()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"\b(rmsnorm_[a-z0-9_]+)\s*\(", text)


def test_header_and_exports_agree(lib):
    names = header_functions()
    assert names == list(pkg.EXPORTS)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in rmsnorm.h but not exported"


def test_exports_are_c_symbols(lib):
    # extern "C": plain names, callable through ctypes without mangling
    for n in pkg.EXPORTS:
        ctypes.cast(getattr(lib, n), ctypes.c_void_p)


def test_status_strings(lib):
    for code in range(8):
        s = pkg.rmsnorm_status_string(code)
        assert s.startswith("RMSNORM_") and "UNKNOWN" not in s
    assert "UNKNOWN" in pkg.rmsnorm_status_string(99)
    assert pkg.rmsnorm_version().count(".") == 2


FAKE = 1 << 20  # aligned non-null addresses; never dereferenced by these calls


def test_argument_checks_need_no_device(lib):
    B, F = pkg.BF16, pkg.F32
    fwd = pkg.rmsnorm_fwd
    # M == 0: nothing to do
    assert fwd(FAKE, FAKE, FAKE, FAKE, 0, 64, 1e-6, B, 0) == pkg.OK
    # shape, dtype and eps
    assert fwd(FAKE, FAKE, FAKE, FAKE, 4, 0, 1e-6, B, 0) == pkg.ERR_INVALID_ARG
    assert fwd(FAKE, FAKE, FAKE, FAKE, -1, 64, 1e-6, B, 0) == pkg.ERR_INVALID_ARG
    assert fwd(FAKE, FAKE, FAKE, FAKE, 4, 1 << 31, 1e-6, B, 0) == pkg.ERR_INVALID_ARG
    assert fwd(FAKE, FAKE, FAKE, FAKE, 4, 64, 1e-6, 5, 0) == pkg.ERR_INVALID_ARG
    assert fwd(FAKE, FAKE, FAKE, FAKE, 4, 64, -1e-6, B, 0) == pkg.ERR_INVALID_ARG
    assert fwd(FAKE, FAKE, FAKE, FAKE, 4, 64, math.nan, B, 0) == pkg.ERR_INVALID_ARG
    # null tensors
    assert fwd(None, FAKE, FAKE, FAKE, 4, 64, 1e-6, B, 0) == pkg.ERR_INVALID_ARG
    assert fwd(FAKE, FAKE, FAKE, None, 4, 64, 1e-6, B, 0) == pkg.ERR_INVALID_ARG
    for code in (-1, 5, 6):
        assert fwd(FAKE, FAKE, FAKE, FAKE, 4, 64, 1e-6, code, 0) == pkg.ERR_INVALID_ARG
    # misaligned element or fp32 pointers; an fp32 weight must be 4-byte
    # aligned even with 16-bit activations
    for code in (pkg.F16, pkg.BF16_W_F32, pkg.F16_W_F32):
        assert fwd(FAKE + 1, FAKE, FAKE, FAKE, 4, 64, 1e-6, code, 0) == pkg.ERR_MISALIGNED
    for code in (pkg.BF16_W_F32, pkg.F16_W_F32):
        assert fwd(FAKE, FAKE + 2, FAKE, FAKE, 4, 64, 1e-6, code, 0) == pkg.ERR_MISALIGNED
        assert pkg.rmsnorm_bwd(FAKE, FAKE + 2, FAKE, FAKE, FAKE, FAKE, 4, 64, code, 0) == \
            pkg.ERR_MISALIGNED
    assert fwd(FAKE + 1, FAKE, FAKE, FAKE, 4, 64, 1e-6, B, 0) == pkg.ERR_MISALIGNED
    assert fwd(FAKE + 2, FAKE, FAKE, FAKE, 4, 64, 1e-6, F, 0) == pkg.ERR_MISALIGNED
    assert fwd(FAKE, FAKE, FAKE, FAKE + 2, 4, 64, 1e-6, B, 0) == pkg.ERR_MISALIGNED

    bwd = pkg.rmsnorm_bwd
    assert bwd(FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, 64, B, 0) == pkg.OK
    assert bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 0, B, 0) == pkg.ERR_INVALID_ARG
    assert bwd(FAKE, FAKE, None, FAKE, FAKE, FAKE, 4, 64, B, 0) == pkg.ERR_INVALID_ARG
    assert bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 2, 4, 64, B, 0) == pkg.ERR_MISALIGNED
    assert bwd(FAKE, FAKE, FAKE, FAKE + 1, FAKE, FAKE, 4, 64, B, 0) == pkg.ERR_MISALIGNED
    ws = pkg.rmsnorm_bwd_ws
    assert ws(FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, 64, B, None, 0, 0) == pkg.OK
    assert ws(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 64, 7, FAKE, 1 << 20, 0) == \
        pkg.ERR_INVALID_ARG
    assert pkg.rmsnorm_bwd_workspace_size(0, 64, B, 0) == 0
    assert pkg.rmsnorm_bwd_workspace_size(4, 0, B, 0) == 0
    # the no-alloc backward takes fp32 and bf16 only
    for code in (pkg.F16, pkg.BF16_W_F32, pkg.F16_W_F32):
        assert pkg.rmsnorm_bwd_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 64, code, 0) == \
            pkg.ERR_INVALID_ARG

    # residual add: the same checks, plus the residual, h and dres
    afwd, abwd = pkg.rmsnorm_add_fwd, pkg.rmsnorm_add_bwd
    assert afwd(FAKE, None, FAKE, None, FAKE, FAKE, 0, 64, 1e-6, B, 0) == pkg.OK
    assert afwd(FAKE, None, FAKE, FAKE, FAKE, FAKE, 4, 64, 1e-6, B, 0) == pkg.ERR_INVALID_ARG
    assert afwd(FAKE, FAKE, FAKE, None, FAKE, FAKE, 4, 64, 1e-6, B, 0) == pkg.ERR_INVALID_ARG
    assert afwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 64, 1e-6, 5, 0) == pkg.ERR_INVALID_ARG
    assert afwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 64, -1.0, B, 0) == pkg.ERR_INVALID_ARG
    assert afwd(FAKE, FAKE + 1, FAKE, FAKE, FAKE, FAKE, 4, 64, 1e-6, B, 0) == pkg.ERR_MISALIGNED
    assert afwd(FAKE, FAKE, FAKE, FAKE + 2, FAKE, FAKE, 4, 64, 1e-6, F, 0) == pkg.ERR_MISALIGNED
    assert abwd(FAKE, FAKE, FAKE, FAKE, None, FAKE, None, 0, 64, B, 0) == pkg.OK
    assert abwd(FAKE, FAKE, FAKE, FAKE, FAKE + 1, FAKE, FAKE, 4, 64, B, 0) == pkg.ERR_MISALIGNED
    assert abwd(FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, 4, 64, B, 0) == pkg.ERR_INVALID_ARG

    # the naive backward: vector rows of at most 1024 vectors only
    nv = pkg.rmsnorm_bwd_naive
    assert nv(FAKE, FAKE, FAKE, FAKE, None, 0, 64, 1e-6, B, 0) == pkg.OK
    assert nv(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 64, -1.0, B, 0) == pkg.ERR_INVALID_ARG
    assert nv(FAKE, FAKE, None, FAKE, FAKE, 4, 64, 1e-6, B, 0) == pkg.ERR_INVALID_ARG
    assert nv(FAKE + 2, FAKE, FAKE, FAKE, FAKE, 4, 64, 1e-6, B, 0) == pkg.ERR_UNSUPPORTED
    assert nv(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 8200, 1e-6, B, 0) == pkg.ERR_UNSUPPORTED
    assert nv(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 4100, 1e-6, F, 0) == pkg.ERR_UNSUPPORTED
    assert nv(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 13, 1e-6, B, 0) == pkg.ERR_UNSUPPORTED
    assert nv(FAKE + 1, FAKE, FAKE, FAKE, FAKE, 4, 64, 1e-6, B, 0) == pkg.ERR_MISALIGNED

    probe = pkg.rmsnorm_probe
    assert probe(7, FAKE, FAKE, FAKE, 1024, 1, 0) == pkg.ERR_INVALID_ARG
    assert probe(pkg.PROBE_COPY, FAKE, FAKE, None, 1000, 1, 0) == pkg.ERR_INVALID_ARG
    assert probe(pkg.PROBE_COPY, FAKE, None, None, 1024, 1, 0) == pkg.ERR_INVALID_ARG
    assert probe(pkg.PROBE_2R1W, FAKE, FAKE, None, 1024, 1, 0) == pkg.ERR_INVALID_ARG
    assert probe(pkg.PROBE_WRITE, FAKE, None, None, 1024, 0, 0) == pkg.ERR_INVALID_ARG
    assert probe(pkg.PROBE_WRITE, FAKE + 8, None, None, 1024, 1, 0) == pkg.ERR_MISALIGNED
    assert probe(pkg.PROBE_WRITE, FAKE, None, None, 0, 1, 0) == pkg.OK

    # test hooks are plain setters
    pkg.rmsnorm_set_wait_limit_ns(0)
    pkg.rmsnorm_test_drop_copy(-1)


WIDTHS = sorted({1, 2, 3, 4, 7, 8, 13, 16, 24, 32, 40, 64, 96, 100, 128, 200, 256, 257, 512,
                 768, 1000, 1024, 1536, 2048, 2049, 2880, 3072, 4096, 5120, 6144, 8192, 12288,
                 16384, 24576, 32768, 49152, 65536, 131072, 262144, 300000, 524288, 1 << 20})


DTYPES = [pkg.BF16, pkg.F32, pkg.F16, pkg.BF16_W_F32, pkg.F16_W_F32]
DTYPE_IDS = ["bf16", "f32", "f16", "bf16_wf32", "f16_wf32"]


@pytest.mark.parametrize("dtype", DTYPES, ids=DTYPE_IDS)
@pytest.mark.parametrize("N", WIDTHS)
def test_width_ladder(lib, N, dtype):
    """Every width maps to one kernel family whose slots cover the row, with
    legal block, cluster and shared-memory sizes."""
    vec = 4 if dtype == pkg.F32 else 8  # elements per 16-byte activation vector
    mixed = dtype in (pkg.BF16_W_F32, pkg.F16_W_F32)
    vector_ok = (N * (16 // vec)) % 16 == 0
    for pass_ in (pkg.PASS_FWD, pkg.PASS_FWD_ADD, pkg.PASS_BWD, pkg.PASS_BWD_RES):
        p = pkg.rmsnorm_plan(1000, N, dtype, pass_, -1)
        assert p.grid == 0  # no device queried
        assert p.threads % 32 == 0 and 32 <= p.threads <= 1024
        # clusters of 16 (a non-portable size) only for backward rows that 8
        # blocks cannot hold
        assert 1 <= p.cluster <= 8 or (p.cluster == 16 and pass_ in (pkg.PASS_BWD, pkg.PASS_BWD_RES))
        assert p.smem_bytes <= 227 * 1024
        name = pkg.VARIANTS[p.variant]
        if not vector_ok:
            assert name == "scalar"
            continue
        if name == "rowgroup":
            assert p.threads_per_row in (4, 8, 16, 32)
            assert p.threads_per_row * p.vectors_per_thread * vec >= N
            assert p.rows_per_unit % (p.threads // p.threads_per_row) == 0
        elif name in ("cta_row", "cluster_row"):
            assert (name == "cluster_row") == (p.cluster > 1)
            assert p.threads % p.row_groups == 0 and (p.threads // p.row_groups) % 32 == 0
            tg = p.threads // p.row_groups
            assert tg * p.vectors_per_thread * p.cluster * vec >= N
            assert p.threads_per_row == tg * p.cluster
            assert 1 <= p.row_groups <= 8 and p.threads <= 512 if p.row_groups > 1 else True
            if mixed and pass_ == pkg.PASS_FWD:
                assert p.threads <= 512  # the fp32-weight row kernel's launch bound
        elif name == "two_pass":
            assert pass_ in (pkg.PASS_FWD, pkg.PASS_FWD_ADD) and N > 512 * 4 * vec
        elif name == "ring":
            # persistent forward: a cluster of blocks whose slices cover the row,
            # at least three stages of the ring (x, and the residual with ADD)
            assert pass_ in (pkg.PASS_FWD, pkg.PASS_FWD_ADD)
            assert p.vectors_per_thread in (4, 8) and p.threads <= 512
            assert p.threads * p.vectors_per_thread * p.cluster * vec >= N
            assert 3 <= p.stages <= 6
            nt = 2 if pass_ == pkg.PASS_FWD_ADD else 1
            assert p.smem_bytes >= nt * p.stages * p.vectors_per_thread * p.threads * 16
        else:
            # the backward's vector kernels cover every row up to 512 KiB
            # (clusters of 16 past 256 KiB); wider rows outgrow shared memory
            assert name == "scalar" and pass_ in (pkg.PASS_BWD, pkg.PASS_BWD_RES)
            assert N * (16 // vec) > 512 * 1024
        if pass_ in (pkg.PASS_BWD, pkg.PASS_BWD_RES) and name != "scalar":
            # the residual backward's rings carry dres too and may be 2 deep, as
            # may an fp32 row over a cluster of 5 blocks of 8 vectors a thread
            res = pass_ == pkg.PASS_BWD_RES
            two_deep = res or (dtype == pkg.F32 and p.cluster in (5, 16) and
                               p.vectors_per_thread == 8)
            assert (2 if two_deep else 3) <= p.stages <= 6
            if name == "rowgroup":
                unit = p.rows_per_unit * N * (16 // vec)
            else:
                unit = p.vectors_per_thread * (p.threads // p.row_groups) * 16 * p.row_groups
            assert p.smem_bytes >= (3 if res else 2) * p.stages * unit


@pytest.mark.parametrize("dtype", [pkg.BF16, pkg.F16, pkg.BF16_W_F32, pkg.F16_W_F32],
                         ids=["bf16", "f16", "bf16_wf32", "f16_wf32"])
def test_ring_forward_16bit_slice_width(lib, dtype):
    """16-bit ring slices take 8 vectors a thread, re-read from their stage,
    in one block of 256-384 threads for rows of 2048-3072 vectors (N = 16384
    to 24576) and past 8192 vectors (clusters of 4 blocks at N = 98304 and
    131072, 8 at 262144); 4 vectors elsewhere (one block of up to 448 threads
    below 2048 vectors, clusters from 24584 to 65536). The residual forward,
    whose two tensors do not fit its stages at 8 vectors, keeps 4."""
    for N, cluster, v, threads in ((12288, 1, 4, 384), (14336, 1, 4, 448), (16384, 1, 8, 256),
                                   (20480, 1, 8, 320), (24576, 1, 8, 384), (24584, 2, 4, 416),
                                   (32768, 2, 4, 512), (65536, 4, 4, 512), (98304, 4, 8, 384),
                                   (131072, 4, 8, 512), (262144, 8, 8, 512)):
        p = pkg.rmsnorm_plan(1000, N, dtype, pkg.PASS_FWD, -1)
        assert pkg.VARIANTS[p.variant] == "ring"
        assert (p.cluster, p.vectors_per_thread, p.threads) == (cluster, v, threads)
        assert p.stages >= 3 and p.smem_bytes <= 227 * 1024
    for N in (98304, 131072):
        a = pkg.rmsnorm_plan(1000, N, dtype, pkg.PASS_FWD_ADD, -1)
        assert pkg.VARIANTS[a.variant] == "ring" and a.vectors_per_thread == 4 and a.cluster == 8
    for N in (16384, 24576):
        a = pkg.rmsnorm_plan(1000, N, dtype, pkg.PASS_FWD_ADD, -1)
        assert pkg.VARIANTS[a.variant] == "ring" and a.vectors_per_thread == 4
    assert pkg.VARIANTS[pkg.rmsnorm_plan(1000, 524288, dtype, pkg.PASS_FWD, -1).variant] == "two_pass"


def _child_plans(env: dict, shapes) -> list:
    """Forward plans of (N, dtype code) pairs in a child process with extra
    environment variables (the tuning knobs are read once per process)."""
    code = ("import json, sys, memory_bound_normalization_gb300 as p; p.load_library(); "
            "out = [p.rmsnorm_plan(1000, n, d, p.PASS_FWD, -1).as_dict() for n, d in "
            "json.loads(sys.argv[1])]; print(json.dumps(out))")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    res = subprocess.run([sys.executable, "-c", code, json.dumps(shapes)], cwd=root,
                         env={**os.environ, **env}, capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stderr[-2000:]
    return json.loads(res.stdout.strip().splitlines()[-1])


def test_ring16_knob(lib):
    """RMSNORM_FWD_RING16_V=4 restores 4-vector 16-bit ring slices everywhere
    (one block of 512 threads at N = 16384, clusters of 2 at 20480, of 8 at
    131072); =8 keeps the width rule's plans."""
    shapes = [[16384, pkg.BF16], [20480, pkg.F16], [131072, pkg.BF16]]
    four = _child_plans({"RMSNORM_FWD_RING16_V": "4"}, shapes)
    assert [(p["cluster"], p["vectors_per_thread"], p["threads"]) for p in four] == \
        [(1, 4, 512), (2, 4, 320), (8, 4, 512)]
    eight = _child_plans({"RMSNORM_FWD_RING16_V": "8"}, shapes)
    assert [(p["cluster"], p["vectors_per_thread"], p["threads"]) for p in eight] == \
        [(1, 8, 256), (1, 8, 320), (4, 8, 512)]
    assert all(p["variant_name"] == "ring" for p in four + eight)


def test_ring_forward_fp32_past_clusters(lib):
    """fp32 rows too wide for a cluster of blocks holding the row take the
    ring at 8 vectors a thread up to 32768 vectors (N = 131072); the residual
    forward and wider rows take the two-pass kernel."""
    for N, threads in ((98304, 384), (131072, 512)):
        p = pkg.rmsnorm_plan(1000, N, pkg.F32, pkg.PASS_FWD, -1)
        assert pkg.VARIANTS[p.variant] == "ring"
        assert (p.cluster, p.vectors_per_thread, p.threads) == (8, 8, threads)
        a = pkg.rmsnorm_plan(1000, N, pkg.F32, pkg.PASS_FWD_ADD, -1)
        assert pkg.VARIANTS[a.variant] == "two_pass"
    assert pkg.VARIANTS[pkg.rmsnorm_plan(1000, 196608, pkg.F32, pkg.PASS_FWD, -1).variant] == "two_pass"


@pytest.mark.parametrize("dtype,N,threads,stages", [
    (pkg.BF16, 196608, 384, 4), (pkg.BF16, 262144, 512, 3), (pkg.F16_W_F32, 262144, 512, 3),
    (pkg.F32, 98304, 384, 4), (pkg.F32, 131072, 512, 3)])
def test_backward_cluster_of_16(lib, dtype, N, threads, stages):
    """Rows of 256..512 KiB, which no cluster of 8 holds with a three-deep
    ring, split over 16 blocks of 4 vectors a thread (the residual backward
    with a two-deep ring); wider rows stay scalar."""
    p = pkg.rmsnorm_plan(1000, N, dtype, pkg.PASS_BWD, -1)
    assert pkg.VARIANTS[p.variant] == "cluster_row"
    assert (p.cluster, p.vectors_per_thread, p.threads, p.stages) == (16, 4, threads, stages)
    r = pkg.rmsnorm_plan(1000, N, dtype, pkg.PASS_BWD_RES, -1)
    assert pkg.VARIANTS[r.variant] == "cluster_row" and (r.cluster, r.stages) == (16, 2)
    wider = pkg.rmsnorm_plan(1000, 2 * 262144, dtype, pkg.PASS_BWD, -1)
    assert pkg.VARIANTS[wider.variant] == "scalar"


def test_backward_fp32_cluster_of_16_two_deep(lib):
    """fp32 rows past 131072, up to 229376, take 16 blocks of 8 vectors a thread
    with a two-deep ring (the residual backward, a third tensor, does not fit
    and stays scalar); wider rows stay scalar."""
    for N, threads in ((163840, 320), (196608, 384), (229376, 448)):
        p = pkg.rmsnorm_plan(1000, N, pkg.F32, pkg.PASS_BWD, -1)
        assert pkg.VARIANTS[p.variant] == "cluster_row"
        assert (p.cluster, p.vectors_per_thread, p.threads, p.stages) == (16, 8, threads, 2)
        assert p.smem_bytes <= 227 * 1024
        r = pkg.rmsnorm_plan(1000, N, pkg.F32, pkg.PASS_BWD_RES, -1)
        assert pkg.VARIANTS[r.variant] == "scalar"
    assert pkg.VARIANTS[pkg.rmsnorm_plan(1000, 262144, pkg.F32, pkg.PASS_BWD, -1).variant] == "scalar"


def test_plan_rejects_bad_arguments(lib):
    with pytest.raises(pkg.RMSNormError):
        pkg.rmsnorm_plan(10, 0, pkg.BF16, pkg.PASS_FWD)
    with pytest.raises(pkg.RMSNormError):
        pkg.rmsnorm_plan(10, 64, pkg.BF16, 7)
    p = pkg.rmsnorm_plan(0, 64, pkg.BF16, pkg.PASS_BWD)
    assert pkg.VARIANTS[p.variant] == "none"


@pytest.mark.parametrize("dtype,N,want", [(pkg.BF16, 1024, "rowgroup"), (pkg.BF16, 1032, "cta_row"),
                                          (pkg.BF16, 2048, "cta_row"), (pkg.F16, 2048, "cta_row"),
                                          (pkg.BF16_W_F32, 1536, "cta_row"),
                                          (pkg.F32, 1024, "rowgroup"), (pkg.F32, 1028, "cta_row")])
def test_short_row_backward_cutoff(lib, dtype, N, want):
    """The backward keeps the row-group kernel up to 128 vectors a row for
    16-bit activations and up to 256 for fp32 (the faster side of each
    measured pair); both passes of the backward follow the same cutoff."""
    for pass_ in (pkg.PASS_BWD, pkg.PASS_BWD_RES):
        p = pkg.rmsnorm_plan(1000, N, dtype, pass_, -1)
        assert pkg.VARIANTS[p.variant] == want


@pytest.mark.parametrize("dtype,N", [(pkg.BF16, 1032), (pkg.BF16, 2048), (pkg.F16, 1536),
                                     (pkg.BF16_W_F32, 2048), (pkg.F32, 1024)])
def test_residual_forward_short_row_cutoff(lib, dtype, N):
    """Rows of 129..256 vectors: the plain forward keeps the short-row kernel,
    the residual forward takes a block per row."""
    plain = pkg.rmsnorm_plan(1000, N, dtype, pkg.PASS_FWD, -1)
    add = pkg.rmsnorm_plan(1000, N, dtype, pkg.PASS_FWD_ADD, -1)
    assert pkg.VARIANTS[plain.variant] == "rowgroup"
    assert pkg.VARIANTS[add.variant] == "cta_row" and add.vectors_per_thread == 4
    vec = 4 if dtype == pkg.F32 else 8
    assert add.threads * 4 * vec >= N


@pytest.mark.parametrize("dtype,N,cluster,vectors,stages", [
    (pkg.F32, 32768, 4, 4, 3), (pkg.F32, 40960, 5, 4, 3), (pkg.F32, 49152, 6, 4, 3),
    (pkg.F32, 65536, 5, 8, 2), (pkg.BF16, 65536, 4, 4, 3), (pkg.BF16, 98304, 6, 4, 3),
    (pkg.BF16, 131072, 8, 4, 3), (pkg.F16, 131072, 8, 4, 3)])
def test_wide_backward_cluster_sizes(lib, dtype, N, cluster, vectors, stages):
    """Rows the power-of-two ladder would split over 8 blocks take 5 or 6
    where 4 vectors a thread and a three-deep ring fit (fp32 also 5 blocks of
    8 vectors with a two-deep ring); 16-bit rows otherwise keep 8."""
    p = pkg.rmsnorm_plan(1000, N, dtype, pkg.PASS_BWD, -1)
    assert pkg.VARIANTS[p.variant] == "cluster_row"
    assert (p.cluster, p.vectors_per_thread, p.stages) == (cluster, vectors, stages)
    vec = 4 if dtype == pkg.F32 else 8
    assert p.threads * vectors * cluster * vec >= N and p.threads <= 512
    # the residual backward keeps the power-of-two ladder
    r = pkg.rmsnorm_plan(1000, N, dtype, pkg.PASS_BWD_RES, -1)
    assert r.cluster in (1, 2, 4, 8)
