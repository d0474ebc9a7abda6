"""Builds librmsnorm.so in-tree from csrc/*.cu for sm_103a (GB300).

Each translation unit is compiled by its own nvcc process (in parallel), then
linked into ``_build/librmsnorm.so`` against the shared CUDA runtime, so the
library and PyTorch share one runtime state. A rebuild happens only when a
source or header is newer than the library.

A second, checked variant of the same sources (``-DRMSNORM_CHECKS``, in
``_build_checked/``) tests every global store, bulk copy and shared-memory
ring access of the kernels against the extent it belongs to and reports a
failed check as RMSNORM_ERR_OUT_OF_BOUNDS instead of making the access. It is
a debug build for the tests; the binding loads it only when
RMSNORM_LIBRARY_VARIANT=checked is set.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
CHECKED_BUILD_DIR = os.path.join(PKG_DIR, "_build_checked")
LIB_NAME = "librmsnorm.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
CHECKED_LIB_PATH = os.path.join(CHECKED_BUILD_DIR, LIB_NAME)

SOURCES = ["api.cu", "fwd.cu", "bwd.cu", "bwd_f32.cu", "bwd_bf16.cu", "bwd_f16.cu",
           "bwd_res_f32.cu", "bwd_res_bf16.cu", "bwd_res_f16.cu", "naive.cu", "probe.cu",
           "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    path = shutil.which("nvcc")
    if path:
        return path
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librmsnorm.so")


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC))
             if f.endswith((".cu", ".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "rmsnorm.h"))
    files.append(os.path.abspath(__file__))
    return files


def source_hash() -> str:
    """sha256 over the sources the library is built from (for run records)."""
    h = hashlib.sha256()
    for f in _inputs():
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


BWD_KERNEL_FILES = ("bwd.cu", "bwd_kernels.cuh", "bwd_f32.cu", "bwd_bf16.cu", "bwd_f16.cu",
                    "bwd_res_f32.cu", "bwd_res_bf16.cu", "bwd_res_f16.cu", "common.cuh",
                    "kernels.h")


FWD_KERNEL_FILES = ("fwd.cu", "common.cuh", "kernels.h")


def kernel_source_hash(names=BWD_KERNEL_FILES) -> str:
    """sha256 over the csrc files that define a kernel family (by default the
    backward), so a profile can be matched to the kernel code it measured."""
    h = hashlib.sha256()
    for n in names:
        h.update(n.encode())
        with open(os.path.join(CSRC, n), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def lib_path(checked: bool = False) -> str:
    return CHECKED_LIB_PATH if checked else LIB_PATH


def is_stale(checked: bool = False) -> bool:
    path = lib_path(checked)
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _run(cmd: list[str], log: str | None) -> None:
    res = subprocess.run(cmd, capture_output=True, text=True)
    out = (res.stdout or "") + (res.stderr or "")
    if log:
        with open(log, "w") as fh:
            fh.write(" ".join(cmd) + "\n" + out)
    if res.returncode != 0:
        raise RuntimeError(f"command failed ({res.returncode}): {' '.join(cmd)}\n{out}")


def _variant_jobs(checked: bool, extra: list[str]):
    """(compile commands, objects, link step) of one variant."""
    nvcc = _nvcc()
    out_dir = CHECKED_BUILD_DIR if checked else BUILD_DIR
    os.makedirs(out_dir, exist_ok=True)
    defs = ["-DRMSNORM_CHECKS"] if checked else []
    objs, cmds = [], []
    for src in SOURCES:
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        log = os.path.join(out_dir, src.replace(".cu", ".log"))
        cmds.append(([nvcc, *ARCH, *FLAGS, *defs, *extra, "-c", os.path.join(CSRC, src), "-o",
                      obj], log))
    return cmds, objs, out_dir


def _link(objs: list[str], checked: bool) -> None:
    path = lib_path(checked)
    tmp = path + f".tmp{os.getpid()}"
    _run([_nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs], None)
    os.replace(tmp, path)
    with open(os.path.join(os.path.dirname(path), "BUILD_INFO"), "w") as fh:
        fh.write(f"source_hash={source_hash()}\nnvcc={_nvcc()}\narch=sm_103a\n"
                 f"checked={int(checked)}\n")


def build(force: bool = False, ptxas_verbose: bool = False, jobs: int | None = None,
          checked: bool = False, both: bool = False) -> str:
    """Compile and link the library if needed; returns its path. `checked`
    builds the checked debug variant instead; `both` builds the library and
    the checked variant together (one pool of compile jobs) and returns the
    library's path."""
    variants = [False, True] if both else [checked]
    todo = [v for v in variants if force or is_stale(v)]
    if not todo:
        return lib_path(checked and not both)
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    plans = {v: _variant_jobs(v, extra) for v in todo}
    cmds = [c for v in todo for c in plans[v][0]]
    workers = jobs or min(len(cmds), max(1, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        for fut in [ex.submit(_run, c, log) for c, log in cmds]:
            fut.result()
    for v in todo:
        _link(plans[v][1], v)
    return lib_path(checked and not both)


if __name__ == "__main__":
    path = build(force="--force" in sys.argv, ptxas_verbose="-v" in sys.argv,
                 checked="--checked" in sys.argv, both="--both" in sys.argv)
    print(path)
