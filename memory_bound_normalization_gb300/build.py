"""Builds librmsnorm.so in-tree from csrc/*.cu for sm_103a (GB300).

Each translation unit is compiled by its own nvcc process (in parallel), then
linked into ``_build/librmsnorm.so`` against the shared CUDA runtime, so the
library and PyTorch share one runtime state. A rebuild happens only when a
source or header is newer than the library.
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
LIB_NAME = "librmsnorm.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)

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


def kernel_source_hash(names=BWD_KERNEL_FILES) -> str:
    """sha256 over the csrc files that define a kernel family (by default the
    backward), so a profile can be matched to the kernel code it measured."""
    h = hashlib.sha256()
    for n in names:
        h.update(n.encode())
        with open(os.path.join(CSRC, n), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _run(cmd: list[str], log: str | None) -> None:
    res = subprocess.run(cmd, capture_output=True, text=True)
    out = (res.stdout or "") + (res.stderr or "")
    if log:
        with open(log, "w") as fh:
            fh.write(" ".join(cmd) + "\n" + out)
    if res.returncode != 0:
        raise RuntimeError(f"command failed ({res.returncode}): {' '.join(cmd)}\n{out}")


def build(force: bool = False, ptxas_verbose: bool = False, jobs: int | None = None) -> str:
    """Compile and link the library if needed; returns its path."""
    if not force and not is_stale():
        return LIB_PATH
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    objs = []
    cmds = []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        log = os.path.join(BUILD_DIR, src.replace(".cu", ".log"))
        cmds.append(([nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj], log))
    workers = jobs or min(len(cmds), max(1, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        for fut in [ex.submit(_run, c, log) for c, log in cmds]:
            fut.result()
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    _run([nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs], None)
    os.replace(tmp, LIB_PATH)
    with open(os.path.join(BUILD_DIR, "BUILD_INFO"), "w") as fh:
        fh.write(f"source_hash={source_hash()}\nnvcc={nvcc}\narch=sm_103a\n")
    return LIB_PATH


if __name__ == "__main__":
    path = build(force="--force" in sys.argv, ptxas_verbose="-v" in sys.argv)
    print(path)
