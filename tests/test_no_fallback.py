"""The product path has no CPU fallback: without librmsnorm.so every entry
point raises, and no module of the package imports the oracle. Runs on the
CPU (no kernel is launched)."""
from __future__ import annotations

import os
import re
import subprocess
import sys

import memory_bound_normalization_gb300 as pkg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG_DIR = os.path.dirname(pkg.__file__)


def test_missing_library_raises():
    """In a fresh process whose library path points nowhere, the binding
    raises OSError from the first call instead of computing anything."""
    code = r"""
import sys
import memory_bound_normalization_gb300 as pkg
from memory_bound_normalization_gb300 import _lib, build
build.LIB_PATH = "/nonexistent/librmsnorm.so"
_lib._lib = None
calls = [
    lambda: pkg.rmsnorm_fwd(1 << 20, 1 << 20, 1 << 20, 1 << 20, 4, 64, 1e-6, pkg.BF16, 0),
    lambda: pkg.rmsnorm_bwd(1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 4, 64, pkg.BF16, 0),
    lambda: pkg.rmsnorm_add_fwd(1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 4, 64, 1e-6, pkg.BF16, 0),
    lambda: pkg.rmsnorm_plan(4, 64, pkg.BF16, pkg.PASS_FWD),
]
for c in calls:
    try:
        c()
    except OSError:
        continue
    sys.exit("a call returned without the library")
print("raised")
"""
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT,
                         timeout=120)
    assert out.returncode == 0 and "raised" in out.stdout, out.stdout + out.stderr


def test_package_never_imports_the_oracle():
    pat = re.compile(r"^\s*(import|from)\s+oracle\b", re.M)
    for dirpath, _, files in os.walk(PKG_DIR):
        for f in files:
            if f.endswith(".py"):
                text = open(os.path.join(dirpath, f)).read()
                assert not pat.search(text), f"{f} imports the oracle"
    # the CUDA sources neither include nor name the oracle's C file
    csrc = os.path.join(PKG_DIR, "csrc")
    for f in os.listdir(csrc):
        text = open(os.path.join(csrc, f)).read()
        assert "rmsnorm_oracle" not in text and "oracle_rmsnorm" not in text, f


def test_host_tensors_are_refused_before_the_library():
    """Tensor arguments must be CUDA tensors: a host tensor raises in the
    binding, so no host address ever reaches a kernel."""
    import pytest
    import torch

    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    w = torch.ones(64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensors"):
        pkg.rmsnorm_fwd(x, w, x, torch.zeros(4), 4, 64, 1e-6, pkg.BF16, 0)
