"""The small-shape GPU tests again, against the checked debug build.

The checked build (-DRMSNORM_CHECKS, see build.py) tests every global store,
bulk copy and shared-memory ring access of the kernels against the extent it
belongs to (the tensor's M*N elements, w's and dw's N, rstd's M, the partial
rows of the workspace, the block's dynamic shared memory); a failed check
skips the access and records RMSNORM_ERR_OUT_OF_BOUNDS, which every test
reads back through rmsnorm_get_last_device_error. The same parity, residual,
naive and guard-band tests run in a child process with
RMSNORM_LIBRARY_VARIANT=checked, so each of their calls also proves that no
index left its tensor or its ring. The full-size cases are left out: they
cover no index path the small ones miss and take most of the time.
"""
from __future__ import annotations

import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FILES = ["tests/test_parity_gpu.py", "tests/test_residual_gpu.py", "tests/test_naive_gpu.py",
         "tests/test_guard_bands_gpu.py", "tests/test_zz_no_alloc.py"]
SKIP = "not full_size and not bitwise_repeatable and not strided_and_host"


def child_env():
    env = dict(os.environ)
    env["RMSNORM_LIBRARY_VARIANT"] = "checked"
    return env


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from memory_bound_normalization_gb300 import build as libbuild

    libbuild.build(checked=True)
    yield


def test_child_loads_the_checked_build():
    code = ("import memory_bound_normalization_gb300 as p; p.load_library(); "
            "print(p.library_path()); print(p.rmsnorm_version())")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=child_env(),
                         capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    path, version = out.stdout.split()[-2:]
    assert path.endswith(os.path.join("_build_checked", "librmsnorm.so"))
    assert version.endswith("+checks")


def test_small_shape_suites_under_checks():
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           "-k", SKIP, *FILES]
    out = subprocess.run(cmd, cwd=ROOT, env=child_env(), capture_output=True, text=True,
                         timeout=1800)
    tail = (out.stdout + out.stderr)[-4000:]
    assert out.returncode == 0, tail
    assert " passed" in tail and " failed" not in tail, tail
