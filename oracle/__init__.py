"""fp64 CPU oracle for RMSNorm forward and backward (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never calls it.

The arithmetic lives in ``rmsnorm_oracle.c`` (plain C, double precision,
ascending-order sums); this module compiles it with gcc and marshals arrays.
Definitions followed:

* forward ``r = 1/sqrt(mean(x^2) + eps)``, ``y = x * r * w`` -- "Chapter 13:
  Fused RMSNorm" (hello-gpu), section 13.1 equation; "Profiling, GPU
  utilisation and writing a fused kernel", Problem 15.
* backward ``dx = r * (g - xhat * mean(g * xhat))`` with ``g = dy * w``,
  ``xhat = x * r`` and ``dw = sum_rows dy * xhat`` -- "RMSNorm backward (almost)
  without the column reduction", sections "The backward pass" and "The naive
  kernel".
* residual add ``h = x + res`` stored in the activation type, then the
  forward on h; backward: the norm's input gradient at h plus the gradient
  reaching h from elsewhere -- "Profiling, GPU utilisation and writing a
  fused kernel", Problem 15 (the step that adds the residual to the kernel).

Inputs may be numpy arrays (float64, float32, float16, or uint16 holding bf16
bits with ``dtype="bf16"``) or CPU torch tensors (float64, float32, bfloat16,
float16). The weight may have its own type (e.g. fp32 with bf16 x and dy);
x and dy share one. Outputs are float64 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rmsnorm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

F64, F32, BF16, F16 = 0, 1, 2, 3
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle C file into a shared library; returns its path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    p, i64, d, i = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double, ctypes.c_int
    lib.oracle_rmsnorm_fwd.argtypes = [p, p, i64, i64, d, i, i, p, i64, p, p]
    lib.oracle_rmsnorm_bwd_dx.argtypes = [p, p, p, i64, i64, d, i, i, p, i64, p]
    lib.oracle_rmsnorm_bwd_dw.argtypes = [p, p, i64, i64, d, i, p]
    lib.oracle_round_to_dtype.argtypes = [p, i64, i, p]
    lib.oracle_rmsnorm_add_fwd.argtypes = [p, p, p, i64, i64, d, i, i, p, i64, p, p, p]
    lib.oracle_rmsnorm_add_bwd_dx.argtypes = [p, p, p, p, i64, i64, d, i, i, p, i64, p]
    for f in (lib.oracle_rmsnorm_fwd, lib.oracle_rmsnorm_bwd_dx, lib.oracle_rmsnorm_bwd_dw,
              lib.oracle_round_to_dtype, lib.oracle_rmsnorm_add_fwd,
              lib.oracle_rmsnorm_add_bwd_dx):
        f.restype = ctypes.c_int
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _as_host_array(a, dtype: str | None = None):
    """Return (contiguous numpy array, oracle dtype code)."""
    try:
        import torch  # noqa: WPS433 (optional dependency)
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(a, torch.Tensor):
        t = a.detach()
        if t.device.type != "cpu":
            raise ValueError("oracle inputs must be host tensors")
        t = t.contiguous()
        if t.dtype == torch.float64:
            return t.numpy(), F64
        if t.dtype == torch.float32:
            return t.numpy(), F32
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16), BF16
        if t.dtype == torch.float16:
            return t.view(torch.int16).numpy().view(np.uint16), F16
        raise TypeError(f"unsupported tensor dtype {t.dtype}")
    arr = np.ascontiguousarray(a)
    if dtype in ("bf16", "f16") or (dtype is None and arr.dtype == np.uint16):
        if arr.dtype != np.uint16:
            raise TypeError("16-bit arrays must be passed as uint16 bit patterns")
        return arr, (F16 if dtype == "f16" else BF16)
    if arr.dtype == np.float16:
        return arr.view(np.uint16), F16
    if arr.dtype == np.float64:
        return arr, F64
    if arr.dtype == np.float32:
        return arr, F32
    raise TypeError(f"unsupported array dtype {arr.dtype}")


def _ptr(arr) -> int | None:
    return arr.ctypes.data if arr is not None and arr.size else None


def _rows_arg(rows, M):
    if rows is None:
        return None, M
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    return r, int(r.size)


def _shape2(x_arr, N):
    if x_arr.ndim == 2:
        M, n = x_arr.shape
        if N is not None and N != n:
            raise ValueError("N does not match x")
        return M, n
    if N is None:
        raise ValueError("N is required for flat inputs")
    return x_arr.size // N, N


def _fwd(lib, x, w, eps, rows=None, N=None, dtype=None):
    xa, code = _as_host_array(x, dtype)
    wa, wcode = _as_host_array(w, dtype)
    M, N = _shape2(xa, N)
    ra, nrows = _rows_arg(rows, M)
    y = np.empty((nrows, N), dtype=np.float64)
    r = np.empty((nrows,), dtype=np.float64)
    rc = lib.oracle_rmsnorm_fwd(_ptr(xa), _ptr(wa), M, N, float(eps), code, wcode,
                                _ptr(ra), nrows, _ptr(y), _ptr(r))
    if rc:
        raise ValueError(f"oracle_rmsnorm_fwd rejected its arguments ({rc})")
    return y, r


def _bwd_dx(lib, x, w, dy, eps, rows=None, N=None, dtype=None):
    xa, code = _as_host_array(x, dtype)
    wa, wcode = _as_host_array(w, dtype)
    da, dcode = _as_host_array(dy, dtype)
    if code != dcode:
        raise TypeError("x and dy must share a dtype")
    M, N = _shape2(xa, N)
    ra, nrows = _rows_arg(rows, M)
    dx = np.empty((nrows, N), dtype=np.float64)
    rc = lib.oracle_rmsnorm_bwd_dx(_ptr(xa), _ptr(wa), _ptr(da), M, N, float(eps), code, wcode,
                                   _ptr(ra), nrows, _ptr(dx))
    if rc:
        raise ValueError(f"oracle_rmsnorm_bwd_dx rejected its arguments ({rc})")
    return dx


def _bwd_dw(lib, x, dy, eps, N=None, dtype=None):
    xa, code = _as_host_array(x, dtype)
    da, dcode = _as_host_array(dy, dtype)
    if code != dcode:
        raise TypeError("x and dy must share a dtype")
    M, N = _shape2(xa, N)
    dw = np.empty((N,), dtype=np.float64)
    rc = lib.oracle_rmsnorm_bwd_dw(_ptr(xa), _ptr(da), M, N, float(eps), code, _ptr(dw))
    if rc:
        raise ValueError(f"oracle_rmsnorm_bwd_dw rejected its arguments ({rc})")
    return dw


def _round(lib, v, dtype: str):
    code = {"f64": F64, "f32": F32, "bf16": BF16, "f16": F16}[dtype]
    va = np.ascontiguousarray(np.asarray(v, dtype=np.float64))
    out = np.empty_like(va)
    rc = lib.oracle_round_to_dtype(_ptr(va), va.size, code, _ptr(out))
    if rc:
        raise ValueError(f"oracle_round_to_dtype rejected its arguments ({rc})")
    return out


def _add_fwd(lib, x, res, w, eps, rows=None, N=None, dtype=None):
    xa, code = _as_host_array(x, dtype)
    sa, scode = _as_host_array(res, dtype)
    wa, wcode = _as_host_array(w, dtype)
    if code != scode:
        raise TypeError("x and the residual must share a dtype")
    M, N = _shape2(xa, N)
    ra, nrows = _rows_arg(rows, M)
    h = np.empty((nrows, N), dtype=np.float64)
    y = np.empty((nrows, N), dtype=np.float64)
    r = np.empty((nrows,), dtype=np.float64)
    rc = lib.oracle_rmsnorm_add_fwd(_ptr(xa), _ptr(sa), _ptr(wa), M, N, float(eps), code, wcode,
                                    _ptr(ra), nrows, _ptr(h), _ptr(y), _ptr(r))
    if rc:
        raise ValueError(f"oracle_rmsnorm_add_fwd rejected its arguments ({rc})")
    return h, y, r


def _add_bwd_dx(lib, h, w, dy, dres, eps, rows=None, N=None, dtype=None):
    ha, code = _as_host_array(h, dtype)
    wa, wcode = _as_host_array(w, dtype)
    da, dcode = _as_host_array(dy, dtype)
    ga = None
    if dres is not None:
        ga, gcode = _as_host_array(dres, dtype)
        if gcode != code:
            raise TypeError("h and dres must share a dtype")
    if code != dcode:
        raise TypeError("h and dy must share a dtype")
    M, N = _shape2(ha, N)
    ra, nrows = _rows_arg(rows, M)
    dx = np.empty((nrows, N), dtype=np.float64)
    rc = lib.oracle_rmsnorm_add_bwd_dx(_ptr(ha), _ptr(wa), _ptr(da), _ptr(ga), M, N, float(eps),
                                       code, wcode, _ptr(ra), nrows, _ptr(dx))
    if rc:
        raise ValueError(f"oracle_rmsnorm_add_bwd_dx rejected its arguments ({rc})")
    return dx


class Oracle:
    """The oracle entry points bound to one compiled library: the real one by
    default, or a deliberately broken copy that the mutation tests build.

    ``fwd(x, w, eps, rows=None)`` returns (y[nrows, N], r[nrows]);
    ``bwd_dx(x, w, dy, eps, rows=None)`` returns dx[nrows, N];
    ``bwd_dw(x, dy, eps)`` returns dw[N] summed over every row;
    ``round_to(v, dtype)`` rounds doubles into "f32", "bf16" or "f16" values;
    ``add_fwd(x, res, w, eps, rows=None)`` returns (h, y, r) of the residual
    add and norm; ``add_bwd_dx(h, w, dy, dres, eps, rows=None)`` returns the
    gradient of x and res (dres may be None).
    """

    def __init__(self, lib: ctypes.CDLL | None = None):
        self.lib = lib if lib is not None else load()

    def fwd(self, x, w, eps, rows=None, N=None, dtype=None):
        return _fwd(self.lib, x, w, eps, rows, N, dtype)

    def bwd_dx(self, x, w, dy, eps, rows=None, N=None, dtype=None):
        return _bwd_dx(self.lib, x, w, dy, eps, rows, N, dtype)

    def bwd_dw(self, x, dy, eps, N=None, dtype=None):
        return _bwd_dw(self.lib, x, dy, eps, N, dtype)

    def round_to(self, v, dtype: str):
        return _round(self.lib, v, dtype)

    def add_fwd(self, x, res, w, eps, rows=None, N=None, dtype=None):
        return _add_fwd(self.lib, x, res, w, eps, rows, N, dtype)

    def add_bwd_dx(self, h, w, dy, dres, eps, rows=None, N=None, dtype=None):
        return _add_bwd_dx(self.lib, h, w, dy, dres, eps, rows, N, dtype)


def fwd(x, w, eps: float, rows=None, N: int | None = None, dtype: str | None = None):
    """Forward on the host. Returns (y[nrows, N], r[nrows]) in float64."""
    return _fwd(load(), x, w, eps, rows, N, dtype)


def bwd_dx(x, w, dy, eps: float, rows=None, N: int | None = None, dtype: str | None = None):
    """Input gradient on the host. Returns dx[nrows, N] in float64."""
    return _bwd_dx(load(), x, w, dy, eps, rows, N, dtype)


def bwd_dw(x, dy, eps: float, N: int | None = None, dtype: str | None = None):
    """Weight gradient over all rows on the host. Returns dw[N] in float64."""
    return _bwd_dw(load(), x, dy, eps, N, dtype)


def round_to(v, dtype: str):
    """Doubles rounded (nearest even) into "f32", "bf16" or "f16" values."""
    return _round(load(), v, dtype)


def add_fwd(x, res, w, eps: float, rows=None, N: int | None = None, dtype: str | None = None):
    """Residual add and forward on the host. Returns (h, y, r) in float64:
    h = x + res as stored in x's type, y and r the forward of that h."""
    return _add_fwd(load(), x, res, w, eps, rows, N, dtype)


def add_bwd_dx(h, w, dy, dres, eps: float, rows=None, N: int | None = None,
               dtype: str | None = None):
    """Gradient of x and of the residual (they are equal) on the host: the
    norm's input gradient at the stored sum h plus dres (None for none)."""
    return _add_bwd_dx(load(), h, w, dy, dres, eps, rows, N, dtype)
