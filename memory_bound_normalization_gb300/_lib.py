"""ctypes binding of librmsnorm.so (declared in include/rmsnorm.h).

Argument marshalling only: every step of the computation runs in the CUDA
library. Functions keep the C names and argument order. Tensor arguments may
be torch tensors (their ``data_ptr()`` is passed) or raw integer device
addresses; ``stream`` may be a ``torch.cuda.Stream``, an integer handle, or
None (the current torch stream of the current device).

There is no fallback: if the library is missing or fails to load, importing
the first function raises.

With RMSNORM_LIBRARY_VARIANT=checked in the environment the binding loads the
checked debug build of the same sources instead (every kernel access tested
against its extent; see build.py), for tests that look for out-of-range
accesses.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

F32 = 0
BF16 = 1
F16 = 2
BF16_W_F32 = 3  # bf16 activations, fp32 weight
F16_W_F32 = 4  # fp16 activations, fp32 weight

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_MISALIGNED = 3
ERR_CUDA = 4
ERR_NOMEM = 5
ERR_DEVICE_TIMEOUT = 6
ERR_OUT_OF_BOUNDS = 7  # reported by the checked debug build only

PASS_FWD = 0
PASS_BWD = 1
PASS_BWD_RES = 2  # rmsnorm_add_bwd with dres
PASS_FWD_ADD = 3  # rmsnorm_add_fwd

PROBE_COPY = 0
PROBE_WRITE = 1
PROBE_2R1W = 2

VARIANTS = {0: "none", 1: "rowgroup", 2: "cta_row", 3: "cluster_row", 4: "scalar",
            5: "two_pass", 6: "ring"}

# Exported symbols, in header order (tests check the library against this
# list and the header against the library).
EXPORTS = (
    "rmsnorm_fwd",
    "rmsnorm_bwd",
    "rmsnorm_bwd_workspace_size",
    "rmsnorm_bwd_ws",
    "rmsnorm_add_fwd",
    "rmsnorm_add_bwd",
    "rmsnorm_noalloc_scratch_bytes",
    "rmsnorm_bwd_noalloc",
    "rmsnorm_bwd_naive",
    "rmsnorm_get_last_device_error",
    "rmsnorm_status_string",
    "rmsnorm_set_wait_limit_ns",
    "rmsnorm_test_drop_copy",
    "rmsnorm_probe",
    "rmsnorm_plan",
    "rmsnorm_version",
)


class RMSNormError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        name = status_string(status)
        super().__init__(f"{what}: {name}" if what else name)


class Plan(ctypes.Structure):
    _fields_ = [
        ("variant", ctypes.c_int),
        ("threads", ctypes.c_int),
        ("vectors_per_thread", ctypes.c_int),
        ("threads_per_row", ctypes.c_int),
        ("rows_per_unit", ctypes.c_int),
        ("cluster", ctypes.c_int),
        ("row_groups", ctypes.c_int),
        ("stages", ctypes.c_int),
        ("smem_bytes", ctypes.c_int),
        ("grid", ctypes.c_int),
        ("partial_rows", ctypes.c_int),
        ("workspace_bytes", ctypes.c_int64),
    ]

    def as_dict(self) -> dict:
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["variant_name"] = VARIANTS.get(self.variant, "?")
        return d


_lock = threading.Lock()
_lib: ctypes.CDLL | None = None


def checked_variant() -> bool:
    """True when this process is to load the checked debug build."""
    return os.environ.get("RMSNORM_LIBRARY_VARIANT", "") == "checked"


def library_path() -> str:
    return _build.lib_path(checked_variant())


def load_library(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load librmsnorm.so (optionally building it first). Raises OSError if
    it cannot be loaded; there is no other implementation to fall back on."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        checked = checked_variant()
        path = _build.lib_path(checked)
        if build_if_missing and (not os.path.exists(path) or _build.is_stale(checked)):
            _build.build(checked=checked)
        if not os.path.exists(path):
            raise OSError(
                f"{path} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        vp, i64, i, f, sz, u64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                                  ctypes.c_size_t, ctypes.c_uint64)
        lib.rmsnorm_fwd.argtypes = [vp, vp, vp, vp, i64, i64, f, i, vp]
        lib.rmsnorm_bwd.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i, vp]
        lib.rmsnorm_bwd_workspace_size.argtypes = [i64, i64, i, i]
        lib.rmsnorm_bwd_workspace_size.restype = sz
        lib.rmsnorm_bwd_ws.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i, vp, sz, vp]
        lib.rmsnorm_add_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, f, i, vp]
        lib.rmsnorm_add_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i, vp]
        lib.rmsnorm_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i, vp]
        lib.rmsnorm_noalloc_scratch_bytes.argtypes = []
        lib.rmsnorm_noalloc_scratch_bytes.restype = sz
        lib.rmsnorm_bwd_naive.argtypes = [vp, vp, vp, vp, vp, i64, i64, f, i, vp]
        lib.rmsnorm_get_last_device_error.argtypes = [vp]
        lib.rmsnorm_status_string.argtypes = [i]
        lib.rmsnorm_status_string.restype = ctypes.c_char_p
        lib.rmsnorm_set_wait_limit_ns.argtypes = [u64]
        lib.rmsnorm_set_wait_limit_ns.restype = None
        lib.rmsnorm_test_drop_copy.argtypes = [i64]
        lib.rmsnorm_test_drop_copy.restype = None
        lib.rmsnorm_probe.argtypes = [i, vp, vp, vp, sz, i, vp]
        lib.rmsnorm_plan.argtypes = [i64, i64, i, i, i, ctypes.POINTER(Plan)]
        lib.rmsnorm_version.argtypes = []
        lib.rmsnorm_version.restype = ctypes.c_char_p
        for name in ("rmsnorm_fwd", "rmsnorm_bwd", "rmsnorm_bwd_ws", "rmsnorm_add_fwd",
                     "rmsnorm_add_bwd", "rmsnorm_bwd_noalloc", "rmsnorm_bwd_naive",
                     "rmsnorm_get_last_device_error",
                     "rmsnorm_probe", "rmsnorm_plan"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(t) -> int | None:
    """Device address of a tensor argument (None and raw integer addresses
    pass through). Host or non-contiguous tensors are refused here, before
    anything reaches the library: its kernels read every tensor as dense
    row-major device memory."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError(f"tensor argument on {t.device}: the library takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensor argument is not contiguous: the library takes dense row-major "
                         "tensors (call .contiguous() first)")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def rmsnorm_fwd(x, w, y, rstd, M: int, N: int, eps: float, dtype: int, stream=None) -> int:
    return load_library().rmsnorm_fwd(_ptr(x), _ptr(w), _ptr(y), _ptr(rstd), M, N, eps, dtype,
                                      _stream(stream))


def rmsnorm_bwd(x, w, dy, rstd, dx, dw, M: int, N: int, dtype: int, stream=None) -> int:
    return load_library().rmsnorm_bwd(_ptr(x), _ptr(w), _ptr(dy), _ptr(rstd), _ptr(dx), _ptr(dw),
                                      M, N, dtype, _stream(stream))


def rmsnorm_bwd_workspace_size(M: int, N: int, dtype: int, device: int) -> int:
    return load_library().rmsnorm_bwd_workspace_size(M, N, dtype, device)


def rmsnorm_bwd_ws(x, w, dy, rstd, dx, dw, M: int, N: int, dtype: int, workspace,
                   workspace_bytes: int, stream=None) -> int:
    return load_library().rmsnorm_bwd_ws(_ptr(x), _ptr(w), _ptr(dy), _ptr(rstd), _ptr(dx),
                                         _ptr(dw), M, N, dtype, _ptr(workspace), workspace_bytes,
                                         _stream(stream))


def rmsnorm_add_fwd(x, residual, w, h, y, rstd, M: int, N: int, eps: float, dtype: int,
                    stream=None) -> int:
    return load_library().rmsnorm_add_fwd(_ptr(x), _ptr(residual), _ptr(w), _ptr(h), _ptr(y),
                                          _ptr(rstd), M, N, eps, dtype, _stream(stream))


def rmsnorm_add_bwd(h, w, dy, rstd, dres, dx, dw, M: int, N: int, dtype: int,
                    stream=None) -> int:
    return load_library().rmsnorm_add_bwd(_ptr(h), _ptr(w), _ptr(dy), _ptr(rstd), _ptr(dres),
                                          _ptr(dx), _ptr(dw), M, N, dtype, _stream(stream))


def rmsnorm_bwd_noalloc(x, w, dy, rstd, dx, dw, M: int, N: int, dtype: int, stream=None) -> int:
    """rmsnorm_bwd without any device allocation (fixed in-library scratch),
    for callers that cannot allocate; see include/rmsnorm.h."""
    return load_library().rmsnorm_bwd_noalloc(_ptr(x), _ptr(w), _ptr(dy), _ptr(rstd), _ptr(dx),
                                              _ptr(dw), M, N, dtype, _stream(stream))


def rmsnorm_noalloc_scratch_bytes() -> int:
    """Size of rmsnorm_bwd_noalloc's fixed scratch array, as the library was
    built with it."""
    return int(load_library().rmsnorm_noalloc_scratch_bytes())


def rmsnorm_bwd_naive(x, w, dy, dx, dw, M: int, N: int, eps: float, dtype: int,
                      stream=None) -> int:
    """The naive three-kernel backward (an ablation); see include/rmsnorm.h."""
    return load_library().rmsnorm_bwd_naive(_ptr(x), _ptr(w), _ptr(dy), _ptr(dx), _ptr(dw), M, N,
                                            eps, dtype, _stream(stream))


def rmsnorm_get_last_device_error(stream=None) -> int:
    return load_library().rmsnorm_get_last_device_error(_stream(stream))


def rmsnorm_status_string(status: int) -> str:
    return load_library().rmsnorm_status_string(status).decode()


status_string = rmsnorm_status_string


def rmsnorm_set_wait_limit_ns(ns: int) -> None:
    load_library().rmsnorm_set_wait_limit_ns(ns)


def rmsnorm_test_drop_copy(unit: int) -> None:
    load_library().rmsnorm_test_drop_copy(unit)


def rmsnorm_probe(kind: int, dst, a, b, nbytes: int, blocks_per_sm: int, stream=None) -> int:
    return load_library().rmsnorm_probe(kind, _ptr(dst), _ptr(a), _ptr(b), nbytes, blocks_per_sm,
                                        _stream(stream))


def rmsnorm_plan(M: int, N: int, dtype: int, pass_: int, device: int = -1) -> Plan:
    p = Plan()
    st = load_library().rmsnorm_plan(M, N, dtype, pass_, device, ctypes.byref(p))
    if st != OK:
        raise RMSNormError(st, "rmsnorm_plan")
    return p


def rmsnorm_version() -> str:
    return load_library().rmsnorm_version().decode()


def check(status: int, what: str = "") -> None:
    if status != OK:
        raise RMSNormError(status, what)
