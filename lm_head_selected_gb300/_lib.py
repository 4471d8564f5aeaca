"""ctypes loader for ``liblinear_logp.so`` (the C ABI in include/linear_logp.h).

Argument marshalling only.  If the library is missing or fails to load, every
call raises: there is no fallback implementation anywhere in this package.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

LLP_OK = 0
LLP_ERR_NULL_POINTER = -1
LLP_ERR_BAD_SHAPE = -2
LLP_ERR_MISALIGNED = -3
LLP_ERR_UNSUPPORTED_DEVICE = -4
LLP_ERR_WORKSPACE_TOO_SMALL = -5
LLP_ERR_CUDA = -6
LLP_ERR_DEVICE_TIMEOUT = -7

EXPORTED = (
    "linear_logp_fwd_workspace_bytes",
    "linear_logp_bwd_workspace_bytes",
    "linear_logp_fwd",
    "linear_logp_bwd",
    "linear_logp_status_string",
    "linear_logp_device_status",
    "linear_logp_profile_start",
    "linear_logp_profile_stop",
    "linear_logp_kernel_name",
    "linear_logp_fwd_noalloc",
    "linear_logp_selftest_wait_timeout",
    "linear_logp_fwd_indexed_workspace_bytes",
    "linear_logp_bwd_indexed_workspace_bytes",
    "linear_logp_fwd_indexed",
    "linear_logp_bwd_indexed",
    "linear_logp_fwd_shard",
    "linear_logp_merge_shards",
    "linear_logp_bwd_shard",
    "linear_logp_sum_partials",
    "linear_logp_fwd_f16",
    "linear_logp_bwd_f16",
    "linear_logp_fwd_indexed_f16",
    "linear_logp_bwd_indexed_f16",
    "linear_logp_fwd_shard_f16",
    "linear_logp_bwd_shard_f16",
    "linear_logp_sum_partials_f16",
    "linear_logp_last_cuda_error",
    "linear_logp_cuda_error_name",
    "linear_logp_last_failure",
)
# include/fused_logp.h (logits-input op, same library)
EXPORTED_FUSED = (
    "fused_logp_workspace_bytes",
    "fused_logp_fwd",
    "fused_logp_bwd",
    "fused_logp_fwd_indexed_workspace_bytes",
    "fused_logp_bwd_indexed_workspace_bytes",
    "fused_logp_fwd_indexed",
    "fused_logp_bwd_indexed",
)
DEVICE_SELFTEST_CODE = 6
LLP_ERR_SCRATCH_LIMIT = -8

_lock = threading.Lock()
_lib = None

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_size = ctypes.c_size_t


class LinearLogpError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed with status {status}: {msg}")
        self.status = status


def library_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Load the shared library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
                "(or lm_head_selected_gb300.build.build()); there is no fallback path")
        lib = ctypes.CDLL(path)
        lib.linear_logp_fwd_workspace_bytes.argtypes = [_i64, _i64, _i64]
        lib.linear_logp_fwd_workspace_bytes.restype = _size
        lib.linear_logp_bwd_workspace_bytes.argtypes = [_i64, _i64, _i64, ctypes.c_int]
        lib.linear_logp_bwd_workspace_bytes.restype = _size
        lib.linear_logp_fwd.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _p, _p, _p, _size, _p]
        lib.linear_logp_fwd.restype = ctypes.c_int
        lib.linear_logp_bwd.argtypes = [_p, _p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _p, _p, _p, _p,
                                        _size, _p]
        lib.linear_logp_bwd.restype = ctypes.c_int
        lib.linear_logp_fwd_f16.argtypes = lib.linear_logp_fwd.argtypes
        lib.linear_logp_fwd_f16.restype = ctypes.c_int
        lib.linear_logp_bwd_f16.argtypes = lib.linear_logp_bwd.argtypes
        lib.linear_logp_bwd_f16.restype = ctypes.c_int
        lib.linear_logp_status_string.argtypes = [ctypes.c_int]
        lib.linear_logp_status_string.restype = ctypes.c_char_p
        lib.linear_logp_device_status.argtypes = [_p, ctypes.POINTER(ctypes.c_uint)]
        lib.linear_logp_device_status.restype = ctypes.c_int
        lib.linear_logp_profile_start.argtypes = [ctypes.c_int]
        lib.linear_logp_profile_start.restype = ctypes.c_int
        lib.linear_logp_profile_stop.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_float),
                                                 ctypes.c_int]
        lib.linear_logp_profile_stop.restype = ctypes.c_int
        lib.linear_logp_kernel_name.argtypes = [ctypes.c_int]
        lib.linear_logp_kernel_name.restype = ctypes.c_char_p
        lib.linear_logp_fwd_noalloc.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _p, _p, _p]
        lib.linear_logp_fwd_noalloc.restype = ctypes.c_int
        lib.linear_logp_selftest_wait_timeout.argtypes = [ctypes.c_ulonglong, _p]
        lib.linear_logp_selftest_wait_timeout.restype = ctypes.c_int
        lib.linear_logp_fwd_indexed_workspace_bytes.argtypes = [_i64, _i64, _i64, _i64]
        lib.linear_logp_fwd_indexed_workspace_bytes.restype = _size
        lib.linear_logp_bwd_indexed_workspace_bytes.argtypes = [_i64, _i64, _i64, _i64, ctypes.c_int]
        lib.linear_logp_bwd_indexed_workspace_bytes.restype = _size
        lib.linear_logp_fwd_indexed.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _p, _i64, _p, _p, _p,
                                                _size, _p]
        lib.linear_logp_fwd_indexed.restype = ctypes.c_int
        lib.linear_logp_bwd_indexed.argtypes = [_p, _p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _p, _i64, _p,
                                                _p, _p, _p, _size, _p]
        lib.linear_logp_bwd_indexed.restype = ctypes.c_int
        lib.linear_logp_fwd_indexed_f16.argtypes = lib.linear_logp_fwd_indexed.argtypes
        lib.linear_logp_fwd_indexed_f16.restype = ctypes.c_int
        lib.linear_logp_bwd_indexed_f16.argtypes = lib.linear_logp_bwd_indexed.argtypes
        lib.linear_logp_bwd_indexed_f16.restype = ctypes.c_int
        lib.linear_logp_fwd_shard.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _p, _p, _p, _p,
                                              _size, _p]
        lib.linear_logp_fwd_shard.restype = ctypes.c_int
        lib.linear_logp_merge_shards.argtypes = [_p, _p, _p, _i64, _i64, _p, _i64, _i64, _p, _p, _p]
        lib.linear_logp_merge_shards.restype = ctypes.c_int
        lib.linear_logp_bwd_shard.argtypes = [_p, _p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _p,
                                              _p, _p, _p, _size, _p]
        lib.linear_logp_bwd_shard.restype = ctypes.c_int
        lib.linear_logp_sum_partials.argtypes = [_p, _i64, _i64, _p, _p]
        lib.linear_logp_sum_partials.restype = ctypes.c_int
        for name in ("fwd_shard", "bwd_shard", "sum_partials"):
            f16, base = getattr(lib, f"linear_logp_{name}_f16"), getattr(lib, f"linear_logp_{name}")
            f16.argtypes = base.argtypes
            f16.restype = ctypes.c_int
        lib.linear_logp_last_cuda_error.argtypes = []
        lib.linear_logp_last_cuda_error.restype = ctypes.c_int
        lib.linear_logp_cuda_error_name.argtypes = [ctypes.c_int]
        lib.linear_logp_cuda_error_name.restype = ctypes.c_char_p
        lib.linear_logp_last_failure.argtypes = [ctypes.POINTER(ctypes.c_int)] * 3
        lib.linear_logp_last_failure.restype = ctypes.c_int
        lib.fused_logp_workspace_bytes.argtypes = [_i64, _i64]
        lib.fused_logp_workspace_bytes.restype = _size
        lib.fused_logp_fwd.argtypes = [_p, ctypes.c_int, _i64, _i64, _p, _i64, _p, _p, _p, _p, _size, _p]
        lib.fused_logp_fwd.restype = ctypes.c_int
        lib.fused_logp_bwd.argtypes = [_p, _p, _p, _p, ctypes.c_int, _i64, _i64, _p, _i64, _p, _p]
        lib.fused_logp_bwd.restype = ctypes.c_int
        lib.fused_logp_fwd_indexed_workspace_bytes.argtypes = [_i64, _i64, _i64]
        lib.fused_logp_fwd_indexed_workspace_bytes.restype = _size
        lib.fused_logp_bwd_indexed_workspace_bytes.argtypes = [_i64, _i64]
        lib.fused_logp_bwd_indexed_workspace_bytes.restype = _size
        lib.fused_logp_fwd_indexed.argtypes = [_p, ctypes.c_int, _i64, _i64, _p, _i64, _p, _i64, _p, _p, _p, _p,
                                               _size, _p]
        lib.fused_logp_fwd_indexed.restype = ctypes.c_int
        lib.fused_logp_bwd_indexed.argtypes = [_p, _p, _p, _p, ctypes.c_int, _i64, _i64, _p, _i64, _p, _i64, _p, _p,
                                               _size, _p]
        lib.fused_logp_bwd_indexed.restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().linear_logp_status_string(int(status)).decode()


def check(fn: str, status: int) -> None:
    if status != LLP_OK:
        msg = status_string(status)
        if status == LLP_ERR_CUDA:
            lib = load()
            code, drv, site = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
            lib.linear_logp_last_failure(ctypes.byref(code), ctypes.byref(drv), ctypes.byref(site))
            detail = [f"check at api.cu:{site.value}"]
            if code.value:
                detail.append(f"{lib.linear_logp_cuda_error_name(code.value).decode()} ({code.value})")
            if drv.value:
                detail.append(f"tensor-map encoding returned CUresult {drv.value}")
            msg += " [" + "; ".join(detail) + "]"
        raise LinearLogpError(fn, status, msg)


def profile_start(capacity: int) -> None:
    check("linear_logp_profile_start", load().linear_logp_profile_start(int(capacity)))


def profile_stop(capacity: int):
    """Returns [(kernel name, milliseconds), ...] in launch order."""
    lib = load()
    ids = (ctypes.c_int * capacity)()
    ms = (ctypes.c_float * capacity)()
    n = lib.linear_logp_profile_stop(ids, ms, capacity)
    if n < 0:
        check("linear_logp_profile_stop", n)
    n = min(n, capacity)
    return [(lib.linear_logp_kernel_name(ids[i]).decode(), float(ms[i])) for i in range(n)]
