"""ctypes loader for librmsnorm_gb300.so (the C ABI of include/rmsnorm.h).

Loading needs no GPU (the CUDA runtime is linked statically and only reaches
the driver on the first CUDA call), so symbol checks run anywhere.  If the
library has not been built, every entry point raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB_PATH

# Names exported by the library, in header order.
EXPORTS = (
    "rmsnorm_fwd",
    "rmsnorm_vjp",
    "rmsnorm_fused_vjp",
    "rmsnorm_fwd_ex",
    "rmsnorm_vjp_ex",
    "rmsnorm_gated_silu",
    "rmsnorm_rope_kv_append",
    "rmsnorm_vjp_workspace_size",
    "rmsnorm_vjp_ws",
    "rmsnorm_vjp_noalloc",
    "rmsnorm_status_string",
    "rmsnorm_last_cuda_error",
    "rmsnorm_device_status",
    "rmsnorm_debug_inject",
    "rmsnorm_debug_fail_allocs",
    "rmsnorm_debug_claim_counters",
    "rmsnorm_describe_dispatch",
)

STATUS = {
    0: "RMSNORM_OK",
    1: "RMSNORM_ERR_INVALID_ARG",
    2: "RMSNORM_ERR_UNSUPPORTED",
    3: "RMSNORM_ERR_CUDA",
    4: "RMSNORM_ERR_NO_MEMORY",
    5: "RMSNORM_ERR_TIMEOUT",
}
DEVSTATUS_WAIT_TIMEOUT = 1
DEVSTATUS_BAD_INDEX = 2
MAX_D = 1 << 24
VJP_NOALLOC_MAX_BYTES = 16 << 20

_vp = ctypes.c_void_p
_f = ctypes.c_float
_i64 = ctypes.c_int64
_i = ctypes.c_int

_lock = threading.Lock()
_lib = None


class RmsnormError(RuntimeError):
    """A non-zero status returned by the C library."""

    def __init__(self, fn: str, status: int, detail: str = ""):
        self.status = status
        name = STATUS.get(status, "status %d" % status)
        msg = "%s failed: %s" % (fn, name)
        if detail:
            msg += " (" + detail + ")"
        super().__init__(msg)


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    lib.rmsnorm_fwd.argtypes = [_vp, _vp, _vp, _f, _f, _vp, _vp, _i64, _i64, _i, _vp]
    lib.rmsnorm_fwd.restype = _i
    lib.rmsnorm_vjp.argtypes = [_vp, _vp, _vp, _f, _f, _vp, _vp, _i64, _i64, _i, _vp]
    lib.rmsnorm_vjp.restype = _i
    lib.rmsnorm_fused_vjp.argtypes = [_vp, _vp, _vp, _vp, _f, _f, _vp, _vp, _i64, _i64, _i, _vp]
    lib.rmsnorm_fused_vjp.restype = _i
    lib.rmsnorm_fwd_ex.argtypes = [_vp, _i64, _vp, _i64, _vp, _f, _f, _vp, _i64, _vp, _i64, _vp,
                                   _i64, _i64, _i, _vp]
    lib.rmsnorm_fwd_ex.restype = _i
    lib.rmsnorm_vjp_ex.argtypes = [_vp, _i64, _vp, _vp, _i64, _vp, _i64, _vp, _f, _f, _vp, _i64,
                                   _vp, _i64, _i64, _i, _vp]
    lib.rmsnorm_vjp_ex.restype = _i
    lib.rmsnorm_gated_silu.argtypes = [_vp, _vp, _i64, _i64, _i, _vp]
    lib.rmsnorm_gated_silu.restype = _i
    lib.rmsnorm_rope_kv_append.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _f,
                                           _i, _i64, _i64, _i64, _i64, _i64, _i, _vp]
    lib.rmsnorm_rope_kv_append.restype = _i
    lib.rmsnorm_vjp_workspace_size.argtypes = [_i64, _i64, _i]
    lib.rmsnorm_vjp_workspace_size.restype = ctypes.c_size_t
    lib.rmsnorm_vjp_ws.argtypes = [_vp, _vp, _vp, _f, _f, _vp, _vp, _i64, _i64, _i, _vp,
                                   ctypes.c_size_t, _vp]
    lib.rmsnorm_vjp_ws.restype = _i
    lib.rmsnorm_vjp_noalloc.argtypes = [_vp, _vp, _vp, _f, _f, _vp, _vp, _i64, _i64, _i, _vp]
    lib.rmsnorm_vjp_noalloc.restype = _i
    lib.rmsnorm_status_string.argtypes = [_i]
    lib.rmsnorm_status_string.restype = ctypes.c_char_p
    lib.rmsnorm_last_cuda_error.argtypes = []
    lib.rmsnorm_last_cuda_error.restype = _i
    lib.rmsnorm_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), _i]
    lib.rmsnorm_device_status.restype = _i
    lib.rmsnorm_debug_inject.argtypes = [_i64, _i64]
    lib.rmsnorm_debug_inject.restype = _i
    lib.rmsnorm_debug_fail_allocs.argtypes = [_i]
    lib.rmsnorm_debug_fail_allocs.restype = _i
    lib.rmsnorm_debug_claim_counters.argtypes = [_i]
    lib.rmsnorm_debug_claim_counters.restype = _i
    lib.rmsnorm_describe_dispatch.argtypes = [_i, _i64, _i64, _i, _i, _i]
    lib.rmsnorm_describe_dispatch.restype = ctypes.c_char_p
    return lib


def lib() -> ctypes.CDLL:
    """The loaded C library.  Raises if it was never built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        "%s is missing: build it with `python -m rmsnorm_fwd_bwd_add_gb300.build` "
                        "(nvcc, sm_103a); there is no CPU fallback" % LIB_PATH)
                _lib = _bind(ctypes.CDLL(LIB_PATH))
    return _lib


def check(fn: str, status: int) -> None:
    if status != 0:
        detail = ""
        if status == 3:
            detail = "cudaError %d" % lib().rmsnorm_last_cuda_error()
        raise RmsnormError(fn, status, detail)
