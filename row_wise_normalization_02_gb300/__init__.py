"""Python binding of the GB300 RMSNorm C ABI (``include/rmsnorm.h``).

Argument marshalling only: every function forwards to the entry point of the
same name in ``librmsnorm_gb300.so`` and raises :class:`RMSNormError` on a
non-OK status.  Pointers are device addresses (ints, or objects with a
``data_ptr()`` method such as torch tensors); ``stream`` is a raw
``cudaStream_t`` (int), an object with a ``cuda_stream`` attribute, or None
for the legacy default stream.  Importing works without the library; the
first call raises if it has not been built (``__graft_entry__.build()``) --
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = ["F32", "BF16", "OP_FWD", "OP_FUSED_ADD", "OP_BWD", "OP_FUSED_ADD_BWD", "RMSNormError",
           "OP_FWD_STRIDED", "OP_FWD_FP8", "OP_FUSED_ADD_FP8", "OP_FWD_NVFP4",
           "OP_FUSED_ADD_NVFP4", "rmsnorm_fwd_fp8", "rmsnorm_fwd_nvfp4", "OP_LAYERNORM_FWD",
           "OP_LAYERNORM_BWD", "layernorm_fwd", "layernorm_bwd_workspace_size", "layernorm_bwd",
           "library_path", "rmsnorm_fused_add_bwd", "rmsnorm_fwd_strided",
           "load_library", "rmsnorm_fwd", "rmsnorm_fused_add_fwd", "rmsnorm_bwd",
           "rmsnorm_bwd_workspace_size", "rmsnorm_status_string", "rmsnorm_describe_plan",
           "rmsnorm_bwd_noalloc", "NOALLOC_SCRATCH_BYTES", "rmsnorm_check_device",
           "rmsnorm_last_error", "rmsnorm_reload_debug_env", "EXPORTED_SYMBOLS"]

F32 = 0
BF16 = 1
OP_FWD, OP_FUSED_ADD, OP_BWD, OP_FUSED_ADD_BWD = 0, 1, 2, 3
OP_FWD_STRIDED, OP_FWD_FP8, OP_FUSED_ADD_FP8, OP_FWD_NVFP4, OP_FUSED_ADD_NVFP4 = 4, 5, 6, 7, 8
OP_LAYERNORM_FWD, OP_LAYERNORM_BWD = 9, 10
_DT_NAMES = {"f32": F32, "bf16": BF16}

EXPORTED_SYMBOLS = ("rmsnorm_fwd", "rmsnorm_fused_add_fwd", "rmsnorm_bwd_workspace_size",
                    "rmsnorm_bwd", "rmsnorm_status_string", "rmsnorm_describe_plan",
                    "rmsnorm_bwd_noalloc", "rmsnorm_check_device", "rmsnorm_last_error",
                    "rmsnorm_fused_add_bwd", "rmsnorm_fwd_strided", "rmsnorm_fwd_fp8",
                    "rmsnorm_fwd_nvfp4", "layernorm_fwd", "layernorm_bwd_workspace_size",
                    "layernorm_bwd", "rmsnorm_reload_debug_env")

# Size of the library-owned scratch of rmsnorm_bwd_noalloc (16 MiB).
NOALLOC_SCRATCH_BYTES = 16 << 20

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "librmsnorm_gb300.so")
_lock = threading.Lock()
_lib = None


class RMSNormError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = f" [{rmsnorm_last_error()}]" if status == 5 else ""
        super().__init__(f"{where}: {rmsnorm_status_string(status)} (status {status}){detail}")


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load the shared library (raises if it is missing: no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise ImportError(f"{_LIB_PATH} is not built; run __graft_entry__.build() "
                                  "(nvcc, sm_103a) first")
            lib = ctypes.CDLL(_LIB_PATH)
            P, I64, I, F, SZ = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                                ctypes.c_size_t)
            lib.rmsnorm_fwd.argtypes = [P, P, P, P, I64, I64, F, I, I, P]
            lib.rmsnorm_fwd.restype = I
            lib.rmsnorm_fused_add_fwd.argtypes = [P, P, P, P, P, I64, I64, F, I, I, P]
            lib.rmsnorm_fused_add_fwd.restype = I
            lib.rmsnorm_bwd_workspace_size.argtypes = [I64, I64, I, I, I, ctypes.POINTER(SZ)]
            lib.rmsnorm_bwd_workspace_size.restype = I
            lib.rmsnorm_bwd.argtypes = [P, P, P, P, P, P, P, SZ, I64, I64, F, I, I, P]
            lib.rmsnorm_bwd.restype = I
            lib.rmsnorm_status_string.argtypes = [I]
            lib.rmsnorm_status_string.restype = ctypes.c_char_p
            lib.rmsnorm_describe_plan.argtypes = [I, I64, I64, I, I, I, I, ctypes.c_char_p, SZ]
            lib.rmsnorm_describe_plan.restype = I
            lib.rmsnorm_bwd_noalloc.argtypes = [P, P, P, P, P, P, I64, I64, F, I, I, P]
            lib.rmsnorm_bwd_noalloc.restype = I
            lib.rmsnorm_check_device.argtypes = [P]
            lib.rmsnorm_check_device.restype = I
            lib.rmsnorm_fused_add_bwd.argtypes = [P, P, P, P, P, P, I, P, SZ, I64, I64, F, I, I, P]
            lib.rmsnorm_fused_add_bwd.restype = I
            lib.rmsnorm_fwd_strided.argtypes = [P, I64, I64, P, P, I64, I64, P, I64, I64, I64, F,
                                                I, I, P]
            lib.rmsnorm_fwd_strided.restype = I
            lib.layernorm_fwd.argtypes = [P, P, P, P, P, P, I64, I64, F, I, I, P]
            lib.layernorm_fwd.restype = I
            lib.layernorm_bwd_workspace_size.argtypes = [I64, I64, I, I, I, ctypes.POINTER(SZ)]
            lib.layernorm_bwd_workspace_size.restype = I
            lib.layernorm_bwd.argtypes = [P, P, P, P, P, P, P, P, P, SZ, I64, I64, F, I, I, P]
            lib.layernorm_bwd.restype = I
            lib.rmsnorm_fwd_fp8.argtypes = [P, P, P, P, P, P, I64, I64, F, I, I, P]
            lib.rmsnorm_fwd_fp8.restype = I
            lib.rmsnorm_fwd_nvfp4.argtypes = [P, P, P, F, P, P, P, I64, I64, F, I, I, P]
            lib.rmsnorm_fwd_nvfp4.restype = I
            lib.rmsnorm_last_error.argtypes = []
            lib.rmsnorm_last_error.restype = ctypes.c_char_p
            lib.rmsnorm_reload_debug_env.argtypes = []
            lib.rmsnorm_reload_debug_env.restype = None
            _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, int):
        return a
    return int(a.data_ptr())


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _dt(d) -> int:
    """dtype name ("f32", "bf16") or raw code (passed through unchanged)."""
    return _DT_NAMES[d] if isinstance(d, str) else int(d)


def _check(status: int, where: str):
    if status != 0:
        raise RMSNormError(status, where)


def rmsnorm_fwd(x, gamma, y, rstd, M, N, eps, x_dtype, w_dtype, stream=None):
    _check(load_library().rmsnorm_fwd(_ptr(x), _ptr(gamma), _ptr(y), _ptr(rstd), M, N, eps,
                                      _dt(x_dtype), _dt(w_dtype), _stream(stream)),
           "rmsnorm_fwd")


def rmsnorm_fused_add_fwd(x, residual, gamma, y, rstd, M, N, eps, x_dtype, w_dtype,
                          stream=None):
    _check(load_library().rmsnorm_fused_add_fwd(_ptr(x), _ptr(residual), _ptr(gamma), _ptr(y),
                                                _ptr(rstd), M, N, eps, _dt(x_dtype),
                                                _dt(w_dtype), _stream(stream)),
           "rmsnorm_fused_add_fwd")


def rmsnorm_bwd_workspace_size(M, N, x_dtype, w_dtype, device=-1) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().rmsnorm_bwd_workspace_size(M, N, _dt(x_dtype), _dt(w_dtype), device,
                                                     ctypes.byref(out)),
           "rmsnorm_bwd_workspace_size")
    return int(out.value)


def rmsnorm_bwd(dy, x, rstd, gamma, dx, dgamma, workspace, workspace_bytes, M, N, eps, x_dtype,
                w_dtype, stream=None):
    _check(load_library().rmsnorm_bwd(_ptr(dy), _ptr(x), _ptr(rstd), _ptr(gamma), _ptr(dx),
                                      _ptr(dgamma), _ptr(workspace), workspace_bytes, M, N, eps,
                                      _dt(x_dtype), _dt(w_dtype), _stream(stream)),
           "rmsnorm_bwd")


def rmsnorm_fwd_strided(x, x_stride_token, x_stride_head, gamma, y, y_stride_token,
                        y_stride_head, rstd, T, H, D, eps, x_dtype, w_dtype, stream=None):
    _check(load_library().rmsnorm_fwd_strided(_ptr(x), x_stride_token, x_stride_head,
                                              _ptr(gamma), _ptr(y), y_stride_token,
                                              y_stride_head, _ptr(rstd), T, H, D, eps,
                                              _dt(x_dtype), _dt(w_dtype), _stream(stream)),
           "rmsnorm_fwd_strided")


def layernorm_fwd(x, gamma, beta, y, mean, rstd, M, N, eps, x_dtype, w_dtype, stream=None):
    _check(load_library().layernorm_fwd(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), _ptr(mean),
                                        _ptr(rstd), M, N, eps, _dt(x_dtype), _dt(w_dtype),
                                        _stream(stream)),
           "layernorm_fwd")


def layernorm_bwd_workspace_size(M, N, x_dtype, w_dtype, device=-1):
    n = ctypes.c_size_t(0)
    _check(load_library().layernorm_bwd_workspace_size(M, N, _dt(x_dtype), _dt(w_dtype), device,
                                                       ctypes.byref(n)),
           "layernorm_bwd_workspace_size")
    return int(n.value)


def layernorm_bwd(dy, x, mean, rstd, gamma, dx, dgamma, dbeta, workspace, workspace_bytes, M, N,
                  eps, x_dtype, w_dtype, stream=None):
    _check(load_library().layernorm_bwd(_ptr(dy), _ptr(x), _ptr(mean), _ptr(rstd), _ptr(gamma),
                                        _ptr(dx), _ptr(dgamma), _ptr(dbeta), _ptr(workspace),
                                        workspace_bytes, M, N, eps, _dt(x_dtype), _dt(w_dtype),
                                        _stream(stream)),
           "layernorm_bwd")


def rmsnorm_fwd_fp8(x, residual, gamma, q, scale, rstd, M, N, eps, x_dtype, w_dtype,
                    stream=None):
    _check(load_library().rmsnorm_fwd_fp8(_ptr(x), _ptr(residual), _ptr(gamma), _ptr(q),
                                          _ptr(scale), _ptr(rstd), M, N, eps, _dt(x_dtype),
                                          _dt(w_dtype), _stream(stream)),
           "rmsnorm_fwd_fp8")


def rmsnorm_fwd_nvfp4(x, residual, gamma, global_scale, q, block_scale, rstd, M, N, eps,
                      x_dtype, w_dtype, stream=None):
    _check(load_library().rmsnorm_fwd_nvfp4(_ptr(x), _ptr(residual), _ptr(gamma),
                                            float(global_scale), _ptr(q), _ptr(block_scale),
                                            _ptr(rstd), M, N, eps, _dt(x_dtype), _dt(w_dtype),
                                            _stream(stream)),
           "rmsnorm_fwd_nvfp4")


def rmsnorm_fused_add_bwd(dy, h, rstd, gamma, dres, dgamma, dgamma_dtype, workspace,
                          workspace_bytes, M, N, eps, x_dtype, w_dtype, stream=None):
    _check(load_library().rmsnorm_fused_add_bwd(_ptr(dy), _ptr(h), _ptr(rstd), _ptr(gamma),
                                                _ptr(dres), _ptr(dgamma), _dt(dgamma_dtype),
                                                _ptr(workspace), workspace_bytes, M, N, eps,
                                                _dt(x_dtype), _dt(w_dtype), _stream(stream)),
           "rmsnorm_fused_add_bwd")


def rmsnorm_bwd_noalloc(dy, x, rstd, gamma, dx, dgamma, M, N, eps, x_dtype, w_dtype,
                        stream=None):
    """rmsnorm_bwd without a workspace argument: for callers that cannot
    allocate, the dgamma partials use a scratch array owned by the library
    (see include/rmsnorm.h for its limit and sharing rules)."""
    _check(load_library().rmsnorm_bwd_noalloc(_ptr(dy), _ptr(x), _ptr(rstd), _ptr(gamma),
                                              _ptr(dx), _ptr(dgamma), M, N, eps, _dt(x_dtype),
                                              _dt(w_dtype), _stream(stream)),
           "rmsnorm_bwd_noalloc")


def rmsnorm_check_device(stream=None):
    """Wait for `stream`, then raise RMSNormError(RMSNORM_ERR_TIMEOUT) if a
    kernel on the current device gave up a bounded wait (clears the flag)."""
    _check(load_library().rmsnorm_check_device(_stream(stream)), "rmsnorm_check_device")


def rmsnorm_reload_debug_env():
    """Re-read RMSNORM_FORCE_VARIANT, RMSNORM_WAIT_LIMIT_CYCLES and
    RMSNORM_NO_PDL from the environment (the library reads them once at load;
    call this after changing them, with no other thread inside the library)."""
    load_library().rmsnorm_reload_debug_env()


def rmsnorm_last_error() -> str:
    """The failing CUDA call behind this thread's last RMSNORM_ERR_CUDA."""
    try:
        return load_library().rmsnorm_last_error().decode()
    except ImportError:
        return ""


def rmsnorm_status_string(status: int) -> str:
    try:
        return load_library().rmsnorm_status_string(status).decode()
    except ImportError:
        return f"status {status}"


def rmsnorm_describe_plan(op, M, N, x_dtype, w_dtype, aligned16=True, device=-1) -> str:
    """aligned16: True / False, or "mixed" (ops 0-3: outputs on 16 bytes, x and
    dy off them)."""
    buf = ctypes.create_string_buffer(256)
    a = 2 if aligned16 == "mixed" else (1 if aligned16 else 0)
    _check(load_library().rmsnorm_describe_plan(op, M, N, _dt(x_dtype), _dt(w_dtype),
                                                a, device, buf, 256),
           "rmsnorm_describe_plan")
    return buf.value.decode()
