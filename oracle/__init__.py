"""ctypes wrapper of the double-precision RMSNorm oracle (``rmsnorm_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
bench's CPU baseline and reference arm, never by the library.  Arrays are numpy:
bf16 tensors as ``uint16`` bit patterns, fp32 tensors as ``float32``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rmsnorm_oracle.c")
_LIB = os.path.join(_HERE, "_librmsnorm_oracle.so")
_lock = threading.Lock()
_lib = None

DTYPE_CODES = {"f32": 0, "bf16": 1}
_P = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = f"{_LIB}.{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                           _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            I64, D, I = ctypes.c_int64, ctypes.c_double, ctypes.c_int
            lib.oracle_rmsnorm_fwd.argtypes = [_P, _P, I64, I64, D, I, I, _P, _P, _P, _P]
            lib.oracle_rmsnorm_fwd.restype = I
            lib.oracle_rmsnorm_fused_add_fwd.argtypes = [_P, _P, _P, I64, I64, D, I, I,
                                                         _P, _P, _P, _P, _P]
            lib.oracle_rmsnorm_fused_add_fwd.restype = I
            lib.oracle_rmsnorm_bwd.argtypes = [_P, _P, _P, _P, I64, I64, D, I, I,
                                               _P, _P, _P, _P, _P, _P, _P]
            lib.oracle_rmsnorm_bwd.restype = I
            lib.oracle_rmsnorm_fused_add_bwd.argtypes = [_P, _P, _P, _P, _P, I64, I64, D, I, I,
                                                         _P, _P, _P, _P, _P]
            lib.oracle_rmsnorm_fused_add_bwd.restype = I
            lib.oracle_rmsnorm_fwd_strided.argtypes = [_P, I64, I64, _P, I64, I64, I64, D, I, I,
                                                       _P, I64, I64, _P, _P]
            lib.oracle_rmsnorm_fwd_strided.restype = I
            lib.oracle_layernorm_fwd.argtypes = [_P, _P, _P, I64, I64, D, I, I, _P, _P, _P, _P,
                                                 _P, _P]
            lib.oracle_layernorm_fwd.restype = I
            lib.oracle_layernorm_bwd.argtypes = [_P, _P, _P, _P, _P, I64, I64, D, I, I, _P, _P,
                                                 _P, _P, _P, _P, _P]
            lib.oracle_layernorm_bwd.restype = I
            lib.oracle_rmsnorm_fwd_fp8.argtypes = [_P, _P, _P, I64, I64, D, I, I, _P, _P, _P, _P,
                                                   _P, _P]
            lib.oracle_rmsnorm_fwd_fp8.restype = I
            lib.oracle_rmsnorm_fwd_nvfp4.argtypes = [_P, _P, _P, I64, I64, D, D, I, I, _P, _P,
                                                     _P, _P, _P, _P]
            lib.oracle_rmsnorm_fwd_nvfp4.restype = I
            for name in ("oracle_round_e4m3", "oracle_round_e2m1"):
                getattr(lib, name).argtypes = [D]
                getattr(lib, name).restype = ctypes.c_uint8
            for name in ("oracle_e4m3_to_double", "oracle_e2m1_to_double"):
                getattr(lib, name).argtypes = [ctypes.c_uint8]
                getattr(lib, name).restype = D
            lib.oracle_round_bf16.argtypes = [D]
            lib.oracle_round_bf16.restype = ctypes.c_uint16
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = D
            _lib = lib
    return _lib


def _np(dtype: str):
    return np.float32 if dtype == "f32" else np.uint16


def _ptr(a):
    return None if a is None else a.ctypes.data


def _check_in(a, dtype, shape=None):
    a = np.ascontiguousarray(a)
    if a.dtype != _np(dtype):
        raise TypeError(f"expected {_np(dtype)} for dtype {dtype}, got {a.dtype}")
    if shape is not None and a.shape != tuple(shape):
        raise ValueError(f"expected shape {shape}, got {a.shape}")
    return a


def round_bf16(v: float) -> int:
    """Nearest bf16 bit pattern of a double (ties to even)."""
    return int(_load().oracle_round_bf16(float(v)))


def bf16_to_double(bits: int) -> float:
    return float(_load().oracle_bf16_to_double(int(bits)))


def bf16_array_to_f64(a: np.ndarray) -> np.ndarray:
    """Decode uint16 bf16 bit patterns exactly (widen to the fp32 bit layout)."""
    with np.errstate(invalid="ignore"):
        return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(
            np.float32).astype(np.float64)


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_array_to_f64(a) if dtype == "bf16" else np.asarray(a, np.float64)


def fwd(x, gamma, eps, x_dtype="bf16", w_dtype=None, want64=True):
    """RMSNorm forward of an M x N matrix.  Returns y (x_dtype), rstd (fp32) and,
    with ``want64``, y64 / rstd64 (float64)."""
    w_dtype = w_dtype or x_dtype
    x = _check_in(x, x_dtype)
    M, N = x.shape
    gamma = _check_in(gamma, w_dtype, (N,))
    y = np.empty((M, N), _np(x_dtype))
    rstd = np.empty(M, np.float32)
    y64 = np.empty((M, N), np.float64) if want64 else None
    r64 = np.empty(M, np.float64) if want64 else None
    rc = _load().oracle_rmsnorm_fwd(_ptr(x), _ptr(gamma), M, N, float(eps),
                                    DTYPE_CODES[x_dtype], DTYPE_CODES[w_dtype], _ptr(y),
                                    _ptr(y64), _ptr(rstd), _ptr(r64))
    if rc != 0:
        raise ValueError("oracle_rmsnorm_fwd rejected its arguments")
    out = {"y": y, "rstd": rstd}
    if want64:
        out.update(y64=y64, rstd64=r64)
    return out


def fused_add_fwd(x, residual, gamma, eps, x_dtype="bf16", w_dtype=None, want64=True):
    """h = residual + x (stored dtype), y = RMSNorm(h) * gamma.  The residual is
    not modified; h is returned."""
    w_dtype = w_dtype or x_dtype
    x = _check_in(x, x_dtype)
    M, N = x.shape
    residual = _check_in(residual, x_dtype, (M, N))
    gamma = _check_in(gamma, w_dtype, (N,))
    h = np.empty((M, N), _np(x_dtype))
    y = np.empty((M, N), _np(x_dtype))
    rstd = np.empty(M, np.float32)
    y64 = np.empty((M, N), np.float64) if want64 else None
    r64 = np.empty(M, np.float64) if want64 else None
    rc = _load().oracle_rmsnorm_fused_add_fwd(_ptr(x), _ptr(residual), _ptr(gamma), M, N,
                                              float(eps), DTYPE_CODES[x_dtype],
                                              DTYPE_CODES[w_dtype], _ptr(h), _ptr(y),
                                              _ptr(y64), _ptr(rstd), _ptr(r64))
    if rc != 0:
        raise ValueError("oracle_rmsnorm_fused_add_fwd rejected its arguments")
    out = {"h": h, "y": y, "rstd": rstd}
    if want64:
        out.update(y64=y64, rstd64=r64)
    return out


def bwd(dy, x, rstd, gamma, eps, x_dtype="bf16", w_dtype=None, want64=True):
    """dx (x_dtype) and dgamma (fp32) of the forward; ``rstd`` None recomputes r
    from x and eps.  With ``want64`` also dx64, dgamma64 and the error scales
    c64, dot_abs64 (per row) and dgamma_sq64 (per column)."""
    w_dtype = w_dtype or x_dtype
    x = _check_in(x, x_dtype)
    M, N = x.shape
    dy = _check_in(dy, x_dtype, (M, N))
    gamma = _check_in(gamma, w_dtype, (N,))
    if rstd is not None:
        rstd = _check_in(rstd, "f32", (M,))
    dx = np.empty((M, N), _np(x_dtype))
    dgamma = np.empty(N, np.float32)
    extra = {}
    if want64:
        extra = {"dx64": np.empty((M, N), np.float64), "dgamma64": np.empty(N, np.float64),
                 "c64": np.empty(M, np.float64), "dot_abs64": np.empty(M, np.float64),
                 "dgamma_sq64": np.empty(N, np.float64)}
    rc = _load().oracle_rmsnorm_bwd(_ptr(dy), _ptr(x), _ptr(rstd), _ptr(gamma), M, N,
                                    float(eps), DTYPE_CODES[x_dtype], DTYPE_CODES[w_dtype],
                                    _ptr(dx), _ptr(extra.get("dx64")),
                                    _ptr(extra.get("dgamma64")), _ptr(dgamma),
                                    _ptr(extra.get("c64")), _ptr(extra.get("dot_abs64")),
                                    _ptr(extra.get("dgamma_sq64")))
    if rc != 0:
        raise ValueError("oracle_rmsnorm_bwd rejected its arguments")
    out = {"dx": dx, "dgamma": dgamma}
    out.update(extra)
    return out


def fused_add_bwd(dy, h, rstd, gamma, dres, eps, x_dtype="bf16", w_dtype=None, want64=True):
    """Backward of h = residual + x, y = RMSNorm(h) * gamma: dh = dx(dy; h) + dres
    (x_dtype), the gradient of both residual and x; dgamma in fp32 and in the
    weight dtype (dgamma_w)."""
    w_dtype = w_dtype or x_dtype
    h = _check_in(h, x_dtype)
    M, N = h.shape
    dy = _check_in(dy, x_dtype, (M, N))
    dres = _check_in(dres, x_dtype, (M, N))
    gamma = _check_in(gamma, w_dtype, (N,))
    if rstd is not None:
        rstd = _check_in(rstd, "f32", (M,))
    dh = np.empty((M, N), _np(x_dtype))
    dgamma = np.empty(N, np.float32)
    dgamma_w = np.empty(N, _np(w_dtype))
    dh64 = np.empty((M, N), np.float64) if want64 else None
    dg64 = np.empty(N, np.float64) if want64 else None
    rc = _load().oracle_rmsnorm_fused_add_bwd(_ptr(dy), _ptr(h), _ptr(rstd), _ptr(gamma),
                                              _ptr(dres), M, N, float(eps), DTYPE_CODES[x_dtype],
                                              DTYPE_CODES[w_dtype], _ptr(dh), _ptr(dh64),
                                              _ptr(dg64), _ptr(dgamma), _ptr(dgamma_w))
    if rc != 0:
        raise ValueError("oracle_rmsnorm_fused_add_bwd rejected its arguments")
    out = {"dh": dh, "dgamma": dgamma, "dgamma_w": dgamma_w}
    if want64:
        out.update(dh64=dh64, dgamma64=dg64)
    return out


def fwd_strided(xbuf, x_st, x_sh, gamma, T, H, D, eps, x_dtype="bf16", w_dtype=None,
                y_st=None, y_sh=None, want64=True):
    """Forward over the [T, H, D] rows of the flat buffer `xbuf` (row (t, h) at
    element t * x_st + h * x_sh).  Returns y as a flat buffer shaped like xbuf
    with rows at t * y_st + h * y_sh (default: the x layout; elements outside
    the rows are zero), rstd [T * H], and y64 [T * H, D]."""
    w_dtype = w_dtype or x_dtype
    xbuf = np.ascontiguousarray(xbuf).reshape(-1)
    if xbuf.dtype != _np(x_dtype):
        raise TypeError("x dtype")
    gamma = _check_in(gamma, w_dtype, (D,))
    same = y_st is None and y_sh is None
    y_st = x_st if y_st is None else y_st
    y_sh = x_sh if y_sh is None else y_sh
    ylen = max((T - 1) * y_st + (H - 1) * y_sh + D, 0) if T * H else 0
    if same:
        ylen = max(ylen, xbuf.size)
    y = np.zeros(ylen, _np(x_dtype))
    rstd = np.empty(T * H, np.float32)
    y64 = np.empty((T * H, D), np.float64) if want64 else None
    rc = _load().oracle_rmsnorm_fwd_strided(_ptr(xbuf), x_st, x_sh, _ptr(gamma), T, H, D,
                                            float(eps), DTYPE_CODES[x_dtype],
                                            DTYPE_CODES[w_dtype], _ptr(y), y_st, y_sh,
                                            _ptr(y64), _ptr(rstd))
    if rc != 0:
        raise ValueError("oracle_rmsnorm_fwd_strided rejected its arguments")
    out = {"y": y, "rstd": rstd}
    if want64:
        out["y64"] = y64
    return out


# ---------------------------------------------------------------- quantised

def round_e4m3(v: float) -> int:
    """FP8 E4M3 code of a double (nearest, ties to even, saturating at 448)."""
    return int(_load().oracle_round_e4m3(float(v)))


def e4m3_to_double(code: int) -> float:
    return float(_load().oracle_e4m3_to_double(int(code)))


def round_e2m1(v: float) -> int:
    """FP4 E2M1 code (4 bits) of a double (nearest, ties to even, saturating at 6)."""
    return int(_load().oracle_round_e2m1(float(v)))


def e2m1_to_double(code: int) -> float:
    return float(_load().oracle_e2m1_to_double(int(code)))


def e4m3_values() -> np.ndarray:
    """Value of each of the 256 E4M3 codes (NaN for 0x7F and 0xFF)."""
    return np.array([e4m3_to_double(c) for c in range(256)])


def e2m1_values() -> np.ndarray:
    """Value of each of the 16 E2M1 codes."""
    return np.array([e2m1_to_double(c) for c in range(16)])


def fwd_fp8(x, gamma, eps, x_dtype="bf16", w_dtype=None, residual=None):
    """Forward (of x, or of h = residual + x) with E4M3 codes q [M, N] and one
    fp32 dequantisation scale per row.  Also scale64, v64 (the exact y / s),
    rstd and, with a residual, h."""
    w_dtype = w_dtype or x_dtype
    x = _check_in(x, x_dtype)
    M, N = x.shape
    gamma = _check_in(gamma, w_dtype, (N,))
    if residual is not None:
        residual = _check_in(residual, x_dtype, (M, N))
    h = np.empty((M, N), _np(x_dtype)) if residual is not None else None
    q = np.empty((M, N), np.uint8)
    scale = np.empty(M, np.float32)
    scale64 = np.empty(M, np.float64)
    v64 = np.empty((M, N), np.float64)
    rstd = np.empty(M, np.float32)
    rc = _load().oracle_rmsnorm_fwd_fp8(_ptr(x), _ptr(residual), _ptr(gamma), M, N, float(eps),
                                        DTYPE_CODES[x_dtype], DTYPE_CODES[w_dtype], _ptr(h),
                                        _ptr(q), _ptr(scale), _ptr(scale64), _ptr(v64),
                                        _ptr(rstd))
    if rc != 0:
        raise ValueError("oracle_rmsnorm_fwd_fp8 rejected its arguments")
    out = {"q": q, "scale": scale, "scale64": scale64, "v64": v64, "rstd": rstd}
    if h is not None:
        out["h"] = h
    return out


def fwd_nvfp4(x, gamma, gs, eps, x_dtype="bf16", w_dtype=None, residual=None):
    """Forward (of x, or of h = residual + x) with NVFP4 output: q [M, N/2]
    (two E2M1 codes per byte, even element in the low nibble) and sf [M, N/16]
    (E4M3 block scales) for the global scale gs.  Also sfv64 (the exact
    gs * amax / 6 per block), v64 (the exact y * gs / S), rstd and, with a
    residual, h."""
    w_dtype = w_dtype or x_dtype
    x = _check_in(x, x_dtype)
    M, N = x.shape
    gamma = _check_in(gamma, w_dtype, (N,))
    if residual is not None:
        residual = _check_in(residual, x_dtype, (M, N))
    h = np.empty((M, N), _np(x_dtype)) if residual is not None else None
    q = np.zeros((M, N // 2), np.uint8)
    sf = np.empty((M, N // 16), np.uint8)
    sfv64 = np.empty((M, N // 16), np.float64)
    v64 = np.empty((M, N), np.float64)
    rstd = np.empty(M, np.float32)
    rc = _load().oracle_rmsnorm_fwd_nvfp4(_ptr(x), _ptr(residual), _ptr(gamma), M, N,
                                          float(eps), float(gs), DTYPE_CODES[x_dtype],
                                          DTYPE_CODES[w_dtype], _ptr(h), _ptr(q), _ptr(sf),
                                          _ptr(sfv64), _ptr(v64), _ptr(rstd))
    if rc != 0:
        raise ValueError("oracle_rmsnorm_fwd_nvfp4 rejected its arguments")
    out = {"q": q, "sf": sf, "sfv64": sfv64, "v64": v64, "rstd": rstd}
    if h is not None:
        out["h"] = h
    return out


def unpack_e2m1(q: np.ndarray) -> np.ndarray:
    """[M, N/2] packed bytes -> [M, N] 4-bit codes (element 2k from the low nibble)."""
    q = np.asarray(q, np.uint8)
    out = np.empty(q.shape[:-1] + (q.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = q & 0xF
    out[..., 1::2] = q >> 4
    return out


# ---------------------------------------------------------------- LayerNorm

def layernorm_fwd(x, gamma, beta, eps, x_dtype="bf16", w_dtype=None):
    """(x - mean) / sqrt(var + eps) * gamma + beta per row (beta None: 0).
    Returns y (x_dtype), y64, mean / rstd (fp32) and mean64 / rstd64."""
    w_dtype = w_dtype or x_dtype
    x = _check_in(x, x_dtype)
    M, N = x.shape
    gamma = _check_in(gamma, w_dtype, (N,))
    if beta is not None:
        beta = _check_in(beta, w_dtype, (N,))
    out = {"y": np.empty((M, N), _np(x_dtype)), "y64": np.empty((M, N)),
           "mean": np.empty(M, np.float32), "rstd": np.empty(M, np.float32),
           "mean64": np.empty(M), "rstd64": np.empty(M)}
    rc = _load().oracle_layernorm_fwd(_ptr(x), _ptr(gamma), _ptr(beta), M, N, float(eps),
                                      DTYPE_CODES[x_dtype], DTYPE_CODES[w_dtype], _ptr(out["y"]),
                                      _ptr(out["y64"]), _ptr(out["mean"]), _ptr(out["rstd"]),
                                      _ptr(out["mean64"]), _ptr(out["rstd64"]))
    if rc != 0:
        raise ValueError("oracle_layernorm_fwd rejected its arguments")
    return out


def layernorm_bwd(dy, x, mean, rstd, gamma, eps, x_dtype="bf16", w_dtype=None):
    """dx (x_dtype), dgamma and dbeta (fp32) of the LayerNorm forward, with the
    saved fp32 mean and rstd (both None: recomputed from x and eps).  Also
    dx64, dgamma64, dbeta64 and dx_scale64 (per row, the size of its terms)."""
    w_dtype = w_dtype or x_dtype
    x = _check_in(x, x_dtype)
    M, N = x.shape
    dy = _check_in(dy, x_dtype, (M, N))
    gamma = _check_in(gamma, w_dtype, (N,))
    if (mean is None) != (rstd is None):
        raise ValueError("give both saved statistics (mean and rstd) or neither")
    if mean is not None:
        mean = _check_in(mean, "f32", (M,))
        rstd = _check_in(rstd, "f32", (M,))
    out = {"dx": np.empty((M, N), _np(x_dtype)), "dx64": np.empty((M, N)),
           "dgamma64": np.empty(N), "dbeta64": np.empty(N), "dgamma": np.empty(N, np.float32),
           "dbeta": np.empty(N, np.float32), "dx_scale64": np.empty(M)}
    rc = _load().oracle_layernorm_bwd(_ptr(dy), _ptr(x), _ptr(mean), _ptr(rstd), _ptr(gamma), M,
                                      N, float(eps), DTYPE_CODES[x_dtype], DTYPE_CODES[w_dtype],
                                      _ptr(out["dx"]), _ptr(out["dx64"]), _ptr(out["dgamma64"]),
                                      _ptr(out["dbeta64"]), _ptr(out["dgamma"]),
                                      _ptr(out["dbeta"]), _ptr(out["dx_scale64"]))
    if rc != 0:
        raise ValueError("oracle_layernorm_bwd rejected its arguments")
    return out
