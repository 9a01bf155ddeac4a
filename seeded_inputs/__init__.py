"""Seeded synthetic inputs shared by the tests and the bench.

This module draws random tensors (the definition of the streams is in
``generator.c``) and describes the workloads; it computes nothing of the
normalisation itself.  bf16 tensors are returned as ``numpy.uint16`` arrays of
bit patterns, fp32 tensors as ``numpy.float32``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .workloads import TENSOR_IDS, WORKLOADS, Workload, tensor_recipes  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "generator.c")
_LIB = os.path.join(_HERE, "_libseeded_inputs.so")
_lock = threading.Lock()
_lib = None

DTYPE_CODES = {"f32": 0, "bf16": 1}
DIST_CODES = {"normal": 0, "uniform": 1}


def build(force: bool = False) -> str:
    """Compile generator.c into a shared library next to it (gcc, -O2)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = f"{_LIB}.{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-D_DEFAULT_SOURCE", _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.gen_fill.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int,
                                     ctypes.c_double, ctypes.c_double, ctypes.c_int64,
                                     ctypes.c_int, ctypes.c_void_p, ctypes.c_int]
            lib.gen_fill.restype = ctypes.c_int
            lib.gen_outlier_positions.argtypes = [ctypes.c_uint64, ctypes.c_uint64,
                                                  ctypes.c_int64, ctypes.c_int64,
                                                  ctypes.c_void_p]
            lib.gen_outlier_positions.restype = ctypes.c_int
            lib.gen_apply_outliers.argtypes = [ctypes.c_uint64, ctypes.c_uint64,
                                               ctypes.c_double, ctypes.c_double,
                                               ctypes.c_double, ctypes.c_void_p,
                                               ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
            lib.gen_apply_outliers.restype = ctypes.c_int
            lib.gen_uniform_at.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
            lib.gen_uniform_at.restype = ctypes.c_double
            lib.gen_normal_at.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
            lib.gen_normal_at.restype = ctypes.c_double
            lib.gen_splitmix64_next.argtypes = [ctypes.c_uint64]
            lib.gen_splitmix64_next.restype = ctypes.c_uint64
            _lib = lib
    return _lib


def _np_dtype(dtype: str):
    return np.float32 if dtype == "f32" else np.uint16


def outlier_positions(n: int, k: int, *, seed: int, tensor_id: int) -> np.ndarray:
    """k distinct positions of [0, n), ascending, uniform (Floyd's sampling)."""
    pos = np.empty(k, dtype=np.int64)
    rc = _load().gen_outlier_positions(seed, tensor_id, n, k, pos.ctypes.data)
    if rc != 0:
        raise ValueError(f"outlier_positions failed (n={n}, k={k})")
    return pos


def fill(shape, *, seed: int, tensor_id: int, dist: str = "normal", p0: float = 0.0,
         p1: float = 1.0, dtype: str = "bf16", outlier_fraction: float = 0.0,
         outlier_scale: float = 1.0, threads: int = 0) -> np.ndarray:
    """Draw one tensor.  normal: p0 = mean, p1 = std; uniform: [p0, p1).

    With ``outlier_fraction`` f > 0, floor(f * size) distinct positions get
    ``p0 + p1 * outlier_scale * z`` instead of ``p0 + p1 * z`` (normal only).
    """
    shape = tuple(int(s) for s in np.atleast_1d(shape)) if not isinstance(shape, int) else (shape,)
    n = int(np.prod(shape)) if shape else 1
    out = np.empty(shape, dtype=_np_dtype(dtype))
    lib = _load()
    rc = lib.gen_fill(seed, tensor_id, DIST_CODES[dist], p0, p1, n, DTYPE_CODES[dtype],
                      out.ctypes.data, threads)
    if rc != 0:
        raise ValueError("gen_fill failed")
    if outlier_fraction > 0.0:
        if dist != "normal":
            raise ValueError("outliers are defined for normal tensors only")
        k = int(np.floor(outlier_fraction * n + 1e-9))
        pos = outlier_positions(n, k, seed=seed, tensor_id=tensor_id)
        rc = lib.gen_apply_outliers(seed, tensor_id, p0, p1, outlier_scale, pos.ctypes.data,
                                    k, DTYPE_CODES[dtype], out.ctypes.data)
        if rc != 0:
            raise ValueError("gen_apply_outliers failed")
    return out


def uniform_at(seed: int, tensor_id: int, i: int) -> float:
    return _load().gen_uniform_at(seed, tensor_id, i)


def normal_at(seed: int, tensor_id: int, i: int) -> float:
    return _load().gen_normal_at(seed, tensor_id, i)


def splitmix64_next(state: int) -> int:
    return _load().gen_splitmix64_next(state)


def make_inputs(wl: "Workload", rows: int | None = None) -> dict:
    """All input tensors of a workload, keyed by name (x, residual, gamma, dy, beta).

    ``rows`` limits the activations to the first ``rows`` rows (the streams are
    counter based, so those rows are identical to the full tensor's)."""
    m = wl.M if rows is None else min(rows, wl.M)
    out = {}
    for name, rec in tensor_recipes(wl).items():
        rec = dict(rec)
        shape = rec.pop("shape", None)
        if shape is None:
            shape = (wl.N,) if name in ("gamma", "beta") else (m, wl.N)
        elif rows is not None:
            shape = (min(rows, shape[0]),) + tuple(shape[1:])
        out[name] = fill(shape, seed=wl.seed, tensor_id=TENSOR_IDS[name], **rec)
    return out
