"""CPU oracle for the autotuned matmul -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg
may import this package.  It shares no code with the library under
``matmul_selection_gb300/`` and imports nothing from it.

Contents
  * ``gemm_f64`` / ``gemm_points`` -- the plain fp64 triple loop in
    ``oracle.c`` (the definition C = A.B; see that file's header).
  * ``round_out`` -- fp64 -> output dtype, IEEE round-to-nearest-even.
  * ``key``      -- the tuning key, restated from the burn "autotune" page,
    section "tuning key: shape bucketing" (anchor, pow2 factor, stride factor,
    layout, scale, kind).
  * ``bounds``   -- the roofline time limit of the same page's section
    "roofline and the hundred thousand launches".
  * ``plan``     -- the group/priority round plan of the section
    "one op, thirty-odd candidates".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

from . import bounds, key, plan  # noqa: F401  (pure-Python restatements)

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lib = None

BF16, F16, F32 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library with gcc (OpenMP)."""
    src = os.path.join(_HERE, "oracle.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", src, "-o", tmp, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        i64, vp, dp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
        ci = ctypes.c_int
        lib.oracle_gemm_f64.argtypes = [vp, ci, i64, i64, i64, vp, ci, i64, i64, i64,
                                        dp, i64, i64, i64, i64]
        lib.oracle_gemm_f64.restype = None
        lib.oracle_gemm_points.argtypes = [vp, ci, i64, i64, i64, vp, ci, i64, i64, i64,
                                           i64, vp, i64, dp]
        lib.oracle_gemm_points.restype = None
        lib.oracle_round_bf16.argtypes = [dp, vp, i64]
        lib.oracle_round_f16.argtypes = [dp, vp, i64]
        lib.oracle_round_f32.argtypes = [dp, vp, i64]
        lib.oracle_num_threads.restype = ci
        lib.oracle_set_num_threads.argtypes = [ci]
        lib.oracle_set_num_threads.restype = None
        _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads for the following oracle calls (timing on one core or all)."""
    _load().oracle_set_num_threads(int(n))


def _strides(ld: int, trans: bool):
    """(row stride, col stride) of a logical matrix stored N (row-major) or T."""
    return (1, ld) if trans else (ld, 1)


def gemm_f64(A, B, M: int, N: int, K: int, batch: int = 1) -> np.ndarray:
    """fp64 C[batch, M, N] for operands given as ``synth.Operand``-like objects.

    Each operand needs: buf (flat numpy array), dtype, ld, trans, bstride.
    """
    lib = _load()
    a_rs, a_cs = _strides(A.ld, A.trans)
    b_rs, b_cs = _strides(B.ld, B.trans)
    C = np.zeros((batch, M, N), dtype=np.float64)
    abuf = np.ascontiguousarray(A.buf)
    bbuf = np.ascontiguousarray(B.buf)
    if C.size:
        lib.oracle_gemm_f64(abuf.ctypes.data, A.dtype, a_rs, a_cs, A.bstride,
                            bbuf.ctypes.data, B.dtype, b_rs, b_cs, B.bstride,
                            C.ctypes.data, M, N, K, batch)
    return C


def gemm_points(A, B, K: int, bij: np.ndarray) -> np.ndarray:
    """fp64 C at the given (b, i, j) points (array of shape [P, 3])."""
    lib = _load()
    a_rs, a_cs = _strides(A.ld, A.trans)
    b_rs, b_cs = _strides(B.ld, B.trans)
    pts = np.ascontiguousarray(bij, dtype=np.int64)
    out = np.zeros(pts.shape[0], dtype=np.float64)
    abuf = np.ascontiguousarray(A.buf)
    bbuf = np.ascontiguousarray(B.buf)
    if out.size:
        lib.oracle_gemm_points(abuf.ctypes.data, A.dtype, a_rs, a_cs, A.bstride,
                               bbuf.ctypes.data, B.dtype, b_rs, b_cs, B.bstride,
                               K, pts.ctypes.data, pts.shape[0], out.ctypes.data)
    return out


def round_out(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round fp64 values to the output dtype; bf16/f16 returned as uint16 bits."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    n = x.size
    if dtype == F32:
        out = np.empty(x.shape, dtype=np.float32)
        lib.oracle_round_f32(x.ctypes.data, out.ctypes.data, n)
    elif dtype == BF16:
        out = np.empty(x.shape, dtype=np.uint16)
        lib.oracle_round_bf16(x.ctypes.data, out.ctypes.data, n)
    elif dtype == F16:
        out = np.empty(x.shape, dtype=np.uint16)
        lib.oracle_round_f16(x.ctypes.data, out.ctypes.data, n)
    else:
        raise ValueError(dtype)
    return out


def decode(bits_or_vals: np.ndarray, dtype: int) -> np.ndarray:
    """Storage array (uint16 bits for bf16/f16) -> float64 values."""
    a = np.asarray(bits_or_vals)
    if dtype == F32:
        return a.astype(np.float64)
    if dtype == BF16:
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if dtype == F16:
        return a.view(np.float16).astype(np.float64) if a.dtype == np.uint16 else a.astype(np.float64)
    raise ValueError(dtype)


__all__ = ["build", "gemm_f64", "gemm_points", "round_out", "decode", "num_threads", "set_num_threads",
           "key", "bounds", "plan"]

if sys.version_info < (3, 8):  # pragma: no cover
    raise RuntimeError("python >= 3.8 required")
