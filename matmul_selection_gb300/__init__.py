"""Python binding of the GB300 autotuned matmul C ABI (include/mm.h).

Argument marshalling only: every entry point forwards to the shared library
built from ``csrc/`` (``_build/libmm_gb300.so``); nothing here computes.  The
names are the C names.  Data arguments accept raw device addresses (int) or
objects with ``data_ptr()`` (torch tensors); ``stream`` accepts an int
handle, a ``torch.cuda.Stream`` or None (legacy default stream).

Importing the package loads the library and fails loudly when it has not
been built (``python matmul_selection_gb300/build.py``).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmm_gb300.so")

# status codes
MM_OK = 0
MM_ERR_INVALID_ARG = 1
MM_ERR_UNSUPPORTED = 2
MM_ERR_CUDA = 3
MM_ERR_NO_VALID_CANDIDATE = 4
MM_ERR_CACHE_VALIDATION = 5
MM_ERR_IO = 6
MM_ERR_TIMEOUT = 7
MM_ERR_NOT_FOUND = 8

MM_BF16, MM_F16, MM_F32 = 0, 1, 2
MM_NN, MM_NT, MM_TN, MM_TT = 0, 1, 2, 3
LAYOUTS = {"NN": MM_NN, "NT": MM_NT, "TN": MM_TN, "TT": MM_TT}


class mm_dtypes(ctypes.Structure):
    _fields_ = [("a", ctypes.c_int32), ("b", ctypes.c_int32), ("c", ctypes.c_int32)]


class mm_batch(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("stride_a", ctypes.c_int64),
                ("stride_b", ctypes.c_int64), ("stride_c", ctypes.c_int64)]


class mm_key(ctypes.Structure):
    _fields_ = [("bytes", ctypes.c_uint8 * 64)]


class mm_stats(ctypes.Structure):
    _fields_ = [("calls", ctypes.c_uint64), ("hits", ctypes.c_uint64),
                ("misses", ctypes.c_uint64), ("tunes", ctypes.c_uint64),
                ("launches", ctypes.c_uint64), ("bench_launches", ctypes.c_uint64),
                ("last_tune_ms", ctypes.c_double), ("total_tune_ms", ctypes.c_double)]


class MMError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"mm status {status}: {message}")
        self.status = status


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python matmul_selection_gb300/build.py` (needs nvcc)")
_lib = ctypes.CDLL(LIB_PATH)

_i64, _i32, _vp, _cp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_char_p
_P32 = ctypes.POINTER(ctypes.c_int32)
_sig = {
    "mm_tune_key": (_i32, [_i64, _i64, _i64, _i64, _i64, _i64, mm_dtypes, ctypes.c_int,
                           ctypes.POINTER(mm_batch), ctypes.POINTER(mm_key), ctypes.c_char_p,
                           ctypes.c_size_t]),
    "mm_autotune_execute": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _i64, mm_dtypes,
                                   ctypes.c_int, ctypes.POINTER(mm_batch), _vp]),
    "mm_autotune_execute_host": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _i64,
                                        mm_dtypes, ctypes.c_int, ctypes.POINTER(mm_batch), _vp]),
    "mm_cache_load": (_i32, [_cp]),
    "mm_cache_save": (_i32, [_cp]),
    "mm_tune_file": (_i32, [_cp, ctypes.POINTER(ctypes.c_int)]),
    "mm_cache_clear": (_i32, []),
    "mm_cache_size": (_i64, []),
    "mm_candidate_count": (_i32, []),
    "mm_candidate_name": (_cp, [_i32]),
    "mm_candidate_launches": (ctypes.c_uint64, [_i32]),
    "mm_candidate_checksum": (ctypes.c_uint64, []),
    "mm_execute_candidate": (_i32, [_i32, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _i64,
                                    mm_dtypes, ctypes.c_int, ctypes.POINTER(mm_batch), _vp]),
    "mm_lookup": (_i32, [ctypes.POINTER(mm_key), _P32]),
    "mm_plan": (_i32, [_i64, _i64, _i64, _i64, _i64, _i64, mm_dtypes, ctypes.c_int,
                       ctypes.POINTER(mm_batch), _i32, _P32, _P32, _P32, _P32, _P32, _P32]),
    "mm_group_name": (_cp, [_i32]),
    "mm_default_candidate": (_i32, [_i64, _i64, _i64, _i64, _i64, _i64, mm_dtypes, ctypes.c_int,
                                    ctypes.POINTER(mm_batch)]),
    "mm_roofline_limit_ns": (ctypes.c_double, [ctypes.c_double] * 6),
    "mm_device_peaks": (_i32, [ctypes.POINTER(ctypes.c_double)] * 3),
    "mm_set_option": (_i32, [_cp, _cp]),
    "mm_get_option": (_i32, [_cp, ctypes.c_char_p, ctypes.c_size_t]),
    "mm_get_stats": (_i32, [ctypes.POINTER(mm_stats)]),
    "mm_reset_stats": (None, []),
    "mm_last_error": (_cp, []),
    "mm_version": (_cp, []),
    "mm_shutdown": (None, []),
    "mm_splitk_gemm_noalloc": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _i64,
                                      mm_dtypes, ctypes.c_int, _vp]),
    "mm_splitk_gemm_noalloc_status": (_i32, [_vp]),
}
for _name, (_res, _args) in _sig.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_sig)


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):  # numpy array (host entry point)
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)}")


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream  # torch.cuda.Stream


def _dt(dt):
    if isinstance(dt, mm_dtypes):
        return dt
    a, b, c = dt
    return mm_dtypes(a, b, c)


def _layout(layout):
    return LAYOUTS[layout] if isinstance(layout, str) else int(layout)


def _batch(batch):
    if batch is None:
        return None
    if isinstance(batch, mm_batch):
        return ctypes.byref(batch)
    return ctypes.byref(mm_batch(*batch))


def mm_last_error() -> str:
    return _lib.mm_last_error().decode()


def mm_version() -> str:
    return _lib.mm_version().decode()


def check(status: int) -> int:
    """Raise MMError for a non-OK status (with the library's message)."""
    if status != MM_OK:
        raise MMError(status, mm_last_error())
    return status


def mm_tune_key(M, N, K, lda, ldb, ldc, dtypes, layout, batch=None):
    """Returns (status, key bytes, canonical text)."""
    k = mm_key()
    buf = ctypes.create_string_buffer(512)
    st = _lib.mm_tune_key(M, N, K, lda, ldb, ldc, _dt(dtypes), _layout(layout), _batch(batch),
                          ctypes.byref(k), buf, 512)
    return st, bytes(k.bytes), buf.value.decode()


def mm_autotune_execute(lhs, rhs, out, M, N, K, lda, ldb, ldc, dtypes, layout, batch=None,
                        stream=None):
    return _lib.mm_autotune_execute(_ptr(lhs), _ptr(rhs), _ptr(out), M, N, K, lda, ldb, ldc,
                                    _dt(dtypes), _layout(layout), _batch(batch), _stream(stream))


def mm_autotune_execute_host(lhs, rhs, out, M, N, K, lda, ldb, ldc, dtypes, layout, batch=None,
                             stream=None):
    return _lib.mm_autotune_execute_host(_ptr(lhs), _ptr(rhs), _ptr(out), M, N, K, lda, ldb, ldc,
                                         _dt(dtypes), _layout(layout), _batch(batch),
                                         _stream(stream))


def mm_execute_candidate(index, lhs, rhs, out, M, N, K, lda, ldb, ldc, dtypes, layout,
                         batch=None, stream=None):
    return _lib.mm_execute_candidate(index, _ptr(lhs), _ptr(rhs), _ptr(out), M, N, K, lda, ldb,
                                     ldc, _dt(dtypes), _layout(layout), _batch(batch),
                                     _stream(stream))


def mm_cache_load(path=None):
    return _lib.mm_cache_load(path.encode() if path else None)


def mm_tune_file(path):
    """Tune every problem recorded in `path` by the record_untuned option;
    returns (status, number tuned)."""
    n = ctypes.c_int(0)
    st = _lib.mm_tune_file(path.encode(), ctypes.byref(n))
    return st, n.value


def mm_cache_save(path=None):
    return _lib.mm_cache_save(path.encode() if path else None)


def mm_cache_clear():
    return _lib.mm_cache_clear()


def mm_cache_size():
    return _lib.mm_cache_size()


def mm_candidate_count():
    return _lib.mm_candidate_count()


def mm_candidate_name(i):
    r = _lib.mm_candidate_name(i)
    return r.decode() if r is not None else None


def mm_candidate_launches(i):
    return _lib.mm_candidate_launches(i)


def mm_candidate_checksum():
    return _lib.mm_candidate_checksum()


def candidate_names():
    return [mm_candidate_name(i) for i in range(mm_candidate_count())]


def mm_lookup(key: bytes):
    k = mm_key()
    ctypes.memmove(k.bytes, key, 64)
    idx = ctypes.c_int32(-1)
    st = _lib.mm_lookup(ctypes.byref(k), ctypes.byref(idx))
    return st, idx.value


def mm_plan(M, N, K, lda, ldb, ldc, dtypes, layout, batch=None, cap=256):
    """Returns a list of dicts {cand, group, tier, supported, group_prio, prio}."""
    arrs = [(ctypes.c_int32 * cap)() for _ in range(6)]
    n = _lib.mm_plan(M, N, K, lda, ldb, ldc, _dt(dtypes), _layout(layout), _batch(batch), cap,
                     *arrs)
    if n < 0:
        raise MMError(MM_ERR_INVALID_ARG, mm_last_error())
    keys = ("cand", "group", "tier", "supported", "group_prio", "prio")
    return [{k: arrs[j][i] for j, k in enumerate(keys)} for i in range(n)]


def mm_default_candidate(M, N, K, lda, ldb, ldc, dtypes, layout, batch=None):
    return _lib.mm_default_candidate(M, N, K, lda, ldb, ldc, _dt(dtypes), _layout(layout),
                                     _batch(batch))


def mm_group_name(g):
    r = _lib.mm_group_name(g)
    return r.decode() if r is not None else None


def mm_device_peaks():
    """(status, bf16 ops/s, bytes/s, launch ns) of the current device."""
    v = [ctypes.c_double(0) for _ in range(3)]
    st = _lib.mm_device_peaks(*[ctypes.byref(x) for x in v])
    return (st,) + tuple(x.value for x in v)


def mm_roofline_limit_ns(ops, peak_ops_per_s, nbytes, peak_bytes_per_s, threshold, launch_ns):
    return _lib.mm_roofline_limit_ns(ops, peak_ops_per_s, nbytes, peak_bytes_per_s, threshold,
                                     launch_ns)


def mm_set_option(name, value):
    return _lib.mm_set_option(name.encode(), str(value).encode())


def mm_get_option(name):
    buf = ctypes.create_string_buffer(1024)
    st = _lib.mm_get_option(name.encode(), buf, 1024)
    return st, buf.value.decode()


def mm_get_stats():
    s = mm_stats()
    _lib.mm_get_stats(ctypes.byref(s))
    return {f: getattr(s, f) for f, _ in mm_stats._fields_}


def mm_reset_stats():
    _lib.mm_reset_stats()


def mm_shutdown():
    _lib.mm_shutdown()


def mm_splitk_gemm_noalloc(lhs, rhs, out, M, N, K, lda, ldb, ldc, dtypes, layout, stream=None):
    """Split-K GEMM into the library's fixed workspace: no device allocation."""
    return _lib.mm_splitk_gemm_noalloc(_ptr(lhs), _ptr(rhs), _ptr(out), M, N, K, lda, ldb, ldc,
                                       _dt(dtypes), _layout(layout), _stream(stream))


def mm_splitk_gemm_noalloc_status(stream=None):
    """Synchronise `stream` and report (and clear) a bounded wait that gave up
    in a no-allocation call since the previous query."""
    return _lib.mm_splitk_gemm_noalloc_status(_stream(stream))


def library_handle():
    return _lib
