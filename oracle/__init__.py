"""CPU oracle for the deterministic sum / scatter-add / scan library.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package.  The library never does, and
the two share no code: the oracle is plain C (``det_oracle.c``) plus this numpy
marshalling layer.

Every function takes numpy arrays, copies nothing it does not have to, and
returns fresh numpy arrays.  f32 inputs are computed in f32 and f64 in f64,
because the association order the library promises is defined in the input's
own precision (drjit-core pull request "Make CUDA floating-point prefix sums
deterministic", Summary: Float32 and Float64 addition).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "det_oracle.c")
_IMPL = os.path.join(_HERE, "det_oracle_impl.h")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

SCAN_INCLUSIVE = 0
SCAN_EXCLUSIVE = 1
SCAN_REVERSE = 2
SCAN_SEGMENT_RESTART = 4


def build(force: bool = False) -> str:
    """Compile the oracle with the flags its header states; returns the path."""
    stale = (not os.path.exists(_LIB_PATH)) or force or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB_PATH) for p in (_SRC, _IMPL))
    if stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True, cwd=_HERE)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32p, vp = ctypes.c_int64, ctypes.POINTER(ctypes.c_int32), ctypes.c_void_p
            for sfx in ("f32", "f64"):
                getattr(lib, f"oracle_sum_{sfx}").argtypes = [vp, i64, vp]
                getattr(lib, f"oracle_scatter_add_{sfx}").argtypes = [vp, i64, vp, vp, i64, vp, vp]
                getattr(lib, f"oracle_scatter_add_rows_{sfx}").argtypes = [vp, i64, i64, vp, i64, vp, i64, vp]
                getattr(lib, f"oracle_scan_{sfx}").argtypes = [vp, vp, i64, ctypes.c_int, vp]
                getattr(lib, f"oracle_segmented_scan_{sfx}").argtypes = [vp, vp, i64, vp, i64, ctypes.c_int]
                getattr(lib, f"oracle_scatter_sub_{sfx}").argtypes = [vp, i64, vp, vp, i64]
                getattr(lib, f"oracle_gather_rows_{sfx}").argtypes = [vp, vp, i64, i64, vp, i64, i64]
                getattr(lib, f"oracle_scatter_add_rows_ordered_{sfx}").argtypes = [vp, i64, i64, vp, i64, vp, i64, vp]
                getattr(lib, f"oracle_scatter_minmax_{sfx}").argtypes = [vp, i64, vp, vp, i64, ctypes.c_int]
            lib.oracle_scan_i32.argtypes = [vp, vp, i64, ctypes.c_int, vp]
            lib.oracle_slot_alloc.argtypes = [vp, i64, vp, i64, vp, i64, vp]
            lib.oracle_scan_chunk_elems.restype = i64
            lib.oracle_scan_chunk_elems.argtypes = [ctypes.c_int]
            lib.oracle_scan_lane_elems.restype = i64
            lib.oracle_scan_lane_elems.argtypes = [ctypes.c_int]
            _ = i32p
            _lib = lib
    return _lib


def _sfx(dtype) -> str:
    dtype = np.dtype(dtype)
    if dtype == np.float32:
        return "f32"
    if dtype == np.float64:
        return "f64"
    raise TypeError(f"oracle supports float32/float64, got {dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: bad argument (code {rc})")


def scan_chunk_elems(dtype) -> int:
    """Elements per scan chunk (32 virtual warps x 32 lanes x E)."""
    return int(_load().oracle_scan_chunk_elems(1 if _sfx(dtype) == "f64" else 0))


def scan_lane_elems(dtype) -> int:
    return int(_load().oracle_scan_lane_elems(1 if _sfx(dtype) == "f64" else 0))


def det_sum(x: np.ndarray):
    x = np.ascontiguousarray(x)
    sfx = _sfx(x.dtype)
    out = np.zeros(1, dtype=x.dtype)
    _check(getattr(_load(), f"oracle_sum_{sfx}")(_ptr(x), x.size, _ptr(out)), "sum")
    return out[0]


def det_scatter_add(out: np.ndarray, bins: np.ndarray, values: np.ndarray):
    """Returns (new_out, perm, seg_offsets); ``out`` itself is not modified."""
    values = np.ascontiguousarray(values)
    sfx = _sfx(values.dtype)
    res = np.array(out, dtype=values.dtype, copy=True)
    bins = np.ascontiguousarray(bins, dtype=np.int32)
    n, m = values.size, res.size
    if bins.size != n:
        raise ValueError("bins and values differ in length")
    valid = int(np.count_nonzero((bins >= 0) & (bins < m)))
    perm = np.empty(valid, dtype=np.int32)
    seg = np.empty(m + 1, dtype=np.int32)
    rc = getattr(_load(), f"oracle_scatter_add_{sfx}")(_ptr(res), m, _ptr(bins), _ptr(values), n,
                                                         _ptr(perm), _ptr(seg))
    _check(rc, "scatter_add")
    return res, perm, seg


def det_scatter_add_rows(dst: np.ndarray, idx: np.ndarray, src: np.ndarray, row_offset: int = 0):
    """Returns (new_dst, prev); ``dst`` itself is not modified."""
    src = np.ascontiguousarray(src)
    sfx = _sfx(src.dtype)
    res = np.array(dst, dtype=src.dtype, copy=True, order="C")
    if res.ndim != 2 or src.ndim != 2 or res.shape[1] != src.shape[1]:
        raise ValueError("dst and src must be 2-D with equal row length")
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    if idx.size != src.shape[0]:
        raise ValueError("idx must have one entry per source row")
    prev = np.empty_like(src)
    rc = getattr(_load(), f"oracle_scatter_add_rows_{sfx}")(
        _ptr(res), res.shape[0], res.shape[1], _ptr(idx), int(row_offset), _ptr(src), src.shape[0], _ptr(prev))
    _check(rc, "scatter_add_rows")
    return res, prev


def det_scan(x: np.ndarray, flags: int = SCAN_INCLUSIVE):
    """Returns (y, total)."""
    x = np.ascontiguousarray(x)
    sfx = _sfx(x.dtype)
    y = np.empty_like(x)
    total = np.zeros(1, dtype=x.dtype)
    _check(getattr(_load(), f"oracle_scan_{sfx}")(_ptr(x), _ptr(y), x.size, int(flags), _ptr(total)), "scan")
    return y, total[0]


def det_segmented_scan(x: np.ndarray, offsets: np.ndarray, flags: int = SCAN_INCLUSIVE):
    x = np.ascontiguousarray(x)
    sfx = _sfx(x.dtype)
    offsets = np.ascontiguousarray(offsets, dtype=np.int64)
    y = np.empty_like(x)
    rc = getattr(_load(), f"oracle_segmented_scan_{sfx}")(_ptr(x), _ptr(y), x.size, _ptr(offsets),
                                                            offsets.size - 1, int(flags))
    _check(rc, "segmented_scan")
    return y


def det_scatter_sub(out: np.ndarray, bins: np.ndarray, values: np.ndarray):
    """out[b] + PT(-values of group b); returns the new out (``out`` unmodified)."""
    values = np.ascontiguousarray(values)
    sfx = _sfx(values.dtype)
    res = np.array(out, dtype=values.dtype, copy=True)
    bins = np.ascontiguousarray(bins, dtype=np.int32)
    if bins.size != values.size:
        raise ValueError("bins and values differ in length")
    _check(getattr(_load(), f"oracle_scatter_sub_{sfx}")(_ptr(res), res.size, _ptr(bins), _ptr(values), values.size),
           "scatter_sub")
    return res


def _scatter_minmax(out, bins, values, is_max):
    values = np.ascontiguousarray(values)
    sfx = _sfx(values.dtype)
    res = np.array(out, dtype=values.dtype, copy=True)
    bins = np.ascontiguousarray(bins, dtype=np.int32)
    if bins.size != values.size:
        raise ValueError("bins and values differ in length")
    _check(getattr(_load(), f"oracle_scatter_minmax_{sfx}")(_ptr(res), res.size, _ptr(bins), _ptr(values),
                                                            values.size, int(is_max)), "scatter_minmax")
    return res


def det_scatter_min(out: np.ndarray, bins: np.ndarray, values: np.ndarray):
    """IEEE 754-2019 minimum of the old value and each group; returns the new out."""
    return _scatter_minmax(out, bins, values, False)


def det_scatter_max(out: np.ndarray, bins: np.ndarray, values: np.ndarray):
    """IEEE 754-2019 maximum of the old value and each group; returns the new out."""
    return _scatter_minmax(out, bins, values, True)


def det_scan_i32(x: np.ndarray, exclusive: bool = False):
    """int32 prefix sum (wrapping modulo 2^32); returns (y, total)."""
    x = np.ascontiguousarray(x, dtype=np.int32)
    y = np.empty_like(x)
    total = np.zeros(1, dtype=np.int32)
    _check(_load().oracle_scan_i32(_ptr(x), _ptr(y), x.size, 1 if exclusive else 0, _ptr(total)), "scan_i32")
    return y, int(total[0])


def det_slot_alloc(counter: np.ndarray, index: np.ndarray, count: np.ndarray | None = None, index_offset: int = 0):
    """Thread-order slot allocation; returns (slots, new_counter) (``counter`` unmodified)."""
    ctr = np.array(counter, dtype=np.int32, copy=True)
    index = np.ascontiguousarray(index, dtype=np.int32)
    cnt = None if count is None else np.ascontiguousarray(count, dtype=np.int32)
    if cnt is not None and cnt.size != index.size:
        raise ValueError("count must have one entry per record")
    slots = np.empty(index.size, dtype=np.int32)
    _check(_load().oracle_slot_alloc(_ptr(ctr), ctr.size, _ptr(index), int(index_offset), _ptr(cnt), index.size,
                                     _ptr(slots)), "slot_alloc")
    return slots, ctr


def det_scatter_add_rows_ordered(dst: np.ndarray, idx: np.ndarray, src: np.ndarray, row_offset: int = 0):
    """Row scatter applied one source row at a time in ascending order; returns (new_dst, prev)."""
    src = np.ascontiguousarray(src)
    sfx = _sfx(src.dtype)
    res = np.array(dst, dtype=src.dtype, copy=True, order="C")
    if res.ndim != 2 or src.ndim != 2 or res.shape[1] != src.shape[1]:
        raise ValueError("dst and src must be 2-D with equal row length")
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    if idx.size != src.shape[0]:
        raise ValueError("idx must have one entry per source row")
    prev = np.empty_like(src)
    rc = getattr(_load(), f"oracle_scatter_add_rows_ordered_{sfx}")(
        _ptr(res), res.shape[0], res.shape[1], _ptr(idx), int(row_offset), _ptr(src), src.shape[0], _ptr(prev))
    _check(rc, "scatter_add_rows_ordered")
    return res, prev


def det_gather_rows(src: np.ndarray, idx: np.ndarray, row_offset: int = 0):
    """out[i] = src[idx[i] + row_offset] (+0.0 rows for indices outside src); src is 1-D or 2-D."""
    src = np.ascontiguousarray(src)
    sfx = _sfx(src.dtype)
    src2 = src.reshape(src.shape[0], -1) if src.ndim != 1 else src.reshape(-1, 1)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    out = np.empty((idx.size, src2.shape[1]), dtype=src.dtype)
    rc = getattr(_load(), f"oracle_gather_rows_{sfx}")(_ptr(out), _ptr(src2), src2.shape[0], src2.shape[1],
                                                        _ptr(idx), int(row_offset), idx.size)
    _check(rc, "gather_rows")
    return out.reshape(-1) if src.ndim == 1 else out
