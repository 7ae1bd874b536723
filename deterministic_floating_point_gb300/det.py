"""Thin Python binding over the C ABI of ``libdet.so`` (see ``include/det.h``).

Argument marshalling only: tensors become raw device pointers and sizes, the
current torch stream becomes the ``stream`` argument, and a workspace of the
size the library asks for is taken from torch's allocator when the caller
does not pass one.  Every step of every operation runs in the library's CUDA
kernels; there is no fallback.  If ``libdet.so`` is missing or cannot be
loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdet.so")

F32, F64 = 0, 1
OK = 0
ERR_CUDA = 6   # DET_ERR_CUDA: a CUDA call or launch failed (detail: det_last_cuda_error)
SCAN_INCLUSIVE, SCAN_EXCLUSIVE, SCAN_REVERSE = 0, 1, 2
SCAN_SEGMENT_RESTART = 4   # det_segmented_scan: each segment scanned as det_scan of the segment alone
SCAN_LANE_ELEMS = {torch.float32: 32, torch.float64: 16}
SCAN_CHUNK = {torch.float32: 32768, torch.float64: 16384}

_lock = threading.Lock()
_lib = None

_i64, _sz, _vp, _int = ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int
_SIGNATURES = {
    "det_sum_workspace_bytes": (_sz, [_i64, _int]),
    "det_sum": (_int, [_vp, _i64, _int, _vp, _vp, _sz, _int, _vp]),
    "det_sum_noalloc": (_int, [_vp, _i64, _int, _vp, _int, _vp]),
    "det_scatter_add_workspace_bytes": (_sz, [_i64, _i64, _int]),
    "det_scatter_add": (_int, [_vp, _i64, _vp, _vp, _i64, _int, _vp, _vp, _vp, _sz, _int, _vp]),
    "det_scatter_add_rows_workspace_bytes": (_sz, [_i64, _i64, _i64, _int]),
    "det_scatter_add_rows": (_int, [_vp, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _int, _vp, _sz, _int, _vp]),
    "det_scan_workspace_bytes": (_sz, [_i64, _int]),
    "det_scan": (_int, [_vp, _vp, _i64, _int, _int, _vp, _vp, _sz, _int, _vp]),
    "det_segmented_scan_workspace_bytes": (_sz, [_i64, _i64, _int]),
    "det_segmented_scan": (_int, [_vp, _vp, _i64, _vp, _i64, _int, _int, _vp, _sz, _int, _vp]),
    "det_scatter_add_rows_ordered": (_int, [_vp, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _int, _vp, _sz, _int, _vp]),
    "det_scatter_add_vec_workspace_bytes": (_sz, [_i64, _i64, _i64, _int]),
    "det_scatter_add_vec": (_int, [_vp, _i64, _i64, _vp, _vp, _i64, _int, _vp, _sz, _int, _vp]),
    "det_gather_rows": (_int, [_vp, _vp, _i64, _i64, _vp, _i64, _i64, _int, _int, _vp]),
    "det_scatter_sub": (_int, [_vp, _i64, _vp, _vp, _i64, _int, _vp, _vp, _vp, _sz, _int, _vp]),
    "det_scatter_minmax_workspace_bytes": (_sz, [_i64, _int]),
    "det_scatter_min": (_int, [_vp, _i64, _vp, _vp, _i64, _int, _vp, _sz, _int, _vp]),
    "det_scatter_max": (_int, [_vp, _i64, _vp, _vp, _i64, _int, _vp, _sz, _int, _vp]),
    "det_scan_i32_workspace_bytes": (_sz, [_i64]),
    "det_scan_i32": (_int, [_vp, _vp, _i64, _int, _vp, _vp, _sz, _int, _vp]),
    "det_slot_alloc_workspace_bytes": (_sz, [_i64, _i64]),
    "det_slot_alloc": (_int, [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _sz, _int, _vp]),
    "det_read_status": (_int, [_vp, _vp, ctypes.POINTER(_int)]),
    "det_status_string": (ctypes.c_char_p, [_int]),
    "det_last_cuda_error": (ctypes.c_char_p, []),
    "det_profile_set_events": (_int, [_vp, _int]),
    "det_profile_event_count": (_int, []),
    "det_profile_event_name": (ctypes.c_char_p, [_int]),
    "det_launch_count": (ctypes.c_ulonglong, []),
    "det_test_scan_withhold": (_int, [_i64, ctypes.c_uint64]),
    "det_profile_add_rate_probe": (_int, [_int, _int, _vp, _vp, ctypes.POINTER(ctypes.c_ulonglong)]),
    "det_atomic_sum": (_int, [_vp, _i64, _int, _vp, _vp]),
    "det_atomic_scatter_add": (_int, [_vp, _i64, _vp, _vp, _i64, _int, _vp]),
    "det_atomic_scatter_add_rows": (_int, [_vp, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _int, _vp]),
    "det_atomic_slot_alloc": (_int, [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp]),
    "det_dlb_scan_workspace_bytes": (_sz, [_i64, _int]),
    "det_dlb_scan": (_int, [_vp, _vp, _i64, _int, _vp, _sz, _vp]),
}


class DetError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        detail = ""
        if code == ERR_CUDA:
            try:
                detail = " [" + lib().det_last_cuda_error().decode() + "]"
            except Exception:  # pragma: no cover - only when the library is absent
                pass
        super().__init__(f"{what}: {status_string(code)} (code {code}){detail}")


def lib():
    """The loaded ``libdet.so``; raises if it has not been built."""
    global _lib
    if _lib is not None:   # loaded: no lock on the per-call path
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                                   "(python -c 'import __graft_entry__ as g; g.build()')")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(handle, name, None)
                if fn is None:
                    continue
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def exported_symbols():
    h = lib()
    return {name for name in _SIGNATURES if getattr(h, name, None) is not None}


def status_string(code: int) -> str:
    try:
        return lib().det_status_string(int(code)).decode()
    except Exception:  # pragma: no cover - only when the library is absent
        return "unknown"


def _code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.float64:
        return F64
    raise TypeError(f"det supports float32 and float64 tensors, got {t.dtype}")


def _dev(t: torch.Tensor, name: str) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def workspace(nbytes: int, device) -> torch.Tensor:
    """A device byte buffer with a 256-byte aligned start of at least nbytes."""
    buf = torch.empty(int(nbytes) + 256, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % 256
    return buf[off:off + int(nbytes)]


def _ws(ws, nbytes, device):
    if ws is None:
        ws = workspace(nbytes, device)
    if ws.numel() < nbytes:
        raise DetError(4, "workspace")
    return ws


def _check(rc: int, what: str):
    if rc != OK:
        raise DetError(rc, what)


def read_status(ws: torch.Tensor, stream=None) -> int:
    st = _int(0)
    _check(lib().det_read_status(_ptr(ws), _stream(stream), ctypes.byref(st)), "det_read_status")
    return int(st.value)


# ---------------------------------------------------------------------------


def det_sum(x: torch.Tensor, out: torch.Tensor | None = None, *, block_threads: int = 0,
            workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[0] = pairwise tree sum of x (see det.h)."""
    _dev(x, "x")
    code = _code(x)
    if out is None:
        out = torch.empty(1, dtype=x.dtype, device=x.device)
    n = x.numel()
    nbytes = lib().det_sum_workspace_bytes(n, code)
    ws = _ws(workspace, nbytes, x.device)
    _check(lib().det_sum(_ptr(x), n, code, _ptr(out), _ptr(ws), ws.numel(), block_threads,
                         _stream(stream)), "det_sum")
    return out


def det_scatter_add(out: torch.Tensor, bins: torch.Tensor, values: torch.Tensor, *,
                    perm_out: torch.Tensor | None = None, seg_offsets_out: torch.Tensor | None = None,
                    block_threads: int = 0, workspace: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """out[bins[i]] += values[i], in a fixed order (see det.h); returns out."""
    _dev(out, "out"), _dev(bins, "bins"), _dev(values, "values")
    code = _code(values)
    if out.dtype != values.dtype or bins.dtype != torch.int32:
        raise TypeError("out must match values' dtype and bins must be int32")
    n, m = values.numel(), out.numel()
    if bins.numel() != n:
        raise ValueError("bins and values differ in length")
    nbytes = lib().det_scatter_add_workspace_bytes(n, m, code)
    ws = _ws(workspace, nbytes, values.device)
    _check(lib().det_scatter_add(_ptr(out), m, _ptr(bins), _ptr(values), n, code, _ptr(perm_out),
                                 _ptr(seg_offsets_out), _ptr(ws), ws.numel(), block_threads,
                                 _stream(stream)), "det_scatter_add")
    return out


def det_gather_rows(src: torch.Tensor, idx: torch.Tensor, out: torch.Tensor | None = None, *, row_offset: int = 0,
                    block_threads: int = 0, stream=None) -> torch.Tensor:
    """out[i] = src[idx[i] + row_offset] (zeros outside src); src is 1-D (scalars) or 2-D (rows)."""
    _dev(src, "src"), _dev(idx, "idx")
    code = _code(src)
    if idx.dtype != torch.int32:
        raise TypeError("idx must be int32")
    W = 1 if src.dim() == 1 else src.shape[1]
    n = idx.numel()
    if out is None:
        out = torch.empty((n,) if src.dim() == 1 else (n, W), dtype=src.dtype, device=src.device)
    _check(lib().det_gather_rows(_ptr(out), _ptr(src), src.shape[0], W, _ptr(idx), int(row_offset), n, code,
                                 block_threads, _stream(stream)), "det_gather_rows")
    return out


def det_scatter_sub(out: torch.Tensor, bins: torch.Tensor, values: torch.Tensor, *,
                    perm_out: torch.Tensor | None = None, seg_offsets_out: torch.Tensor | None = None,
                    block_threads: int = 0, workspace: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """out[bins[i]] -= values[i]: the values negated and added in det_scatter_add's order; returns out."""
    _dev(out, "out"), _dev(bins, "bins"), _dev(values, "values")
    code = _code(values)
    if out.dtype != values.dtype or bins.dtype != torch.int32:
        raise TypeError("out must match values' dtype and bins must be int32")
    n, m = values.numel(), out.numel()
    if bins.numel() != n:
        raise ValueError("bins and values differ in length")
    nbytes = lib().det_scatter_add_workspace_bytes(n, m, code)
    ws = _ws(workspace, nbytes, values.device)
    _check(lib().det_scatter_sub(_ptr(out), m, _ptr(bins), _ptr(values), n, code, _ptr(perm_out),
                                 _ptr(seg_offsets_out), _ptr(ws), ws.numel(), block_threads,
                                 _stream(stream)), "det_scatter_sub")
    return out


def _scatter_minmax(fn, out, bins, values, block_threads, workspace, stream):
    _dev(out, "out"), _dev(bins, "bins"), _dev(values, "values")
    code = _code(values)
    if out.dtype != values.dtype or bins.dtype != torch.int32:
        raise TypeError("out must match values' dtype and bins must be int32")
    n, m = values.numel(), out.numel()
    if bins.numel() != n:
        raise ValueError("bins and values differ in length")
    ws = _ws(workspace, lib().det_scatter_minmax_workspace_bytes(m, code), values.device)
    _check(getattr(lib(), fn)(_ptr(out), m, _ptr(bins), _ptr(values), n, code, _ptr(ws), ws.numel(),
                              block_threads, _stream(stream)), fn)
    return out


def det_scatter_min(out: torch.Tensor, bins: torch.Tensor, values: torch.Tensor, *, block_threads: int = 0,
                    workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[b] = IEEE minimum of out[b] and the values aimed at b (see det.h); returns out."""
    return _scatter_minmax("det_scatter_min", out, bins, values, block_threads, workspace, stream)


def det_scatter_max(out: torch.Tensor, bins: torch.Tensor, values: torch.Tensor, *, block_threads: int = 0,
                    workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[b] = IEEE maximum of out[b] and the values aimed at b (see det.h); returns out."""
    return _scatter_minmax("det_scatter_max", out, bins, values, block_threads, workspace, stream)


def det_scan_i32(x: torch.Tensor, y: torch.Tensor | None = None, *, exclusive: bool = False,
                 total_out: torch.Tensor | None = None, block_threads: int = 0,
                 workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """int32 prefix sum modulo 2^32 (see det.h); y may be x; returns y."""
    _dev(x, "x")
    if x.dtype != torch.int32 or (y is not None and y.dtype != torch.int32):
        raise TypeError("det_scan_i32 takes int32 tensors")
    if total_out is not None and (total_out.dtype != torch.int32 or total_out.numel() < 1):
        raise TypeError("total_out must hold one int32")
    if y is None:
        y = torch.empty_like(x)
    n = x.numel()
    ws = _ws(workspace, lib().det_scan_i32_workspace_bytes(n), x.device)
    _check(lib().det_scan_i32(_ptr(x), _ptr(y), n, SCAN_EXCLUSIVE if exclusive else SCAN_INCLUSIVE, _ptr(total_out),
                              _ptr(ws), ws.numel(), block_threads, _stream(stream)), "det_scan_i32")
    return y


def det_slot_alloc(counter: torch.Tensor, index: torch.Tensor, *, count: torch.Tensor | None = None,
                   slot_out: torch.Tensor | None = None, index_offset: int = 0, block_threads: int = 0,
                   workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """slot = atomic_add(counter, index[i], count[i]) in thread order (see det.h); returns the slots."""
    _dev(counter, "counter"), _dev(index, "index")
    if counter.dtype != torch.int32 or index.dtype != torch.int32 or (count is not None and count.dtype != torch.int32):
        raise TypeError("det_slot_alloc takes int32 tensors")
    n = index.numel()
    if count is not None and count.numel() != n:
        raise ValueError("count must have one entry per record")
    if slot_out is None:
        slot_out = torch.empty(n, dtype=torch.int32, device=index.device)
    ws = _ws(workspace, lib().det_slot_alloc_workspace_bytes(n, counter.numel()), index.device)
    _check(lib().det_slot_alloc(_ptr(counter), counter.numel(), _ptr(index), int(index_offset), _ptr(count), n,
                                _ptr(slot_out), _ptr(ws), ws.numel(), block_threads, _stream(stream)),
           "det_slot_alloc")
    return slot_out


def det_scatter_add_rows(dst: torch.Tensor, idx: torch.Tensor, src: torch.Tensor, *, row_offset: int = 0,
                         prev_out: torch.Tensor | None = None, block_threads: int = 0,
                         workspace: torch.Tensor | None = None, stream=None, ordered: bool = False) -> torch.Tensor:
    """dst[idx[s] + row_offset] += src[s] row by row, in a fixed order; returns dst.

    ordered=False: per destination the rows are added by the pairwise tree and
    every contributor's prev is the row before the call.  ordered=True: the
    rows are applied one at a time in ascending s and prev is the running value
    (det_scatter_add_rows_ordered)."""
    _dev(dst, "dst"), _dev(idx, "idx"), _dev(src, "src")
    code = _code(src)
    if dst.dim() != 2 or src.dim() != 2 or dst.shape[1] != src.shape[1] or dst.dtype != src.dtype:
        raise ValueError("dst and src must be 2-D of one dtype with equal row length")
    if idx.dtype != torch.int32 or idx.numel() != src.shape[0]:
        raise ValueError("idx must be int32 with one entry per source row")
    R, W = dst.shape
    M = src.shape[0]
    nbytes = lib().det_scatter_add_rows_workspace_bytes(M, R, W, code)
    ws = _ws(workspace, nbytes, src.device)
    fn = "det_scatter_add_rows_ordered" if ordered else "det_scatter_add_rows"
    _check(getattr(lib(), fn)(_ptr(dst), R, W, _ptr(idx), int(row_offset), _ptr(src), M, _ptr(prev_out), code,
                              _ptr(ws), ws.numel(), block_threads, _stream(stream)), fn)
    return dst


def det_scatter_add_vec(out: torch.Tensor, bins: torch.Tensor, values: torch.Tensor, *, block_threads: int = 0,
                        workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[bins[i], :] += values[i, :] for composite values, component-wise in a fixed order; returns out."""
    _dev(out, "out"), _dev(bins, "bins"), _dev(values, "values")
    code = _code(values)
    if out.dim() != 2 or values.dim() != 2 or out.shape[1] != values.shape[1] or out.dtype != values.dtype:
        raise ValueError("out and values must be 2-D of one dtype with equal width")
    if bins.dtype != torch.int32 or bins.numel() != values.shape[0]:
        raise ValueError("bins must be int32 with one entry per record")
    m, width = out.shape
    n = values.shape[0]
    ws = _ws(workspace, lib().det_scatter_add_vec_workspace_bytes(n, m, width, code), values.device)
    _check(lib().det_scatter_add_vec(_ptr(out), m, width, _ptr(bins), _ptr(values), n, code, _ptr(ws), ws.numel(),
                                     block_threads, _stream(stream)), "det_scatter_add_vec")
    return out


def det_scan(x: torch.Tensor, y: torch.Tensor | None = None, *, flags: int = SCAN_INCLUSIVE,
             total_out: torch.Tensor | None = None, block_threads: int = 0,
             workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Anchored look-back prefix sum (see det.h); y may be x; returns y."""
    _dev(x, "x")
    code = _code(x)
    if y is None:
        y = torch.empty_like(x)
    n = x.numel()
    nbytes = lib().det_scan_workspace_bytes(n, code)
    ws = _ws(workspace, nbytes, x.device)
    _check(lib().det_scan(_ptr(x), _ptr(y), n, code, int(flags), _ptr(total_out), _ptr(ws), ws.numel(),
                          block_threads, _stream(stream)), "det_scan")
    return y


def det_segmented_scan(x: torch.Tensor, seg_offsets: torch.Tensor, y: torch.Tensor | None = None, *,
                       flags: int = SCAN_INCLUSIVE, block_threads: int = 0,
                       workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Segmented anchored look-back prefix sum over int64 CSR offsets."""
    _dev(x, "x"), _dev(seg_offsets, "seg_offsets")
    code = _code(x)
    if seg_offsets.dtype != torch.int64:
        raise TypeError("seg_offsets must be int64")
    if y is None:
        y = torch.empty_like(x)
    n, S = x.numel(), seg_offsets.numel() - 1
    nbytes = lib().det_segmented_scan_workspace_bytes(n, S, code)
    ws = _ws(workspace, nbytes, x.device)
    _check(lib().det_segmented_scan(_ptr(x), _ptr(y), n, _ptr(seg_offsets), S, code, int(flags), _ptr(ws),
                                    ws.numel(), block_threads, _stream(stream)), "det_segmented_scan")
    return y


# ---------------------------------------------------------------------------
# measurement hooks (include/det_profile.h)


class KernelTimer:
    """Records a CUDA event pair around each kernel the library launches
    while active; ``kernels()`` returns [(name, ms), ...] in launch order."""

    def __init__(self, capacity: int = 256):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * capacity)]
        for e in self.events:
            e.record()  # materialise the underlying cudaEvent_t
        torch.cuda.synchronize()
        self._arr = (ctypes.c_void_p * len(self.events))(*[e.cuda_event for e in self.events])
        self.capacity = capacity

    def __enter__(self):
        lib().det_profile_set_events(self._arr, self.capacity)
        return self

    def __exit__(self, *exc):
        self._count = lib().det_profile_event_count()
        self._names = [lib().det_profile_event_name(i).decode() for i in range(self._count)]
        lib().det_profile_set_events(None, 0)
        return False

    def kernels(self):
        torch.cuda.synchronize()
        return [(self._names[i], self.events[2 * i].elapsed_time(self.events[2 * i + 1]))
                for i in range(self._count)]


def launch_count() -> int:
    return int(lib().det_launch_count())


def add_rate_probe(dtype: torch.dtype, iters: int, sink: torch.Tensor, stream=None) -> int:
    """Enqueue the add-only probe launch; returns the additions it performs."""
    adds = ctypes.c_ulonglong(0)
    code = F32 if dtype == torch.float32 else F64
    _check(lib().det_profile_add_rate_probe(code, int(iters), _ptr(sink), _stream(stream), ctypes.byref(adds)),
           "det_profile_add_rate_probe")
    return int(adds.value)


# ---------------------------------------------------------------------------
# nondeterministic baselines (include/det_baselines.h): comparison only


def atomic_sum(x: torch.Tensor, out: torch.Tensor, stream=None) -> torch.Tensor:
    _check(lib().det_atomic_sum(_ptr(x), x.numel(), _code(x), _ptr(out), _stream(stream)), "det_atomic_sum")
    return out


def atomic_scatter_add(out: torch.Tensor, bins: torch.Tensor, values: torch.Tensor, stream=None) -> torch.Tensor:
    _check(lib().det_atomic_scatter_add(_ptr(out), out.numel(), _ptr(bins), _ptr(values), values.numel(),
                                        _code(values), _stream(stream)), "det_atomic_scatter_add")
    return out


def atomic_scatter_add_rows(dst, idx, src, prev_out=None, row_offset: int = 0, stream=None):
    R, W = dst.shape
    _check(lib().det_atomic_scatter_add_rows(_ptr(dst), R, W, _ptr(idx), int(row_offset), _ptr(src), src.shape[0],
                                             _ptr(prev_out), _code(src), _stream(stream)),
           "det_atomic_scatter_add_rows")
    return dst


def dlb_scan(x: torch.Tensor, y: torch.Tensor, workspace: torch.Tensor | None = None, stream=None):
    nbytes = lib().det_dlb_scan_workspace_bytes(x.numel(), _code(x))
    ws = _ws(workspace, nbytes, x.device)
    _check(lib().det_dlb_scan(_ptr(x), _ptr(y), x.numel(), _code(x), _ptr(ws), ws.numel(), _stream(stream)),
           "det_dlb_scan")
    return y


def atomic_slot_alloc(counter: torch.Tensor, index: torch.Tensor, slot_out: torch.Tensor, *,
                      count: torch.Tensor | None = None, index_offset: int = 0, stream=None) -> torch.Tensor:
    """Baseline: slot = atomicAdd(counter[index[i]], ...) in arrival order (see det_baselines.h)."""
    _check(lib().det_atomic_slot_alloc(_ptr(counter), counter.numel(), _ptr(index), int(index_offset), _ptr(count),
                                       index.numel(), _ptr(slot_out), _stream(stream)), "det_atomic_slot_alloc")
    return slot_out
