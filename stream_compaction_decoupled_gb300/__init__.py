"""Device-wide prefix sums and stream compaction for the GB300 (sm_103a).

A thin binding over the C ABI of ``libgbscan.so`` (declared in include/gbscan.h):
every function marshals torch tensors into device pointers, sizes and the current
CUDA stream, and calls the entry point of the same name (without the ``gb_``
prefix).  All compute runs in the library's CUDA kernels; torch only provides
device memory and streams.  There is no fallback: if the library is not built, or
there is no GPU, the calls raise.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgbscan.so")

# Mirrors of the enums in include/gbscan.h.
I32, U32, I64, U64, F32, F64 = range(6)
ADD, MAX, MIN, MUL, AFFINE = range(5)
LT, LE, GT, GE, EQ, NE, BIT_CLEAR = range(7)
KIND_SCAN, KIND_BATCHED_AXIS1, KIND_BATCHED_AXIS0, KIND_COMPACT, KIND_PACK, KIND_REDUCE_THEN_SCAN, \
    KIND_PARTITION, KIND_SEGMENTED = range(8)
OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_TEMP, ERR_NO_IDENTITY, ERR_RANGE, ERR_CUDA, ERR_TIMEOUT = range(8)

OPS = {"add": ADD, "max": MAX, "min": MIN, "mul": MUL, "affine": AFFINE}
PREDS = {"lt": LT, "le": LE, "gt": GT, "ge": GE, "eq": EQ, "ne": NE, "bit_clear": BIT_CLEAR}
_NP_OF = {I32: np.int32, U32: np.uint32, I64: np.int64, U64: np.uint64, F32: np.float32, F64: np.float64}

# Exported symbols and their ctypes signatures (the whole of include/gbscan.h).
_vp, _i, _i64, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
SIGNATURES = {
    "gb_scan_inclusive": (_i, [_i, _i, _i, _vp, _vp, _i64, _vp, _sz, _vp]),
    "gb_scan_exclusive": (_i, [_i, _i, _i, _vp, _vp, _i64, _vp, _vp, _sz, _vp]),
    "gb_scan_batched": (_i, [_i, _i, _i, _i, _vp, _vp, _i64, _i64, _i, _vp, _vp, _sz, _vp]),
    "gb_compact": (_i, [_i, _vp, _i64, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
    "gb_partition": (_i, [_i, _vp, _i64, _i, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "gb_pack_by_counts": (_i, [_vp, _i64, _vp, _vp, _i64, _vp, _vp, _sz, _vp]),
    "gb_scan_reduce_then_scan": (_i, [_i, _i, _i, _vp, _vp, _i64, _vp, _vp, _sz, _vp]),
    "gb_scan_then_fan": (_i, [_i, _i, _i, _vp, _vp, _i64, _vp, _vp, _sz, _vp]),
    "gb_scan_segmented": (_i, [_i, _i, _i, _vp, _vp, _vp, _i64, _vp, _vp, _sz, _vp]),
    "gb_temp_storage_bytes": (_sz, [_i, _i, _i, _i64, _i64]),
    "gb_device_error": (_i, [_vp]),
    "gb_last_device_error": (_i, [_vp, _vp]),
    "gb_status_string": (ctypes.c_char_p, [_i]),
    "gb_last_cuda_error": (_i, []),
    "gb_version": (_i, []),
    "gb_set_profile_events": (None, [_vp, _vp]),
    "gb_set_wait_limit_ns": (None, [ctypes.c_uint64]),
    "gb_set_stalled_tile": (None, [_i64]),
    "gb_scan_inclusive_noalloc": (_i, [_i, _i, _vp, _vp, _i64, _vp]),
    "gb_scan_inclusive_host": (_i, [_i, _i, _vp, _vp, _i64, _i64, _vp, _sz, _vp]),
    "gb_host_scan_work_bytes": (_sz, [_i, _i64, _i64]),
}

_lib = None


class GbError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        self.code = code
        msg = load().gb_status_string(code).decode()
        if code == ERR_CUDA:
            msg += " (cudaError %d)" % load().gb_last_cuda_error()
        super().__init__("%s%s" % (where + ": " if where else "", msg))


def load(path: str = LIB_PATH):
    """Load libgbscan.so (built by __graft_entry__.build()) and declare its symbols."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError("libgbscan.so is not built (%s); run __graft_entry__.build()" % path)
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib


def _check(rc: int, where: str):
    if rc != OK:
        raise GbError(rc, where)


def dtype_code(t) -> int:
    import torch
    table = {torch.int32: I32, torch.int64: I64, torch.float32: F32, torch.float64: F64}
    for name, code in (("uint32", U32), ("uint64", U64)):
        if hasattr(torch, name):
            table[getattr(torch, name)] = code
    if t not in table:
        raise TypeError("unsupported dtype %s" % t)
    return table[t]


def _stream(x, stream):
    import torch
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    return ctypes.c_void_p(torch.cuda.current_stream(x.device).cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def _torch_stream(x, stream):
    """The torch stream a call runs on: the current one, or the caller's (a
    torch.cuda.Stream, or any object with a cuda_stream handle, or a raw handle)."""
    import torch
    if stream is None:
        return torch.cuda.current_stream(x.device)
    if isinstance(stream, torch.cuda.Stream):
        return stream
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return torch.cuda.ExternalStream(handle, device=x.device)


def _temp(x, kind, dtype, lanes, rows, cols, temp, stream=None):
    import torch
    if temp is not None:
        return ctypes.c_void_p(temp.data_ptr()), temp.numel() * temp.element_size()
    nbytes = load().gb_temp_storage_bytes(kind, dtype, lanes, rows, cols)
    # Allocated on the stream the call runs on and freed when the call returns: the
    # caching allocator hands the block only to later allocations on that stream,
    # which run after this call's kernels.  (Allocated on another stream, the block
    # could go to work on that stream while the kernels still use it.)
    with torch.cuda.stream(_torch_stream(x, stream)):
        buf = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=x.device)
    return ctypes.c_void_p(buf.data_ptr()), nbytes


def _host_value(code, value, lanes):
    if value is None:
        return None, None
    arr = np.ascontiguousarray(np.broadcast_to(np.asarray(value, dtype=_NP_OF[code]).reshape(-1), (lanes,)))
    return arr, ctypes.c_void_p(arr.ctypes.data)


def temp_storage_bytes(kind: int, dtype, lanes: int, rows: int, cols: int = 0) -> int:
    code = dtype if isinstance(dtype, int) else dtype_code(dtype)
    return load().gb_temp_storage_bytes(kind, code, lanes, rows, cols)


def scan_inclusive(x, op: str = "add", lanes: int = 1, out=None, temp=None, stream=None):
    """Inclusive scan of x viewed as n elements of `lanes` values."""
    import torch
    out = torch.empty_like(x) if out is None else out
    _need_cuda(x, out)
    code, n = dtype_code(x.dtype), x.numel() // lanes
    tp, tb = _temp(x, KIND_SCAN, code, lanes, n, 0, temp, stream)
    _check(load().gb_scan_inclusive(code, lanes, OPS[op], ctypes.c_void_p(x.data_ptr()),
                                    ctypes.c_void_p(out.data_ptr()), n, tp, tb, _stream(x, stream)),
           "gb_scan_inclusive")
    return out


def scan_exclusive(x, op: str = "add", init=None, lanes: int = 1, out=None, temp=None, stream=None):
    """Exclusive scan: out_i = init (+) x_0 (+) ... (+) x_{i-1}."""
    import torch
    out = torch.empty_like(x) if out is None else out
    _need_cuda(x, out)
    code, n = dtype_code(x.dtype), x.numel() // lanes
    keep, ip = _host_value(code, init, lanes)
    tp, tb = _temp(x, KIND_SCAN, code, lanes, n, 0, temp, stream)
    _check(load().gb_scan_exclusive(code, lanes, OPS[op], ctypes.c_void_p(x.data_ptr()),
                                    ctypes.c_void_p(out.data_ptr()), n, ip, tp, tb, _stream(x, stream)),
           "gb_scan_exclusive")
    del keep
    return out


def scan_batched(x, axis: int, op: str = "add", inclusive: bool = True, init=None, lanes: int = 1,
                 out=None, temp=None, stream=None):
    """Scan a row-major (rows, cols[, lanes]) array along axis 1 (rows) or 0 (columns)."""
    import torch
    out = torch.empty_like(x) if out is None else out
    _need_cuda(x, out)
    rows, cols = x.shape[0], x.shape[1]
    code = dtype_code(x.dtype)
    keep, ip = _host_value(code, init, lanes)
    kind = KIND_BATCHED_AXIS1 if axis == 1 else KIND_BATCHED_AXIS0
    tp, tb = _temp(x, kind, code, lanes, rows, cols, temp, stream)
    _check(load().gb_scan_batched(code, lanes, OPS[op], 1 if inclusive else 0, ctypes.c_void_p(x.data_ptr()),
                                  ctypes.c_void_p(out.data_ptr()), rows, cols, axis, ip, tp, tb,
                                  _stream(x, stream)), "gb_scan_batched")
    del keep
    return out


def compact(x, pred: str, threshold, out_idx=None, out_count=None, temp=None, stream=None):
    """Stable compaction: int32 indices i with x[i] <pred> threshold, and their count (device)."""
    import torch
    n = x.numel()
    out_idx = torch.empty(max(n, 1), dtype=torch.int32, device=x.device) if out_idx is None else out_idx
    out_count = torch.empty(1, dtype=torch.int32, device=x.device) if out_count is None else out_count
    _need_cuda(x, out_idx, out_count)
    code = dtype_code(x.dtype)
    keep, tptr = _host_value(code, threshold, 1)
    tp, tb = _temp(x, KIND_COMPACT, code, 1, n, 0, temp, stream)
    _check(load().gb_compact(code, ctypes.c_void_p(x.data_ptr()), n, PREDS[pred], tptr,
                             ctypes.c_void_p(out_idx.data_ptr()), ctypes.c_void_p(out_count.data_ptr()),
                             tp, tb, _stream(x, stream)), "gb_compact")
    del keep
    return out_idx, out_count


def partition(x, pred: str, threshold, with_idx: bool = True, out=None, out_idx=None, out_count=None, temp=None,
              stream=None):
    """Stable partition: (out, out_idx or None, count (device int32)); out holds the
    elements with x <pred> threshold first, then the others, each in input order.
    pred "bit_clear" (integers) selects the elements whose bit `threshold` is 0."""
    import torch
    n = x.numel()
    out = torch.empty(max(n, 1), dtype=x.dtype, device=x.device) if out is None else out
    if with_idx and out_idx is None:
        out_idx = torch.empty(max(n, 1), dtype=torch.int32, device=x.device)
    out_count = torch.empty(1, dtype=torch.int32, device=x.device) if out_count is None else out_count
    _need_cuda(x, out, out_count)
    code = dtype_code(x.dtype)
    keep, tptr = _host_value(code, threshold, 1)
    tp, tb = _temp(x, KIND_PARTITION, code, 1, n, 0, temp, stream)
    _check(load().gb_partition(code, ctypes.c_void_p(x.data_ptr()), n, PREDS[pred], tptr,
                               ctypes.c_void_p(out.data_ptr()),
                               ctypes.c_void_p(out_idx.data_ptr()) if out_idx is not None else None,
                               ctypes.c_void_p(out_count.data_ptr()), tp, tb, _stream(x, stream)), "gb_partition")
    del keep
    return out, out_idx, out_count


def pack_by_counts(counts, capacity: int, offsets: bool = True, out_records=None, out_total=None,
                   temp=None, stream=None):
    """Variable-length packing: (offsets or None, records, total (device int32))."""
    import torch
    n = counts.numel()
    offs = torch.empty(max(n, 1), dtype=torch.int32, device=counts.device) if offsets else None
    out_records = (torch.empty(max(capacity, 1), dtype=torch.int32, device=counts.device)
                   if out_records is None else out_records)
    out_total = torch.empty(1, dtype=torch.int32, device=counts.device) if out_total is None else out_total
    _need_cuda(counts, offs, out_records, out_total)
    if counts.dtype.itemsize != 4 or counts.dtype.is_floating_point:
        raise TypeError("counts must be int32")
    tp, tb = _temp(counts, KIND_PACK, I32, 1, n, 0, temp, stream)
    _check(load().gb_pack_by_counts(ctypes.c_void_p(counts.data_ptr()), n,
                                    ctypes.c_void_p(offs.data_ptr()) if offs is not None else None,
                                    ctypes.c_void_p(out_records.data_ptr()), capacity,
                                    ctypes.c_void_p(out_total.data_ptr()), tp, tb, _stream(counts, stream)),
           "gb_pack_by_counts")
    return offs, out_records, out_total


def scan_inclusive_host(x, op: str = "add", out=None, chunk_elems: int = 0, work=None, stream=None):
    """Inclusive scan of a host (CPU) tensor into a host tensor through the device,
    chunk by chunk with the copies overlapping the scans (pin both tensors for the
    overlap).  Runs on `stream` (default: the current CUDA stream); synchronise it
    before reading `out`."""
    import torch
    if x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous host tensor")
    out = torch.empty_like(x, pin_memory=x.is_pinned()) if out is None else out
    if out.is_cuda or not out.is_contiguous() or out.numel() != x.numel() or out.dtype != x.dtype:
        raise ValueError("out must be a contiguous host tensor like x")
    code, n = dtype_code(x.dtype), x.numel()
    if work is not None:
        wp, wb = ctypes.c_void_p(work.data_ptr()), work.numel() * work.element_size()
    else:
        wp, wb = None, 0
    s = ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)) if stream is not None \
        else ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    _check(load().gb_scan_inclusive_host(code, OPS[op], ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                         n, chunk_elems, wp, wb, s), "gb_scan_inclusive_host")
    return out


def host_scan_work_bytes(dtype, n: int, chunk_elems: int = 0) -> int:
    return load().gb_host_scan_work_bytes(dtype_code(dtype), n, chunk_elems)


def scan_reduce_then_scan(x, op: str = "add", inclusive: bool = True, init=None, out=None, temp=None,
                          stream=None):
    """The three-launch reduce-then-scan variant (same results as the single-pass scans)."""
    import torch
    out = torch.empty_like(x) if out is None else out
    _need_cuda(x, out)
    code, n = dtype_code(x.dtype), x.numel()
    keep, ip = _host_value(code, init, 1)
    tp, tb = _temp(x, KIND_REDUCE_THEN_SCAN, code, 1, n, 0, temp, stream)
    _check(load().gb_scan_reduce_then_scan(code, OPS[op], 1 if inclusive else 0, ctypes.c_void_p(x.data_ptr()),
                                           ctypes.c_void_p(out.data_ptr()), n, ip, tp, tb, _stream(x, stream)),
           "gb_scan_reduce_then_scan")
    del keep
    return out


def device_error(stream=None) -> int:
    """Synchronise and return (and clear) the sticky device-side error code."""
    import torch
    s = ctypes.c_void_p(stream.cuda_stream if stream is not None else torch.cuda.current_stream().cuda_stream)
    return load().gb_device_error(s)


def last_device_error(temp, stream=None) -> int:
    """Synchronise and return the device-side status of the last call that ran with
    this scratch tensor (its `temp`, or the host scan's `work`)."""
    import torch
    s = _stream(temp, stream)
    return load().gb_last_device_error(ctypes.c_void_p(temp.data_ptr()), s)


def _event_handle(ev):
    # torch creates the CUDA event on its first record(); make sure it exists.
    if ev.cuda_event == 0:
        ev.record()
    return ctypes.c_void_p(ev.cuda_event)


def set_profile_events(before, after):
    """Have the next calls record `before`/`after` (torch.cuda.Event) around their main kernel."""
    if before is None or after is None:
        load().gb_set_profile_events(None, None)
    else:
        load().gb_set_profile_events(_event_handle(before), _event_handle(after))


def set_wait_limit_ns(ns: int):
    load().gb_set_wait_limit_ns(ns)


def set_stalled_tile(tile: int):
    load().gb_set_stalled_tile(tile)


def scan_then_fan(x, op: str = "add", inclusive: bool = True, init=None, out=None, temp=None, stream=None):
    """The three-launch scan-then-fan variant (same results as the single-pass scans)."""
    import torch
    out = torch.empty_like(x) if out is None else out
    _need_cuda(x, out)
    code, n = dtype_code(x.dtype), x.numel()
    keep, ip = _host_value(code, init, 1)
    tp, tb = _temp(x, KIND_REDUCE_THEN_SCAN, code, 1, n, 0, temp, stream)
    _check(load().gb_scan_then_fan(code, OPS[op], 1 if inclusive else 0, ctypes.c_void_p(x.data_ptr()),
                                   ctypes.c_void_p(out.data_ptr()), n, ip, tp, tb, _stream(x, stream)),
           "gb_scan_then_fan")
    del keep
    return out


def scan_segmented(x, flags, op: str = "add", inclusive: bool = True, init=None, out=None, temp=None, stream=None):
    """Segmented scan: flags (uint8 or bool, same length) marks the first element of
    each segment; every segment is scanned on its own (element 0 always starts one)."""
    import torch
    out = torch.empty_like(x) if out is None else out
    if flags.dtype == torch.bool:
        flags = flags.view(torch.uint8)
    if flags.dtype != torch.uint8 or flags.numel() != x.numel() or not flags.is_contiguous():
        raise ValueError("flags must be a contiguous uint8 (or bool) tensor with one entry per element")
    _need_cuda(x, out, flags)
    code, n = dtype_code(x.dtype), x.numel()
    keep, ip = _host_value(code, init, 1)
    tp, tb = _temp(x, KIND_SEGMENTED, code, 1, n, 0, temp, stream)
    _check(load().gb_scan_segmented(code, OPS[op], 1 if inclusive else 0, ctypes.c_void_p(x.data_ptr()),
                                    ctypes.c_void_p(flags.data_ptr()), ctypes.c_void_p(out.data_ptr()), n, ip,
                                    tp, tb, _stream(x, stream)), "gb_scan_segmented")
    del keep
    return out
