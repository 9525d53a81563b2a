"""The sequential CPU oracle for prefix sums and stream compaction.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The GPU library never
does, and nothing here imports the GPU library: the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, one left-to-right loop per scanned
line, fp64 accumulation for floating point); this module only builds it, loads it
with ctypes and marshals numpy arrays.  Definitions followed are those of
B. Merry, "Prefix sums on GPUs" (slides "Exclusive Prefix Sum", "Inclusive Prefix
Sum", "Output Format", "Solution", "Other Applications": compaction, partitioning),
and for the one operator that is not commutative (composition of affine maps) the
caveat on commutativity in The CUDA Handbook, 13.3.4.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

# The oracle's own numbering (mirrors the enums at the top of oracle.c).
_DTYPES = {"i32": 0, "u32": 1, "i64": 2, "u64": 3, "f32": 4, "f64": 5}
_NP = {"i32": np.int32, "u32": np.uint32, "i64": np.int64, "u64": np.uint64,
       "f32": np.float32, "f64": np.float64}
_OPS = {"add": 0, "max": 1, "min": 2, "mul": 3}
_PREDS = {"lt": 0, "le": 1, "gt": 2, "ge": 3, "eq": 4, "ne": 5, "bit_clear": 6}

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, vp, i = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        lib.oracle_scan.argtypes = [i, i, i, vp, vp, i64, i64, i64, vp, i64]
        lib.oracle_scan.restype = i
        lib.oracle_compact.argtypes = [i, vp, i64, i, vp, vp]
        lib.oracle_compact.restype = i64
        lib.oracle_scan_segmented.argtypes = [i, i, i, vp, vp, vp, i64, vp]
        lib.oracle_scan_segmented.restype = i
        lib.oracle_partition.argtypes = [i, vp, i64, i, vp, vp, vp]
        lib.oracle_partition.restype = i64
        lib.oracle_scan_affine.argtypes = [i, i, vp, vp, i64, vp]
        lib.oracle_scan_affine.restype = i
        lib.oracle_pack_by_counts.argtypes = [vp, i64, vp, vp, i64]
        lib.oracle_pack_by_counts.restype = i64
        _lib = lib
    return _lib


def dtype_name(a: np.ndarray) -> str:
    for k, v in _NP.items():
        if a.dtype == np.dtype(v):
            return k
    raise TypeError("oracle: unsupported dtype %s" % a.dtype)


class NoIdentity(ValueError):
    """An exclusive max/min scan was asked for without an initial value."""


def scan3(x: np.ndarray, op: str = "add", inclusive: bool = True, init=None) -> np.ndarray:
    """Scan a (B, R, C) array along axis 1 (the middle axis).

    Integer inputs give the same integer type (wrapping add and multiply); float
    inputs give fp64.  ``init`` (exclusive only) is a scalar or a sequence of lane values;
    lane c starts from init[c % len(init)].
    """
    x = np.ascontiguousarray(x)
    if x.ndim != 3:
        raise ValueError("scan3 wants a (B, R, C) array")
    dt = dtype_name(x)
    out = np.empty(x.shape, dtype=np.float64 if dt in ("f32", "f64") else x.dtype)
    init_arr = None
    if init is not None:
        init_arr = np.ascontiguousarray(np.atleast_1d(np.asarray(init, dtype=x.dtype)))
    rc = _load().oracle_scan(
        _DTYPES[dt], _OPS[op], 1 if inclusive else 0,
        x.ctypes.data, out.ctypes.data, x.shape[0], x.shape[1], x.shape[2],
        None if init_arr is None else init_arr.ctypes.data,
        0 if init_arr is None else init_arr.size)
    if rc == -2:
        raise NoIdentity("exclusive %s scan needs an initial value" % op)
    if rc != 0:
        raise ValueError("oracle_scan rejected its arguments (%d)" % rc)
    return out


def scan(x: np.ndarray, op: str = "add", inclusive: bool = True, init=None,
         lanes: int = 1) -> np.ndarray:
    """1-D scan of n elements of ``lanes`` values each (x has n*lanes values)."""
    x = np.ascontiguousarray(x).reshape(1, -1, lanes)
    return scan3(x, op, inclusive, init).reshape(-1)


def scan_batched(x: np.ndarray, axis: int, op: str = "add", inclusive: bool = True,
                 init=None, lanes: int = 1) -> np.ndarray:
    """Scan a row-major (rows, cols) matrix of ``lanes``-value elements.

    axis=1 scans along each row (contiguous); axis=0 scans down each column.
    """
    rows, cols = x.shape[0], x.shape[1]
    x = np.ascontiguousarray(x)
    if axis == 1:
        out = scan3(x.reshape(rows, cols, lanes), op, inclusive, init)
    elif axis == 0:
        out = scan3(x.reshape(1, rows, cols * lanes), op, inclusive, init)
    else:
        raise ValueError("axis must be 0 or 1")
    return out.reshape(x.shape)


def compact(x: np.ndarray, pred: str, threshold) -> np.ndarray:
    """Ascending int64 indices i with pred(x[i], threshold), compared in x's dtype."""
    x = np.ascontiguousarray(x).reshape(-1)
    dt = dtype_name(x)
    t = np.asarray(threshold, dtype=x.dtype).reshape(1)
    out = np.empty(max(x.size, 1), dtype=np.int64)
    cnt = _load().oracle_compact(_DTYPES[dt], x.ctypes.data, x.size, _PREDS[pred],
                                 t.ctypes.data, out.ctypes.data)
    if cnt < 0:
        raise ValueError("oracle_compact rejected its arguments (%d)" % cnt)
    return out[:cnt].copy()


def scan_segmented(x: np.ndarray, flags: np.ndarray, op: str = "add", inclusive: bool = True,
                   init=None) -> np.ndarray:
    """Scan restarting at head flags (flags[i] != 0: element i starts a segment;
    element 0 always does).  Integers keep their type; floats give fp64."""
    x = np.ascontiguousarray(x).reshape(-1)
    fl = np.ascontiguousarray(flags, dtype=np.uint8).reshape(-1)
    if fl.size != x.size:
        raise ValueError("one flag per element")
    dt = dtype_name(x)
    out = np.empty(max(x.size, 1), dtype=np.float64 if dt in ("f32", "f64") else x.dtype)
    ia = None if init is None else np.asarray(init, dtype=x.dtype).reshape(1)
    rc = _load().oracle_scan_segmented(_DTYPES[dt], _OPS[op], 1 if inclusive else 0, x.ctypes.data,
                                       fl.ctypes.data, out.ctypes.data, x.size,
                                       None if ia is None else ia.ctypes.data)
    if rc == -2:
        raise NoIdentity("exclusive %s scan needs an initial value" % op)
    if rc != 0:
        raise ValueError("oracle_scan_segmented rejected its arguments (%d)" % rc)
    return out[:x.size].copy()


def scan_affine(x: np.ndarray, inclusive: bool = True, init=None) -> np.ndarray:
    """Scan of affine maps y -> a*y + b under composition in index order (the earlier
    map applied first).  x holds n pairs (a_i, b_i) as 2n consecutive integers (any
    shape whose size is even); the result has x's shape and type.  init (exclusive
    only) is a pair (a, b); None means the identity map (1, 0)."""
    x = np.ascontiguousarray(x)
    if x.size % 2:
        raise ValueError("affine maps are pairs (a, b)")
    dt = dtype_name(x)
    out = np.empty(max(x.size, 2), dtype=x.dtype)
    ia = None if init is None else np.ascontiguousarray(np.asarray(init).astype(x.dtype).reshape(2))
    rc = _load().oracle_scan_affine(_DTYPES[dt], 1 if inclusive else 0, x.ctypes.data, out.ctypes.data,
                                    x.size // 2, None if ia is None else ia.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_scan_affine rejected its arguments (%d)" % rc)
    return out[:x.size].reshape(x.shape).copy()


def partition(x: np.ndarray, pred: str, threshold):
    """Stable partition: (values, int64 input indices, m).  The m elements with
    pred(x[i], threshold) come first, then the others, each in input order;
    pred "bit_clear" (integers) selects the elements whose bit `threshold` is 0."""
    x = np.ascontiguousarray(x).reshape(-1)
    dt = dtype_name(x)
    t = np.asarray(threshold, dtype=x.dtype).reshape(1)
    vals = np.empty(max(x.size, 1), dtype=x.dtype)
    idx = np.empty(max(x.size, 1), dtype=np.int64)
    m = _load().oracle_partition(_DTYPES[dt], x.ctypes.data, x.size, _PREDS[pred], t.ctypes.data,
                                 vals.ctypes.data, idx.ctypes.data)
    if m < 0:
        raise ValueError("oracle_partition rejected its arguments (%d)" % m)
    return vals[:x.size].copy(), idx[:x.size].copy(), int(m)


def pack_by_counts(counts: np.ndarray, capacity: int | None = None):
    """Variable-length packing: returns (offsets int64, records int32, total)."""
    counts = np.ascontiguousarray(counts, dtype=np.int32).reshape(-1)
    n = counts.size
    offsets = np.empty(max(n, 1), dtype=np.int64)
    total_guess = int(counts.astype(np.int64).sum()) if n else 0
    cap = total_guess if capacity is None else int(capacity)
    records = np.full(max(cap, 1), -1, dtype=np.int32)
    total = _load().oracle_pack_by_counts(counts.ctypes.data, n, offsets.ctypes.data,
                                          records.ctypes.data, cap)
    if total < 0:
        raise ValueError("oracle_pack_by_counts rejected its arguments (%d)" % total)
    return offsets[:n].copy(), records[:cap].copy(), int(total)
