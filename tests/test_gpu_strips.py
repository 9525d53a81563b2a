"""GPU parity: the strip kernel (scans down the columns of arrays with at least as
many 64-byte column strips as the GPU has SMs; each CTA walks whole strips with no
look-back) against the CPU oracle.

Shapes cross the kernel's tile (512 rows), leave ragged last tiles and a ragged last
strip (columns not a multiple of the 16 four-byte / 8 eight-byte lanes of a strip), and include
lane-vector elements of 2,432 to 4,096 lanes scanned as one chain.  Every operator,
inclusive and exclusive with a per-lane initial value, against the usual bars
(bit-exact for integers and max/min, the stated tolerance for float add).
"""
import numpy as np
import pytest
import torch

import stream_compaction_decoupled_gb300 as gb
from stream_compaction_decoupled_gb300 import workloads
from parity import as3, assert_scan_matches

pytestmark = pytest.mark.gpu

NP = {"f32": np.float32, "f64": np.float64, "i32": np.int32, "i64": np.int64, "u32": np.uint32,
      "u64": np.uint64}


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    gb.load()
    yield
    torch.cuda.synchronize()


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def values(dt, op, n, seed, cols):
    if op == "mul":
        if dt[0] != "f":
            return workloads.odd_ints(n, seed, np.int64).astype(NP[dt])
        rows = n // cols  # one +-2^k walk per column: every running product stays in range
        return np.stack([workloads.signs_pow2(rows, NP[dt], seed + c) for c in range(cols)], axis=1).reshape(-1)
    if dt[0] == "f":
        return workloads.normal(n, NP[dt], seed)
    if dt[0] == "u":
        return workloads.full_range_uints(n, seed, NP[dt])
    return workloads.small_ints(n, seed, -1000, 1000, dtype=np.int64).astype(NP[dt])


# (rows, cols): 152 strips and more for 4-byte (16 lanes a strip) and 8-byte integers (8 lanes)
SHAPES = {
    4: [(1, 2432), (3, 4096), (511, 2440), (513, 2432), (1025, 4100), (2000, 3000)],
    8: [(1, 1216), (5, 2048), (511, 1220), (513, 1216), (1025, 1300), (1500, 1250)],
}


@pytest.mark.parametrize("dt", ["f32", "i32", "u32", "i64", "u64"])
@pytest.mark.parametrize("op", ["add", "max", "min", "mul"])
def test_strips_axis0(dt, op):
    if dt[0] == "u" and not hasattr(torch, "uint32"):
        pytest.skip("this torch has no unsigned 32/64-bit tensors")
    for rows, cols in SHAPES[np.dtype(NP[dt]).itemsize]:
        x = values(dt, op, rows * cols, rows * 7 + cols, cols)
        xd = dev(x).reshape(rows, cols)
        what = "%s %s %d x %d" % (dt, op, rows, cols)
        got = gb.scan_batched(xd, axis=0, op=op).cpu().numpy()
        assert_scan_matches(got, as3(x, 1, rows, cols), op, True, what="incl " + what)
        init = x[0] if op in ("max", "min") else (NP[dt](1) if op == "mul" else NP[dt](3))
        got = gb.scan_batched(xd, axis=0, op=op, inclusive=False, init=init).cpu().numpy()
        assert_scan_matches(got, as3(x, 1, rows, cols), op, False, init, what="excl " + what)
    assert gb.device_error() == gb.OK


@pytest.mark.parametrize("dt,lanes", [("f32", 4096), ("f32", 2432), ("i32", 3000), ("i64", 2048), ("i64", 1216)])
def test_strips_lane_vectors(dt, lanes):
    """One chain of elements of many lanes, each lane its own initial value."""
    for n in (1, 700, 1300):
        x = values(dt, "add", n * lanes, n + lanes, lanes)
        xd = dev(x)
        got = gb.scan_inclusive(xd, "add", lanes=lanes).cpu().numpy()
        assert_scan_matches(got, as3(x, 1, n, lanes), "add", True, what="lanes=%d n=%d" % (lanes, n))
        init = (np.arange(lanes) % 97).astype(NP[dt])
        got = gb.scan_exclusive(xd, "add", init=init, lanes=lanes).cpu().numpy()
        assert_scan_matches(got, as3(x, 1, n, lanes), "add", False, init, what="lanes excl %d n=%d" % (lanes, n))
        got = gb.scan_exclusive(xd, "max", init=x[:lanes], lanes=lanes).cpu().numpy()
        assert_scan_matches(got, as3(x, 1, n, lanes), "max", False, x[:lanes], what="lanes max %d n=%d" % (lanes, n))
    assert gb.device_error() == gb.OK


def test_strips_unaligned_view_takes_lane_kernel():
    """A view that starts off a 16-byte boundary cannot take the strip kernel; the lane
    kernel scans it, with the same results."""
    rows, cols = 600, 2433
    x = values("f32", "add", rows * cols + 1, 5, cols)
    xd = dev(x)[1:].reshape(rows, cols)
    got = gb.scan_batched(xd, axis=0).cpu().numpy()
    assert_scan_matches(got, as3(x[1:], 1, rows, cols), "add", True, what="unaligned columns")


def test_strips_call_status_is_clean():
    """The strip kernel resets the call's status word (it has no waits of its own)."""
    rows, cols = 1000, 4096
    x = dev(values("f32", "add", rows * cols, 9, cols)).reshape(rows, cols)
    nbytes = gb.temp_storage_bytes(gb.KIND_BATCHED_AXIS0, gb.F32, 1, rows, cols)
    temp = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    temp.fill_(0xFF)  # a stale status word from some earlier use
    gb.scan_batched(x, axis=0, temp=temp)
    assert gb.last_device_error(temp) == gb.OK


@pytest.mark.parametrize("dt,rows,cols,lanes", [("f32", 12, 300, 256), ("i32", 10, 513, 272), ("i64", 12, 700, 128),
                                                ("f32", 3, 1025, 1024)])
def test_strips_rows_of_lane_vectors(dt, rows, cols, lanes):
    """Rows of lane-vector elements scanned along the rows: every row is its own set of
    chains (B > 1), with enough strips in all to take the strip kernel."""
    x = values(dt, "add", rows * cols * lanes, rows + cols + lanes, lanes)
    xd = dev(x).reshape(rows, cols, lanes)
    got = gb.scan_batched(xd, axis=1, lanes=lanes).cpu().numpy()
    assert_scan_matches(got, as3(x, rows, cols, lanes), "add", True, what="rows of %d lanes" % lanes)
    init = (np.arange(lanes) % 13).astype(NP[dt])
    got = gb.scan_batched(xd, axis=1, lanes=lanes, inclusive=False, init=init).cpu().numpy()
    assert_scan_matches(got, as3(x, rows, cols, lanes), "add", False, init, what="rows excl %d lanes" % lanes)
    got = gb.scan_batched(xd, axis=1, op="max", lanes=lanes).cpu().numpy()
    assert_scan_matches(got, as3(x, rows, cols, lanes), "max", True, what="rows max %d lanes" % lanes)
    assert gb.device_error() == gb.OK
