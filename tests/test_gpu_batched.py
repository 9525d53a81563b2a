"""GPU parity: batched scans along either axis, and lane-vector elements
(96-byte structs of 24 fp32 lanes, 17-lane fp64 duals), against the CPU oracle.
"""
import numpy as np
import pytest
import torch

import stream_compaction_decoupled_gb300 as gb
from stream_compaction_decoupled_gb300 import workloads
from parity import as3, assert_scan_matches

pytestmark = pytest.mark.gpu

NP = {"f32": np.float32, "f64": np.float64, "i32": np.int32, "i64": np.int64}


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    gb.load()
    yield
    torch.cuda.synchronize()


def make(dt, n, seed):
    if dt.startswith("f"):
        return workloads.normal(n, NP[dt], seed)
    return workloads.small_ints(n, seed, -1000, 1000, dtype=NP[dt])


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


@pytest.mark.parametrize("dt", ["i32", "f32", "f64", "i64"])
@pytest.mark.parametrize("op", ["add", "max"])
@pytest.mark.parametrize("shape", [(1, 1), (3, 5), (7, 4096), (5, 4097), (2, 9001), (300, 33), (4, 2048 * 3 + 1)])
def test_rows_axis1(dt, op, shape):
    rows, cols = shape
    x = make(dt, rows * cols, rows * 131 + cols)
    xd = dev(x).reshape(rows, cols)
    got = gb.scan_batched(xd, axis=1, op=op).cpu().numpy()
    assert_scan_matches(got, as3(x, rows, cols, 1), op, True, what="axis1 %s %s %s" % (dt, op, shape))
    init = x[0] if op != "add" else 3
    got = gb.scan_batched(xd, axis=1, op=op, inclusive=False, init=init).cpu().numpy()
    assert_scan_matches(got, as3(x, rows, cols, 1), op, False, init, what="axis1 excl %s" % (shape,))


# Few long rows (B <= 64, at least 65536 elements, 16-byte rows, at most 96 MiB in
# all) take the segment kernel with segments per row; the other shapes here sit just
# outside those limits and take the row kernel.
@pytest.mark.parametrize("dt", ["i32", "f32", "i64"])
@pytest.mark.parametrize("op", ["add", "max", "min"])
@pytest.mark.parametrize("shape", [(2, 65536), (3, 65536 + 4), (64, 65536), (5, 1_000_004), (65, 65536),
                                   (5, 1_000_003), (3, 65532)])
def test_rows_axis1_segments(dt, op, shape):
    rows, cols = shape
    x = make(dt, rows * cols, rows * 17 + cols)
    xd = dev(x).reshape(rows, cols)
    got = gb.scan_batched(xd, axis=1, op=op).cpu().numpy()
    assert_scan_matches(got, as3(x, rows, cols, 1), op, True, what="seg rows %s %s %s" % (dt, op, shape))
    init = x[0] if op != "add" else 5
    got = gb.scan_batched(xd, axis=1, op=op, inclusive=False, init=init).cpu().numpy()
    assert_scan_matches(got, as3(x, rows, cols, 1), op, False, init, what="seg rows excl %s" % (shape,))
    assert gb.device_error() == gb.OK


def test_rows_axis1_above_segment_limit():
    """2 rows of 12,582,912 fp32 (100.7 MB in all, above 96 MiB) take the row kernel."""
    rows, cols = 2, 12_582_912
    x = make("f32", rows * cols, 99)
    got = gb.scan_batched(dev(x).reshape(rows, cols), axis=1).cpu().numpy()
    assert_scan_matches(got, as3(x, rows, cols, 1), "add", True, what="rows kernel 2 x 12.6M")


@pytest.mark.parametrize("dt", ["i32", "f32", "f64", "i64"])
@pytest.mark.parametrize("op", ["add", "min"])
@pytest.mark.parametrize("shape", [(1, 7), (5, 3), (513, 8), (1000, 17), (130, 24), (65, 64), (200, 65),
                                   (97, 100), (129, 300), (3, 1)])
def test_columns_axis0(dt, op, shape):
    rows, cols = shape
    x = make(dt, rows * cols, rows * 7 + cols)
    xd = dev(x).reshape(rows, cols)
    got = gb.scan_batched(xd, axis=0, op=op).cpu().numpy()
    assert_scan_matches(got, as3(x, 1, rows, cols), op, True, what="axis0 %s %s %s" % (dt, op, shape))
    init = x[0] if op != "add" else 2
    got = gb.scan_batched(xd, axis=0, op=op, inclusive=False, init=init).cpu().numpy()
    assert_scan_matches(got, as3(x, 1, rows, cols), op, False, init, what="axis0 excl %s" % (shape,))


@pytest.mark.parametrize("dt", ["f32", "f64", "i32"])
@pytest.mark.parametrize("lanes", [2, 3, 5, 17, 24, 33])
@pytest.mark.parametrize("n", [1, 100, 1001, 5003])
def test_lane_vectors_1d(dt, lanes, n):
    x = make(dt, n * lanes, n * lanes + 5)
    xd = dev(x)
    got = gb.scan_inclusive(xd, "add", lanes=lanes).cpu().numpy()
    assert_scan_matches(got, as3(x, 1, n, lanes), "add", True, what="lanes=%d n=%d" % (lanes, n))
    init = np.arange(lanes).astype(NP[dt])
    got = gb.scan_exclusive(xd, "add", init=init, lanes=lanes).cpu().numpy()
    assert_scan_matches(got, as3(x, 1, n, lanes), "add", False, init, what="lanes excl")


def test_lane_vectors_max_needs_init():
    x = dev(workloads.normal(24 * 10, np.float32, 1))
    with pytest.raises(gb.GbError) as e:
        gb.scan_exclusive(x, "max", lanes=24)
    assert e.value.code == gb.ERR_NO_IDENTITY


@pytest.mark.parametrize("lanes", [17, 24])
def test_lane_vectors_along_rows(lanes):
    rows, cols = 3, 1001
    x = make("f32" if lanes == 24 else "f64", rows * cols * lanes, 31)
    xd = dev(x).reshape(rows, cols, lanes)
    got = gb.scan_batched(xd, axis=1, lanes=lanes).cpu().numpy()
    assert_scan_matches(got, as3(x, rows, cols, lanes), "add", True, what="rows of lane vectors")
    got = gb.scan_batched(xd, axis=0, lanes=lanes).cpu().numpy()
    assert_scan_matches(got, as3(x, 1, rows, cols * lanes), "add", True, what="columns of lane vectors")


# ---- lane-vector scans over many tiles: one tile, several waves of tiles, ragged last
# tiles, batches, 16-byte and odd row widths (tiles hold 320 rows of 24 fp32 lanes, 1024
# rows of 8, 480 rows of 17 fp64 lanes).  8-byte lanes in a long single chain here take
# reduce-then-scan, the rest the look-back lane kernel.

LANE_SHAPES = [(1, 320, 24), (1, 321, 24), (1, 200_000, 24), (3, 100_003, 24), (1, 1_000_000, 8),
               (2, 4097, 8), (1, 300_000, 17), (5, 20_000, 17), (1, 150_000, 32), (1, 40_000, 64),
               (1, 50_000, 65), (2, 10_001, 6)]


@pytest.mark.parametrize("dt", ["f32", "f64", "i32", "i64"])
@pytest.mark.parametrize("op", ["add", "max"])
@pytest.mark.parametrize("shape", LANE_SHAPES)
def test_lane_tiles(dt, op, shape):
    b, n, lanes = shape
    x = make(dt, b * n * lanes, b * n + lanes)
    xd = dev(x).reshape(b, n, lanes)
    got = gb.scan_batched(xd, axis=1, op=op, lanes=lanes).cpu().numpy()
    assert_scan_matches(got, as3(x, b, n, lanes), op, True, what="lanes %s %s %s" % (dt, op, shape))
    init = (np.arange(lanes) - 3).astype(NP[dt]) if op == "add" else x[:lanes].copy()
    got = gb.scan_batched(xd, axis=1, op=op, inclusive=False, init=init, lanes=lanes).cpu().numpy()
    assert_scan_matches(got, as3(x, b, n, lanes), op, False, init, what="lanes excl %s" % (shape,))
    assert gb.device_error() == gb.OK


# 8-byte lanes in at most 4 chains of at least 128 look-back tiles, in at most 160 MiB,
# take reduce-then-scan: whole rows (1 and 3 batches), 64-lane strips (2 strips x 2
# batches), an 8-lane last strip, a 1-lane last strip (plain loads), 2 lanes (1024-row
# tiles), and each through a view one element off 16-byte alignment (plain loads).
RTS_SHAPES = [(1, 300_000, 17), (2, 70_000, 64), (1, 130_000, 40), (1, 130_000, 33), (1, 300_000, 2),
              (3, 130_000, 17)]


@pytest.mark.parametrize("dt", ["f64", "i64"])
@pytest.mark.parametrize("op", ["add", "max"])
@pytest.mark.parametrize("shape", RTS_SHAPES)
@pytest.mark.parametrize("offset", [0, 1])
def test_rts_lanes(dt, op, shape, offset):
    b, n, lanes = shape
    x = make(dt, b * n * lanes + offset, b * n + lanes + offset)
    xd = dev(x)[offset:].reshape(b, n, lanes)
    x = x[offset:]
    got = gb.scan_batched(xd, axis=1, op=op, lanes=lanes).cpu().numpy()
    assert_scan_matches(got, as3(x, b, n, lanes), op, True, what="rts %s %s %s +%d" % (dt, op, shape, offset))
    init = (np.arange(lanes) - 3).astype(NP[dt]) if op == "add" else x[:lanes].copy()
    got = gb.scan_batched(xd, axis=1, op=op, inclusive=False, init=init, lanes=lanes).cpu().numpy()
    assert_scan_matches(got, as3(x, b, n, lanes), op, False, init, what="rts excl %s +%d" % (shape, offset))
    assert gb.device_error() == gb.OK


# Above 160 MiB, 8-byte lanes in one long chain take the look-back lane kernel again.
@pytest.mark.parametrize("op", ["add", "min"])
@pytest.mark.parametrize("dt", ["f64", "i64"])
def test_lane_kernel_long_chain_above_rts_limit(dt, op):
    b, n, lanes = 1, 1_250_000, 17
    x = make(dt, b * n * lanes, 77)
    got = gb.scan_batched(dev(x).reshape(b, n, lanes), axis=1, op=op, lanes=lanes).cpu().numpy()
    assert_scan_matches(got, as3(x, b, n, lanes), op, True, what="look-back lanes %s %s" % (dt, op))
    assert gb.device_error() == gb.OK


# ---- the full-size batched and large-element workloads, element by element -------

BATCHED = ["fp32_4096x4096_axis0", "fp32_4096x4096_axis1", "fp32_2x1e7_axis1", "fp32_1e6x8_axis0",
           "fp64_1000x1e4_axis0", "struct96_1e6", "struct96_3x1e5_axis1", "dual16_1e6",
           "dual16_3x1e5_axis1"]


@pytest.mark.parametrize("name", BATCHED)
def test_full_size_workload(name):
    w = workloads.BY_NAME[name]
    x = w.make()
    xd = dev(x)
    if w.kind == "scan":  # 1-D scan of lane-vector elements
        n = w.shape[0]
        got = gb.scan_inclusive(xd, w.op, lanes=w.lanes).cpu().numpy()
        x3 = as3(x, 1, n, w.lanes)
    else:
        rows, cols = w.shape
        got = gb.scan_batched(xd.reshape(rows, cols, w.lanes), axis=w.axis, op=w.op, lanes=w.lanes).cpu().numpy()
        x3 = as3(x, rows, cols, w.lanes) if w.axis == 1 else as3(x, 1, rows, cols * w.lanes)
    assert_scan_matches(got, x3, w.op, True, what=name)
    assert gb.device_error() == gb.OK
