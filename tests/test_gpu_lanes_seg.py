"""GPU parity: the lane segment kernel (one aligned chain of 4, 8 or 16 four-byte
lanes that fits in L2) against the CPU oracle.

These are the scans of small structs (the 32-byte struct of 8 fp32 lanes) and of
the columns of narrow matrices down axis 0 (1e6 x 8).  Sizes cross the kernel's
chunk (128 / 64 / 32 elements for 4 / 8 / 16 lanes), the point where every warp of
every CTA has a chunk (152 x 24 = 3648 chunks) and several chunks a warp; every operator,
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

CHUNK = {4: 128, 8: 64, 16: 32}


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    gb.load()
    yield
    torch.cuda.synchronize()


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def values(dt, op, n, seed, lanes=1):
    if op == "mul":
        if np.dtype(dt).kind != "f":
            return workloads.odd_ints(n, seed, np.int64).astype(dt)
        # one +-2^k walk per lane, so that every lane's running product stays in range
        m = n // lanes
        return np.stack([workloads.signs_pow2(m, dt, seed + c) for c in range(lanes)], axis=1).reshape(-1)
    if np.dtype(dt).kind == "f":
        return workloads.normal(n, dt, seed)
    return workloads.small_ints(n, seed, -1000, 1000, dtype=np.int64).astype(dt)


def sizes(lanes):
    ch = CHUNK[lanes]
    return [1, 2, ch - 1, ch, ch + 1, 1000, 3648 * ch - 1, 3648 * ch + 3, 300_007]


@pytest.mark.parametrize("lanes", [4, 8, 16])
@pytest.mark.parametrize("op", ["add", "max", "min", "mul"])
@pytest.mark.parametrize("dt", [np.float32, np.int32])
def test_lane_segments(lanes, op, dt):
    for n in sizes(lanes):
        x = values(dt, op, n * lanes, n + lanes, lanes)
        xd = dev(x)
        what = "%s %s lanes=%d n=%d" % (np.dtype(dt).name, op, lanes, n)
        got = gb.scan_inclusive(xd, op, lanes=lanes).cpu().numpy()
        assert_scan_matches(got, as3(x, 1, n, lanes), op, True, what=what + " incl")
        init = x[:lanes].copy() if op in ("max", "min") else (np.arange(lanes).astype(dt) + 1)
        got = gb.scan_exclusive(xd, op, init=init, lanes=lanes).cpu().numpy()
        assert_scan_matches(got, as3(x, 1, n, lanes), op, False, init, what=what + " excl")
    assert gb.device_error() == gb.OK


@pytest.mark.parametrize("cols", [4, 8, 16])
def test_narrow_columns_axis0(cols):
    rows = 250_003
    x = workloads.normal(rows * cols, np.float32, cols)
    got = gb.scan_batched(dev(x).reshape(rows, cols), axis=0).cpu().numpy()
    assert_scan_matches(got, as3(x, 1, rows, cols), "add", True, what="columns %d" % cols)
    assert gb.device_error() == gb.OK


@pytest.mark.parametrize("name", ["fp32_1e6x8_axis0", "struct32_1e6"])
def test_full_size_workloads(name):
    w = workloads.BY_NAME[name]
    x = w.make()
    if w.kind == "batched":
        rows, cols = w.shape
        got = gb.scan_batched(dev(x).reshape(rows, cols), axis=0).cpu().numpy()
        x3 = as3(x, 1, rows, cols)
    else:
        got = gb.scan_inclusive(dev(x), lanes=w.lanes).cpu().numpy()
        x3 = as3(x, 1, w.shape[0], w.lanes)
    assert_scan_matches(got, x3, "add", True, what=name)
    # The segments combine in a fixed order: the same bits on every call.
    again = (gb.scan_batched(dev(x).reshape(*w.shape), axis=0) if w.kind == "batched"
             else gb.scan_inclusive(dev(x), lanes=w.lanes)).cpu().numpy()
    assert np.array_equal(again, got)
    assert gb.device_error() == gb.OK


def test_unaligned_view_takes_the_lane_kernel():
    """A view that is not 16-byte aligned goes to the lane look-back kernel instead."""
    n, lanes = 20_001, 8
    base = workloads.normal(n * lanes + 1, np.float32, 3)
    got = gb.scan_inclusive(dev(base)[1:], lanes=lanes).cpu().numpy()
    assert_scan_matches(got, as3(base[1:], 1, n, lanes), "add", True, what="unaligned lanes")
