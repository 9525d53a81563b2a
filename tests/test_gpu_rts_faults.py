"""GPU parity of the reduce-then-scan variant, and failure detection: a tile that
never publishes its status makes its successors' bounded waits run out; the
kernel reports GB_ERR_TIMEOUT through the sticky device error and returns, and the
context stays usable.  No fault, trap or hang is involved: the wait limit is a
few milliseconds of the GPU's global timer."""
import numpy as np
import pytest
import torch

import oracle
import stream_compaction_decoupled_gb300 as gb
from stream_compaction_decoupled_gb300 import workloads
from parity import as3, assert_scan_matches

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    gb.load()
    yield
    torch.cuda.synchronize()


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


@pytest.mark.parametrize("dt", [np.int32, np.float32, np.float64, np.int64])
@pytest.mark.parametrize("op", ["add", "max", "min"])
@pytest.mark.parametrize("n", [1, 100, 4096, 4097, 3 * 4096 + 77, 1_000_003])
def test_rts_matches(dt, op, n):
    x = (workloads.normal(n, dt, n) if np.dtype(dt).kind == "f"
         else workloads.small_ints(n, n, -1000, 1000, dtype=dt))
    xd = dev(x)
    got = gb.scan_reduce_then_scan(xd, op).cpu().numpy()
    assert_scan_matches(got, as3(x, 1, n, 1), op, True, what="rts %s %s %d" % (np.dtype(dt).name, op, n))
    init = x[0] if op != "add" else None
    got = gb.scan_reduce_then_scan(xd, op, inclusive=False, init=init).cpu().numpy()
    assert_scan_matches(got, as3(x, 1, n, 1), op, False, init, what="rts excl")


@pytest.mark.parametrize("dt", [np.int32, np.float32, np.float64, np.int64, np.uint32])
@pytest.mark.parametrize("op", ["add", "max", "min", "mul"])
@pytest.mark.parametrize("n", [1, 100, 4097, 3 * 4096 + 77, 1_000_003, 12_000_001])
def test_scan_then_fan_matches(dt, op, n):
    """Scan-then-fan ([HB] 13.3.2): per-block scans, a scan of the block totals, the fan."""
    if dt == np.uint32 and not hasattr(torch, "uint32"):
        pytest.skip("no torch uint32")
    if op == "mul":
        x = (workloads.signs_pow2(n, dt, n) if np.dtype(dt).kind == "f"
             else workloads.odd_ints(n, n, np.int64).astype(dt))
    else:
        x = (workloads.normal(n, dt, n) if np.dtype(dt).kind == "f"
             else workloads.small_ints(n, n, 0 if np.dtype(dt).kind == "u" else -1000, 1000, dtype=dt))
    xd = dev(x)
    got = gb.scan_then_fan(xd, op).cpu().numpy()
    assert_scan_matches(got, as3(x, 1, n, 1), op, True, what="stf %s %s %d" % (np.dtype(dt).name, op, n))
    init = x[0] if op in ("max", "min") else (x[1 % n] if op == "add" else None)
    got = gb.scan_then_fan(xd, op, inclusive=False, init=init).cpu().numpy()
    assert_scan_matches(got, as3(x, 1, n, 1), op, False, init, what="stf excl %s %s" % (op, n))
    if n > 1:  # in place, through an unaligned view
        y = dev(np.concatenate([x[:1], x]))[1:]
        gb.scan_then_fan(y, op, out=y)
        assert_scan_matches(y.cpu().numpy(), as3(x, 1, n, 1), op, True, what="stf in place %s" % op)
    assert gb.device_error() == gb.OK


def test_scan_then_fan_full_size():
    w = workloads.BY_NAME["fp32_1e8"]
    x = w.make()
    got = gb.scan_then_fan(dev(x)).cpu().numpy()
    assert_scan_matches(got, as3(x, 1, x.size, 1), "add", True, what="stf fp32 1e8")
    assert gb.device_error() == gb.OK


def test_rts_full_size_matches_single_pass():
    w = workloads.BY_NAME["fp32_1e8"]
    x = w.make()
    xd = dev(x)
    got = gb.scan_reduce_then_scan(xd).cpu().numpy()
    assert_scan_matches(got, as3(x, 1, x.size, 1), "add", True, what="rts fp32 1e8")
    assert gb.device_error() == gb.OK


@pytest.fixture
def stall():
    yield
    gb.set_stalled_tile(-1)
    gb.set_wait_limit_ns(0)


@pytest.mark.parametrize("kind", ["rows_f32", "rows_f64", "lanes", "lanes_wide", "segments", "segments_f64",
                                  "compact_segments", "compact_tiles", "pack", "l2_resident", "partition",
                                  "segmented"])
def test_stalled_tile_times_out(stall, kind):
    n = 64 * 4096 if kind != "l2_resident" else 26_000_000
    x = workloads.uniform01(n, np.float32, 1)
    gb.set_wait_limit_ns(5_000_000)   # 5 ms
    gb.set_stalled_tile(3)
    if kind == "rows_f32":  # an unaligned view: the row kernel
        gb.scan_inclusive(dev(np.concatenate([x[:1], x]))[1:])
    elif kind == "rows_f64":
        gb.scan_inclusive(dev(np.concatenate([x[:1], x]).astype(np.float64))[1:])
    elif kind == "segments_f64":  # 512 chunks of 512 doubles -> 32 segments
        gb.scan_inclusive(dev(x.astype(np.float64)))
    elif kind == "lanes":
        gb.scan_inclusive(dev(x), lanes=8)
    elif kind == "lanes_wide":  # 65 lanes: 64-lane strips
        gb.scan_inclusive(dev(x[: n // 65 * 65]), lanes=65)
    elif kind == "segments":  # 512 chunks -> 16 segments; segment 3 never publishes
        gb.scan_inclusive(dev(x))
    elif kind == "l2_resident":  # one long row: the stalled index is a run of tiles
        gb.scan_inclusive(dev(x))
    elif kind == "compact_segments":
        gb.compact(dev(x), "lt", 0.5)
    elif kind == "segmented":  # head-flag scan: segment 3 never publishes its pair
        gb.scan_segmented(dev(x), dev(workloads.head_flags(n, 0.01, 2)))
    elif kind == "partition":  # every segment waits for all counts; segment 3 never publishes
        gb.partition(dev(x), "lt", 0.5)
    elif kind == "compact_tiles":
        gb.compact(dev(np.concatenate([x[:1], x]))[1:], "lt", 0.5)
    else:
        gb.pack_by_counts(dev((x * 8).astype(np.int32)), 8 * n)
    assert gb.device_error() == gb.ERR_TIMEOUT
    # The context is still usable and a normal call is exact again.
    gb.set_stalled_tile(-1)
    gb.set_wait_limit_ns(0)
    xi = workloads.small_ints(n, 2)
    assert np.array_equal(gb.scan_inclusive(dev(xi)).cpu().numpy(), oracle.scan(xi))
    assert gb.device_error() == gb.OK
