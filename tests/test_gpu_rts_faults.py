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
             else workloads.full_range_uints(n, n, dt) if np.dtype(dt).kind == "u"
             else workloads.small_ints(n, n, -1000, 1000, dtype=dt))
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
                                  "segmented", "affine_segments", "affine_tiles"])
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
    elif kind in ("affine_segments", "affine_tiles"):  # composition of affine maps, two lanes
        xi = dev(workloads.small_ints(n, 5))
        gb.scan_inclusive(xi if kind == "affine_segments" else dev(workloads.small_ints(n + 2, 5))[2:], "affine",
                          lanes=2)
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


def test_per_call_status_keeps_streams_apart(stall):
    """gb_last_device_error(temp, stream) reads the status word in a call's own
    scratch: a call that timed out on one stream does not show in an independent
    call on another stream with its own scratch, and the next call with the first
    scratch clears it.  The device-wide word sees both."""
    n = 64 * 4096
    x = dev(workloads.uniform01(n, np.float32, 1))
    nbytes = gb.temp_storage_bytes(gb.KIND_SCAN, gb.F32, 1, n)
    temp_a = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    temp_b = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    assert gb.device_error() == gb.OK
    gb.set_wait_limit_ns(5_000_000)   # 5 ms
    gb.set_stalled_tile(3)
    gb.scan_inclusive(x, temp=temp_a)                 # segment 3 never publishes
    torch.cuda.synchronize()
    gb.set_stalled_tile(-1)
    gb.set_wait_limit_ns(0)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        out_b = gb.scan_inclusive(x, temp=temp_b, stream=side)
    assert gb.last_device_error(temp_b, side) == gb.OK
    assert gb.last_device_error(temp_a) == gb.ERR_TIMEOUT
    assert gb.last_device_error(temp_a) == gb.ERR_TIMEOUT   # reading does not clear it
    assert gb.device_error() == gb.ERR_TIMEOUT              # the device-wide view
    want = oracle.scan(x.cpu().numpy())
    assert_scan_matches(out_b.cpu().numpy(), as3(x.cpu().numpy(), 1, n, 1), "add", True, what="side stream")
    gb.scan_inclusive(x, temp=temp_a)                 # the next call clears the word
    assert gb.last_device_error(temp_a) == gb.OK
    del want


def test_per_call_status_of_host_scan_and_comparators(stall):
    """The host-array scan collects every chunk's status in its work area's header;
    the three-launch comparators clear their header too."""
    n = 8 * 65_536
    xh = torch.from_numpy(workloads.small_ints(n, 3)).pin_memory()
    work = torch.empty(gb.host_scan_work_bytes(torch.int32, n, 65_536), dtype=torch.uint8, device="cuda")
    gb.set_wait_limit_ns(5_000_000)
    gb.set_stalled_tile(0)     # segment 0 of every chunk scan never publishes
    gb.scan_inclusive_host(xh, chunk_elems=65_536, work=work)
    assert gb.last_device_error(work) == gb.ERR_TIMEOUT
    assert gb.device_error() == gb.ERR_TIMEOUT
    gb.set_stalled_tile(-1)
    gb.set_wait_limit_ns(0)
    out = gb.scan_inclusive_host(xh, chunk_elems=65_536, work=work)
    assert gb.last_device_error(work) == gb.OK
    assert np.array_equal(out.numpy(), oracle.scan(xh.numpy()))
    xd = dev(workloads.normal(1_000_003, np.float32, 4))
    temp = torch.empty(gb.temp_storage_bytes(gb.KIND_REDUCE_THEN_SCAN, gb.F32, 1, xd.numel()), dtype=torch.uint8,
                       device="cuda")
    temp.fill_(0xff)           # a stale error word must not survive the call's clear
    gb.scan_reduce_then_scan(xd, temp=temp)
    assert gb.last_device_error(temp) == gb.OK
    temp.fill_(0xff)
    gb.scan_then_fan(xd, temp=temp)
    assert gb.last_device_error(temp) == gb.OK
    assert gb.device_error() == gb.OK
