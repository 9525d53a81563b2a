"""GPU parity: segmented scans by head flags against the CPU oracle.

Integers, max and min compare exactly; float add within 1e-5 of each segment's prefix
sum of |x| (plus 1e-6); float multiply on +-2^k factors, exact in any bracketing.
"""
import numpy as np
import pytest
import torch

import oracle
import stream_compaction_decoupled_gb300 as gb
from stream_compaction_decoupled_gb300 import workloads

pytestmark = pytest.mark.gpu

NP = {"i32": np.int32, "u32": np.uint32, "i64": np.int64, "u64": np.uint64, "f32": np.float32,
      "f64": np.float64}


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    gb.load()
    yield
    torch.cuda.synchronize()


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def values(dt, op, n, seed):
    if op == "mul":
        if dt[0] == "f":
            return workloads.signs_pow2(n, NP[dt], seed)
        return workloads.odd_ints(n, seed, np.int64).astype(NP[dt])
    if dt[0] == "f":
        return workloads.normal(n, NP[dt], seed)
    if dt[0] == "u":  # the whole range: max/min must compare as unsigned
        return workloads.full_range_uints(n, seed, NP[dt])
    return workloads.small_ints(n, seed, -1000, 1000, dtype=np.int64).astype(NP[dt])


def check(got, x, fl, op, inclusive, init, what):
    want = oracle.scan_segmented(x, fl, op, inclusive, init)
    got = np.asarray(got)
    if x.dtype.kind != "f" or op != "add":
        ok = got.astype(want.dtype) == want
    else:
        mag = oracle.scan_segmented(np.abs(x.astype(np.float64)), fl, "add")
        if not inclusive:  # the exclusive value covers the elements before i in its segment
            mag = np.where(np.r_[True, fl[1:] != 0], 0.0, np.r_[0.0, mag[:-1]])
            if init is not None:
                mag = mag + abs(float(init))
        ok = np.abs(got.astype(np.float64) - want) <= 1e-5 * mag + 1e-6
    if not ok.all():
        i = int(np.flatnonzero(~ok)[0])
        raise AssertionError("%s: %d mismatches, first at %d: got %r want %r" % (what, int((~ok).sum()), i,
                                                                                 got[i], want[i]))


SIZES = [1, 7, 513, 16_384 + 5, 1_000_003, 6_000_017]
DENSITY = [0.0, 1e-4, 0.01, 0.5, 1.0]


@pytest.mark.parametrize("dt", ["i32", "f32", "f64", "i64"])
@pytest.mark.parametrize("op", ["add", "max", "min", "mul"])
@pytest.mark.parametrize("n", SIZES)
def test_segmented(dt, op, n):
    x = values(dt, op, n, n % 991)
    for p in DENSITY:
        fl = workloads.head_flags(n, p, n % 7 + int(p * 100))
        xd, fd = dev(x), dev(fl)
        check(gb.scan_segmented(xd, fd, op).cpu().numpy(), x, fl, op, True, None, "%s %s n=%d p=%g" % (dt, op, n, p))
        init = (x[0] if op in ("max", "min") else None) if n > 0 else None
        got = gb.scan_segmented(xd, fd, op, inclusive=False, init=init).cpu().numpy()
        check(got, x, fl, op, False, init, "%s %s excl n=%d p=%g" % (dt, op, n, p))
    assert gb.device_error() == gb.OK


@pytest.mark.parametrize("dt", ["u32", "u64"])
def test_segmented_unsigned(dt):
    n = 300_001
    x = values(dt, "add", n, 3)
    fl = workloads.head_flags(n, 0.003, 4)
    check(gb.scan_segmented(dev(x), dev(fl), "add").cpu().numpy(), x, fl, "add", True, None, dt)


@pytest.mark.parametrize("offs", [(1, 0, 0), (0, 3, 0), (0, 0, 5), (1, 1, 1)])
def test_segmented_unaligned_and_in_place(offs):
    """Views off 16-byte alignment take the element-wise path; in == out is allowed."""
    n = 1_000_003
    ox, of, oo = offs
    x = values("f32", "add", n + ox, 9)
    fl = workloads.head_flags(n + of, 0.002, 10)
    xd = dev(x)[ox:]
    fd = dev(fl)[of:]
    out = torch.empty(n + oo, dtype=torch.float32, device="cuda")[oo:]
    got = gb.scan_segmented(xd, fd, out=out).cpu().numpy()
    check(got, x[ox:], fl[of:], "add", True, None, "unaligned %s" % (offs,))
    y = dev(x[ox:])
    gb.scan_segmented(y, fd, "add", out=y)
    check(y.cpu().numpy(), x[ox:], fl[of:], "add", True, None, "in place")


def test_segmented_equal_segments_match_batched_rows():
    rows, cols = 1000, 4097
    x = values("i32", "add", rows * cols, 11)
    fl = np.zeros(rows * cols, np.uint8)
    fl[::cols] = 1
    got = gb.scan_segmented(dev(x), dev(fl)).cpu().numpy()
    rowscan = gb.scan_batched(dev(x).reshape(rows, cols), axis=1).cpu().numpy().reshape(-1)
    assert np.array_equal(got, rowscan)


def test_segmented_errors():
    x = dev(np.arange(10, dtype=np.float32))
    with pytest.raises(gb.GbError) as e:
        gb.scan_segmented(x, dev(np.zeros(10, np.uint8)), "max", inclusive=False)
    assert e.value.code == gb.ERR_NO_IDENTITY
    with pytest.raises(ValueError):
        gb.scan_segmented(x, dev(np.zeros(9, np.uint8)))


def test_segmented_full_size_workload():
    w = workloads.BY_NAME["fp32_1e7_segmented"]
    x = w.make()
    fl = workloads.head_flags(x.size, w.extra["p_head"], w.extra["flag_seed"])
    check(gb.scan_segmented(dev(x), dev(fl)).cpu().numpy(), x, fl, "add", True, None, w.name)
    assert gb.device_error() == gb.OK
