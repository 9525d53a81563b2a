"""GPU parity: the multiply operator (cumprod) through every kernel family, and the
wider lane-vector elements (the 32-byte struct, elements up to 2080 bytes with and
without a neutral element), against the CPU oracle.

Integer products wrap to their low bits and are compared bit-exactly.  Float
products of +-2^k factors are exact in any bracketing, so those compare
bit-exactly too; other float products are held to the rounding bound of a
k-factor product (tests/parity.py).
"""
import numpy as np
import pytest
import torch

import oracle
import stream_compaction_decoupled_gb300 as gb
from stream_compaction_decoupled_gb300 import workloads
from parity import as3, assert_scan_matches

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


def host(t):
    return t.cpu().numpy()


def factors(dt, n, seed, exact=True):
    """Odd integers (never 0 modulo 2^w), exact +-2^k floats, or log-normal floats."""
    if dt[0] in "iu":
        x = workloads.odd_ints(n, seed, np.int64)
        return x.astype(NP[dt]) if dt[0] == "i" else (x & 0x7FFFFFFF | 1).astype(NP[dt])
    if exact:
        return workloads.signs_pow2(n, NP[dt], seed)
    return workloads.lognormal(n, NP[dt], seed, 0.02 if n <= 100_000 else 0.004)


def check_mul(got, x3, inclusive=True, init=None, exact=True, what=""):
    if exact:
        want = oracle.scan3(x3, "mul", inclusive, init)
        got = np.asarray(got).reshape(x3.shape)
        ok = got.astype(want.dtype) == want
        if not ok.all():
            bad = np.argwhere(~ok)[:3]
            raise AssertionError("%s: %d mismatches, first at %s: got %r want %r" % (
                what, int((~ok).sum()), bad[0].tolist(), got[tuple(bad[0])], want[tuple(bad[0])]))
    else:
        assert_scan_matches(got, x3, "mul", inclusive, init, what=what)


# ---- one row: the segment kernels (<= 96 MiB, fp64 thread-contiguous) ---------------

SIZES = [1, 17, 513, 16_389, 1_245_185, 3_000_017]


@pytest.mark.parametrize("dt", ["i32", "u32", "i64", "u64", "f32", "f64"])
@pytest.mark.parametrize("n", SIZES)
def test_mul_one_row(dt, n):
    x = factors(dt, n, n % 977)
    xd = dev(x)
    check_mul(host(gb.scan_inclusive(xd, "mul")), as3(x, 1, n, 1), what="mul %s n=%d" % (dt, n))
    check_mul(host(gb.scan_exclusive(xd, "mul")), as3(x, 1, n, 1), False, what="mul excl %s" % dt)
    init = x[:1].copy()
    check_mul(host(gb.scan_exclusive(xd, "mul", init=init)), as3(x, 1, n, 1), False, init, what="mul excl init")
    assert gb.device_error() == gb.OK


@pytest.mark.parametrize("dt", ["f32", "f64"])
@pytest.mark.parametrize("n", [100_000, 3_000_017])
def test_mul_rounding_bound(dt, n):
    x = factors(dt, n, 5, exact=False)
    check_mul(host(gb.scan_inclusive(dev(x), "mul")), as3(x, 1, n, 1), exact=False, what="lognormal %s" % dt)


# ---- one long row (L2-resident look-back kernel) and unaligned views (row kernel) -----

@pytest.mark.parametrize("dt,n", [("f32", 26_000_003), ("i32", 26_000_000), ("i64", 13_000_003)])
def test_mul_l2_resident(dt, n):
    x = factors(dt, n, 3)
    xd = dev(x)
    check_mul(host(gb.scan_inclusive(xd, "mul")), as3(x, 1, n, 1), what="stash mul %s" % dt)
    check_mul(host(gb.scan_exclusive(xd, "mul")), as3(x, 1, n, 1), False, what="stash mul excl %s" % dt)
    assert gb.device_error() == gb.OK


@pytest.mark.parametrize("dt", ["i32", "f32", "f64"])
@pytest.mark.parametrize("n", [4097, 1_000_003])
def test_mul_row_kernel(dt, n):
    base = factors(dt, n + 1, 11)
    xd = dev(base)[1:]
    check_mul(host(gb.scan_inclusive(xd, "mul")), as3(base[1:], 1, n, 1), what="rows mul %s" % dt)


# ---- batched and lane vectors -------------------------------------------------------

@pytest.mark.parametrize("dt", ["i32", "f32", "f64", "i64"])
@pytest.mark.parametrize("shape", [(3, 70_001), (5, 65536), (300, 33), (4096, 16)])
def test_mul_batched_axis1(dt, shape):
    rows, cols = shape
    x = factors(dt, rows * cols, rows + cols)
    got = host(gb.scan_batched(dev(x).reshape(rows, cols), axis=1, op="mul"))
    check_mul(got, as3(x, rows, cols, 1), what="mul axis1 %s %s" % (dt, shape))


@pytest.mark.parametrize("dt", ["i32", "f32", "f64", "i64"])
@pytest.mark.parametrize("shape", [(1000, 17), (4096, 64), (513, 65), (300_000, 17)])
def test_mul_columns_and_lanes(dt, shape):
    rows, cols = shape
    # each column its own factor sequence (a column of one flattened +-2^k walk would
    # be a strided subsequence, whose products are not bounded)
    x = np.ascontiguousarray(factors(dt, rows * cols, rows * 3 + cols).reshape(cols, rows).T).reshape(-1)
    xd = dev(x).reshape(rows, cols)
    check_mul(host(gb.scan_batched(xd, axis=0, op="mul")), as3(x, 1, rows, cols), what="mul axis0 %s %s" % (dt, shape))
    got = host(gb.scan_batched(xd, axis=0, op="mul", inclusive=False))
    check_mul(got, as3(x, 1, rows, cols), False, what="mul axis0 excl")
    assert gb.device_error() == gb.OK


def test_mul_reduce_then_scan_and_host():
    x = factors("f32", 5_000_003, 8)
    got = host(gb.scan_reduce_then_scan(dev(x), "mul"))
    check_mul(got, as3(x, 1, x.size, 1), what="rts mul")
    xi = factors("i32", 5_000_003, 9)
    got = gb.scan_inclusive_host(torch.from_numpy(xi).pin_memory(), "mul", chunk_elems=1 << 20)
    torch.cuda.synchronize()
    check_mul(got.numpy(), as3(xi, 1, xi.size, 1), what="host mul")


# ---- wider elements: 32-byte structs, and elements up to 2080 bytes -------------------

@pytest.mark.parametrize("lanes", [8, 16, 130, 520])
@pytest.mark.parametrize("op", ["add", "max"])
def test_wide_elements(lanes, op):
    n = max(64, 2_000_000 // lanes)
    x = workloads.normal(n * lanes, np.float32, lanes)
    xd = dev(x)
    got = host(gb.scan_inclusive(xd, op, lanes=lanes))
    assert_scan_matches(got, as3(x, 1, n, lanes), op, True, what="%d lanes %s" % (lanes, op))
    init = x[:lanes].copy() if op == "max" else None
    got = host(gb.scan_exclusive(xd, op, init=init, lanes=lanes))
    assert_scan_matches(got, as3(x, 1, n, lanes), op, False, init, what="%d lanes %s excl" % (lanes, op))
    assert gb.device_error() == gb.OK


# ---- the full-size workloads ----------------------------------------------------------

@pytest.mark.parametrize("name", ["fp32_1e7_cumprod", "i32_1e6_cumprod", "struct32_1e6", "elem2080_2e4",
                                  "elem2080_2e4_max"])
def test_full_size_workload(name):
    w = workloads.BY_NAME[name]
    x = w.make()
    n = w.shape[0]
    got = host(gb.scan_inclusive(dev(x), w.op, lanes=w.lanes))
    assert_scan_matches(got, as3(x, 1, n, w.lanes), w.op, True, what=name)
    assert gb.device_error() == gb.OK
