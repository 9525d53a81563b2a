"""GPU parity: scans under composition of affine maps, an operator that is
associative but not commutative, through the C ABI against the CPU oracle.

Element i is the map y -> a_i*y + b_i of an integer type (lanes = 2); the earlier map
is applied first.  The kernels must combine in index order everywhere (The CUDA
Handbook, 13.3.4: its packed descriptor assumes a commutative operator), so any
reordering shows as wrong bits.  Results are compared bit for bit.  Cases cover the
segment kernel (aligned rows up to 96 MiB: one or several chunks per warp, several
segments) and the decoupled look-back tile kernel (views that are not 16-byte
aligned, and rows past 96 MiB), inclusive and exclusive, with and without an
initial map, and repeated calls of the look-back path.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import stream_compaction_decoupled_gb300 as gb
from stream_compaction_decoupled_gb300 import workloads

pytestmark = pytest.mark.gpu

NP = {"i32": np.int32, "i64": np.int64, "u32": np.uint32, "u64": np.uint64}


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    gb.load()
    yield
    torch.cuda.synchronize()


def maps(dt, n, seed):
    """n maps (a, b) with a and b over the type's whole range (products wrap)."""
    npt = NP[dt]
    bits = 8 * np.dtype(npt).itemsize
    u = workloads.full_range_uints(2 * n, seed, np.uint32 if bits == 32 else np.uint64)
    return u.view(npt) if np.dtype(npt).kind == "i" else u


def on_device(x, off):
    """x (2n values) on the device, `off` maps past a 256-byte aligned allocation,
    and an output view like it."""
    if dt_unsupported(x.dtype):
        pytest.skip("no torch dtype")
    base = torch.empty(x.size + 2 * off, dtype=torch.from_numpy(x[:2]).dtype, device="cuda")
    base[2 * off:].copy_(torch.from_numpy(x))
    out = torch.empty_like(base)
    return base[2 * off:], out[2 * off:]


def dt_unsupported(npdt):
    return np.dtype(npdt).kind == "u" and not hasattr(torch, "uint32")


def check(got, x, inclusive, init, what):
    want = oracle.scan_affine(x, inclusive, init)
    g = got.cpu().numpy()
    if not np.array_equal(g, want):
        bad = np.flatnonzero(g != want)
        raise AssertionError("%s: %d values differ, first at map %d: got %s want %s" % (
            what, bad.size, bad[0] // 2, g[bad[0] // 2 * 2: bad[0] // 2 * 2 + 2], want[bad[0] // 2 * 2: bad[0] // 2 * 2 + 2]))


# Segment kernel chunk: 256 (32-bit) or 128 (64-bit) maps; 152 SMs x 2 CTAs x 16 warps.
SIZES = [1, 2, 7, 8, 9, 255, 256, 257, 4095, 10_001, 1_000_003, 5_000_017]


@pytest.mark.parametrize("dt", ["i32", "u32", "i64", "u64"])
@pytest.mark.parametrize("n", SIZES)
def test_affine_segment_kernel(dt, n):
    x = maps(dt, n, 100 + n % 97)
    xd, out = on_device(x, 0)
    gb.scan_inclusive(xd, "affine", lanes=2, out=out)
    check(out, x, True, None, "%s incl n=%d" % (dt, n))
    gb.scan_exclusive(xd, "affine", lanes=2, out=out)
    check(out, x, False, None, "%s excl n=%d" % (dt, n))
    init = np.array([3, -7], dtype=np.int64).astype(NP[dt])
    gb.scan_exclusive(xd, "affine", init=init, lanes=2, out=out)
    check(out, x, False, init, "%s excl init n=%d" % (dt, n))
    assert gb.device_error() == gb.OK


@pytest.mark.parametrize("dt", ["i32", "u32"])
@pytest.mark.parametrize("n", [1, 3, 2047, 2048, 2049, 100_003, 3_000_001])
def test_affine_lookback_kernel_unaligned(dt, n):
    """A view one map (8 bytes) past a 16-byte boundary takes the tile kernel."""
    x = maps(dt, n, 200 + n % 89)
    xd, out = on_device(x, 1)
    gb.scan_inclusive(xd, "affine", lanes=2, out=out)
    check(out, x, True, None, "%s tiles incl n=%d" % (dt, n))
    init = np.array([5, 11], dtype=np.int64).astype(NP[dt])
    gb.scan_exclusive(xd, "affine", init=init, lanes=2, out=out)
    check(out, x, False, init, "%s tiles excl n=%d" % (dt, n))
    assert gb.device_error() == gb.OK


@pytest.mark.parametrize("dt,n", [("u32", 12_600_001), ("i64", 6_300_007)])
def test_affine_lookback_kernel_past_l2(dt, n):
    """Rows past 96 MiB take the tile kernel whatever their alignment (64-bit maps are
    16 bytes, so every view of them is aligned)."""
    x = maps(dt, n, 300)
    xd, out = on_device(x, 0)
    gb.scan_inclusive(xd, "affine", lanes=2, out=out)
    check(out, x, True, None, "%s past L2 incl n=%d" % (dt, n))
    gb.scan_exclusive(xd, "affine", lanes=2, out=out)
    check(out, x, False, None, "%s past L2 excl n=%d" % (dt, n))
    assert gb.device_error() == gb.OK


def test_affine_lookback_repeated():
    """The look-back under many interleavings: 60 calls, the same bits every time."""
    n = 1_500_001
    x = maps("i32", n, 400)
    xd, out = on_device(x, 1)
    want = torch.from_numpy(oracle.scan_affine(x)).cuda()
    for k in range(60):
        gb.scan_inclusive(xd, "affine", lanes=2, out=out)
        assert torch.equal(out, want), "call %d differs" % k
    assert gb.device_error() == gb.OK


def test_affine_recurrence_and_equal_maps():
    """The b lane of the inclusive scan solves y_i = a_i y_{i-1} + b_i; equal maps give
    (a^(i+1), b (1 + a + ... + a^i)) (checked on the device against numpy powers)."""
    n = 2_000_003
    a, b = 3, 5
    x = np.tile(np.array([a, b], dtype=np.int64), n)
    xd, out = on_device(x, 0)
    gb.scan_inclusive(xd, "affine", lanes=2, out=out)
    got = out.cpu().numpy().reshape(n, 2).astype(np.uint64)
    pw = np.cumprod(np.full(n, a, dtype=np.uint64), dtype=np.uint64)           # a^(i+1) mod 2^64
    # 1 + a + ... + a^i (all uint64: an int64 operand would promote the sum to float64)
    geo = np.cumsum(np.concatenate([np.ones(1, dtype=np.uint64), pw[:-1]]), dtype=np.uint64)
    assert np.array_equal(got[:, 0], pw)
    assert np.array_equal(got[:, 1], (geo * np.uint64(b)).astype(np.uint64))


def test_affine_argument_errors():
    lib = gb.load()
    x = torch.zeros(64, dtype=torch.int32, device="cuda")
    p = ctypes.c_void_p(x.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.gb_scan_inclusive(gb.F32, 2, gb.AFFINE, p, p, 32, None, 0, s) == gb.ERR_UNSUPPORTED
    assert lib.gb_scan_inclusive(gb.I32, 1, gb.AFFINE, p, p, 32, None, 0, s) == gb.ERR_UNSUPPORTED
    assert lib.gb_scan_inclusive(gb.I32, 3, gb.AFFINE, p, p, 16, None, 0, s) == gb.ERR_UNSUPPORTED
    q = ctypes.c_void_p(x.data_ptr() + 2)
    assert lib.gb_scan_inclusive(gb.I32, 2, gb.AFFINE, q, q, 16, None, 0, s) == gb.ERR_INVALID
    assert lib.gb_scan_batched(gb.I32, 2, gb.AFFINE, 1, p, p, 4, 4, 1, None, None, 0, s) == gb.ERR_UNSUPPORTED
    assert lib.gb_scan_then_fan(gb.I32, gb.AFFINE, 1, p, p, 16, None, None, 0, s) == gb.ERR_UNSUPPORTED
    assert lib.gb_scan_inclusive(gb.I32, 2, gb.AFFINE, p, p, 0, None, 0, s) == gb.OK
    assert gb.device_error() == gb.OK


def test_affine_full_size_workload():
    """The benchmark's i32_1e7_affine workload, bit for bit, inclusive and exclusive."""
    w = workloads.BY_NAME["i32_1e7_affine"]
    x = w.make()
    xd, out = on_device(x, 0)
    gb.scan_inclusive(xd, "affine", lanes=2, out=out)
    check(out, x, True, None, "i32_1e7_affine incl")
    gb.scan_exclusive(xd, "affine", lanes=2, out=out)
    check(out, x, False, None, "i32_1e7_affine excl")
    assert gb.device_error() == gb.OK
