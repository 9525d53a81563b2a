"""GPU parity: single-pass 1-D scans through the C ABI against the CPU oracle.

Small cases span several tiles and a ragged tail for every type, operator and
kind; the full-size cases are the 1-D workloads of the benchmark table (int32
1e6, fp32 1e8, fp64 1e7, fp32 1e7 max) compared element by element.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import stream_compaction_decoupled_gb300 as gb
from stream_compaction_decoupled_gb300 import workloads
from parity import as3, assert_scan_matches

pytestmark = pytest.mark.gpu

DTYPES = {"i32": (np.int32, torch.int32), "i64": (np.int64, torch.int64),
          "f32": (np.float32, torch.float32), "f64": (np.float64, torch.float64)}
if hasattr(torch, "uint32"):
    DTYPES["u32"] = (np.uint32, torch.uint32)
    DTYPES["u64"] = (np.uint64, torch.uint64)

# Tile sizes of the row kernel: 4096 (4-byte) and 2048 (8-byte) elements.
SIZES = [1, 2, 31, 32, 33, 2047, 2048, 2049, 4095, 4096, 4097, 3 * 4096 + 77, 40_000 + 3]


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    gb.load()
    yield
    torch.cuda.synchronize()


def make(dt: str, n: int, seed: int) -> np.ndarray:
    npt = DTYPES[dt][0]
    if dt.startswith("f"):
        return workloads.normal(n, npt, seed)
    if dt.startswith("u"):  # the whole range: max/min must compare as unsigned
        return workloads.full_range_uints(n, seed, npt)
    return workloads.small_ints(n, seed, -1000, 1000, dtype=npt)


def to_dev(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def to_host(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


@pytest.mark.parametrize("dt", sorted(DTYPES))
@pytest.mark.parametrize("op", ["add", "max", "min"])
@pytest.mark.parametrize("n", SIZES)
def test_scan_small(dt, op, n):
    x = make(dt, n, 1000 + n)
    xd = to_dev(x)
    got = to_host(gb.scan_inclusive(xd, op))
    assert_scan_matches(got, as3(x, 1, n, 1), op, True, what="%s %s incl n=%d" % (dt, op, n))
    init = x[0] if op != "add" else None
    got = to_host(gb.scan_exclusive(xd, op, init=init))
    assert_scan_matches(got, as3(x, 1, n, 1), op, False, init, what="%s %s excl n=%d" % (dt, op, n))


@pytest.mark.parametrize("dt", ["i32", "f64"])
def test_exclusive_add_with_init(dt):
    n = 3 * 4096 + 5
    x = make(dt, n, 7)
    init = DTYPES[dt][0](11)
    got = to_host(gb.scan_exclusive(to_dev(x), "add", init=init))
    assert_scan_matches(got, as3(x, 1, n, 1), "add", False, init, what="excl add init")


def test_all_ones_closed_form():
    for dt, n in (("i32", 10_000_019), ("f32", 1 << 24), ("f64", 3 * 2048 + 1)):
        x = np.ones(n, dtype=DTYPES[dt][0])
        got = to_host(gb.scan_inclusive(to_dev(x)))
        assert np.array_equal(got, np.arange(1, n + 1, dtype=np.float64).astype(got.dtype)), dt
        got = to_host(gb.scan_exclusive(to_dev(x)))
        assert np.array_equal(got, np.arange(0, n, dtype=np.float64).astype(got.dtype)), dt


def test_last_inclusive_is_reduction_and_excl_relation():
    x = workloads.small_ints(1_000_003, 9, -100_000, 100_000)
    s = to_host(gb.scan_inclusive(to_dev(x))).astype(np.int64)
    e = to_host(gb.scan_exclusive(to_dev(x))).astype(np.int64)
    assert s[-1] == int(x.astype(np.int64).sum())
    assert np.array_equal(e, s - x)


def test_int32_wraparound():
    n = 5 * 4096 + 3
    x = np.full(n, 2**31 - 7, dtype=np.int32)
    x[::3] = -(2**31) + 5
    got = to_host(gb.scan_inclusive(to_dev(x)))
    assert np.array_equal(got, oracle.scan(x))


def test_max_scan_monotone_closed_forms():
    up = np.arange(-50_000, 50_000, dtype=np.int32)
    assert np.array_equal(to_host(gb.scan_inclusive(to_dev(up), "max")), up)
    down = up[::-1].copy()
    assert np.all(to_host(gb.scan_inclusive(to_dev(down), "max")) == down[0])


def test_unaligned_and_inplace():
    base = workloads.normal(3 * 4096 + 9, np.float32, 3)
    bd = to_dev(base)
    x = bd[1:]                      # 4-byte offset: no 16-byte alignment, plain-load path
    out = torch.empty(x.numel() + 1, dtype=x.dtype, device=x.device)[1:]
    got = to_host(gb.scan_inclusive(x, out=out))
    assert_scan_matches(got, as3(base[1:], 1, x.numel(), 1), "add", True, what="unaligned")
    y = to_dev(base)
    gb.scan_inclusive(y, out=y)     # in place
    assert_scan_matches(to_host(y), as3(base, 1, base.size, 1), "add", True, what="in place")


def test_library_allocated_temp():
    """temp = NULL: the library draws scratch from the stream-ordered allocator."""
    x = workloads.normal(100_000, np.float32, 4)
    xd, out = to_dev(x), torch.empty(100_000, dtype=torch.float32, device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = gb.load().gb_scan_inclusive(gb.F32, 1, gb.ADD, ctypes.c_void_p(xd.data_ptr()),
                                     ctypes.c_void_p(out.data_ptr()), x.size, None, 0, s)
    assert rc == gb.OK
    assert_scan_matches(to_host(out), as3(x, 1, x.size, 1), "add", True, what="temp NULL")


def test_side_stream_calls_without_temp():
    """Calls on a side stream with scratch chosen by the binding: it allocates the
    scratch on that stream, so allocations on the default stream made while the call
    runs cannot be handed the same block."""
    side = torch.cuda.Stream()
    x = to_dev(workloads.small_ints(3_000_017, 5, -9, 10))
    want = to_dev(oracle.scan(x.cpu().numpy()))
    side.wait_stream(torch.cuda.current_stream())
    outs = []
    for _ in range(10):
        with torch.cuda.stream(side):
            outs.append(gb.scan_inclusive(x, stream=side))
        junk = torch.full((1 << 16,), -1, dtype=torch.int32, device="cuda")  # default-stream work
        junk += 1
    torch.cuda.synchronize()
    for k, o in enumerate(outs):
        assert torch.equal(o, want), "side-stream call %d differs" % k
    assert gb.device_error() == gb.OK


def test_argument_errors():
    lib = gb.load()
    x = torch.zeros(4096, dtype=torch.float32, device="cuda")
    p = ctypes.c_void_p(x.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.gb_scan_exclusive(gb.F32, 1, gb.MAX, p, p, 4096, None, None, 0, s) == gb.ERR_NO_IDENTITY
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    assert lib.gb_scan_inclusive(gb.F32, 1, gb.ADD, p, p, 4096, ctypes.c_void_p(small.data_ptr()), 16,
                                 s) == gb.ERR_TEMP
    assert lib.gb_scan_inclusive(9, 1, gb.ADD, p, p, 4096, None, 0, s) == gb.ERR_INVALID
    assert lib.gb_scan_inclusive(gb.F32, 0, gb.ADD, p, p, 4096, None, 0, s) == gb.ERR_INVALID
    assert lib.gb_scan_inclusive(gb.F32, 1, gb.ADD, None, p, 4096, None, 0, s) == gb.ERR_INVALID
    assert lib.gb_scan_inclusive(gb.F32, 1, gb.ADD, p, p, 0, None, 0, s) == gb.OK
    assert gb.device_error() == gb.OK


def test_repeated_calls_segment_kernel():
    """An aligned 1e7 int32 row takes the segment kernel, which has no look-back: each
    segment gathers every earlier segment's aggregate once they are all published.
    Thirty calls, whichever segments publish first, must give the same bits."""
    x = workloads.small_ints(10_000_000, 77, -5, 6)
    xd = to_dev(x)
    want = oracle.scan(x)
    out = torch.empty_like(xd)
    for _ in range(30):
        gb.scan_inclusive(xd, out=out)
        assert np.array_equal(to_host(out), want)
    assert gb.device_error() == gb.OK


# ---- stress of the decoupled look-back itself (many calls, bit-exact) ----------------
# Integer add is exact in any bracketing, so every call must give the oracle's bits
# whatever order the tiles publish in and however far each look-back walks.

@pytest.mark.parametrize("dt,n", [("i32", 3000 * 4096 + 1), ("i64", 3000 * 2048 + 1), ("i32", 300 * 4096 + 5)])
def test_lookback_stress_row_kernel(dt, n):
    """A view 4 bytes past a 16-byte boundary can only take the row kernel: one CTA
    per tile (4096 four-byte or 2048 eight-byte elements), each tile's warp 0 looking
    back over its predecessors' status words (one packed word for 4-byte values, a
    flag and a value slot for 8-byte ones).  3000 tiles per call, 100 calls."""
    npt = DTYPES[dt][0]
    base = workloads.small_ints(n + 1, 91 + n % 7, -7, 8, dtype=npt)
    want = to_dev(oracle.scan(base[1:]))
    xd = to_dev(base)[1:]
    out = torch.empty(n + 1, dtype=xd.dtype, device=xd.device)[1:]   # unaligned output too
    for k in range(100):
        gb.scan_inclusive(xd, out=out)
        assert torch.equal(out, want), "call %d differs" % k
    assert gb.device_error() == gb.OK


@pytest.mark.parametrize("dt,n", [("i32", 30_000_001), ("i64", 13_000_003)])
def test_lookback_stress_l2_resident_kernel(dt, n):
    """An aligned row past 96 MiB takes the L2-resident kernel: persistent CTAs claim
    runs of tiles and look back over run status words.  20 calls, in place and not."""
    npt = DTYPES[dt][0]
    x = workloads.small_ints(n, 92, -7, 8, dtype=npt)
    want = to_dev(oracle.scan(x))
    xd = to_dev(x)
    out = torch.empty_like(xd)
    for k in range(20):
        if k % 4 == 3:
            y = xd.clone()
            gb.scan_inclusive(y, out=y)
            assert torch.equal(y, want), "in-place call %d differs" % k
        else:
            gb.scan_inclusive(xd, out=out)
            assert torch.equal(out, want), "call %d differs" % k
    assert gb.device_error() == gb.OK


# ---- the full-size 1-D workloads, compared element by element ------------------

@pytest.mark.parametrize("name", ["i32_1e6", "i32_1e6_excl", "fp32_1e8", "fp32_1e8_excl", "fp64_1e7",
                                  "fp32_1e7_max"])
def test_full_size_workload(name):
    w = workloads.BY_NAME[name]
    x = w.make()
    xd = to_dev(x)
    if w.inclusive:
        got = to_host(gb.scan_inclusive(xd, w.op))
        assert_scan_matches(got, as3(x, 1, x.size, 1), w.op, True, what=name)
    else:
        got = to_host(gb.scan_exclusive(xd, w.op))
        assert_scan_matches(got, as3(x, 1, x.size, 1), w.op, False, what=name)
    if w.op == "max":  # exclusive max with init = x_0 (identity-free operator)
        got = to_host(gb.scan_exclusive(xd, "max", init=x[0]))
        assert_scan_matches(got, as3(x, 1, x.size, 1), "max", False, x[0], what=name + " excl")
    del xd
    assert gb.device_error() == gb.OK


# ---- the segment kernels (one aligned row of at most 96 MiB) -----------------------
# A warp's chunk holds 512 four-byte or 256 eight-byte elements; 152 SMs x 32 warps
# saturate at 4864 chunks (2,490,368 / 1,245,184 elements), beyond which warps take
# several chunks.  fp64 runs the thread-contiguous variant: chunks of 32 lanes x 16
# doubles, 152 SMs x 16 warps, so 2432 chunks (1,245,184 doubles) saturate it.

SEG_SMALL = [1, 15, 16, 17, 511, 512, 513, 16_384 + 5, 2 * 16_384 + 1, 1_245_184, 1_245_184 + 1,
             2_490_368, 2_490_368 + 1, 3_000_017]


@pytest.mark.parametrize("dt", ["i32", "u32", "f32", "i64", "u64", "f64"])
@pytest.mark.parametrize("op", ["add", "max", "min"])
@pytest.mark.parametrize("n", SEG_SMALL)
def test_segment_path(dt, op, n):
    if dt not in DTYPES:
        pytest.skip("no torch dtype")
    x = make(dt, n, 7 + n % 1000)
    xd = to_dev(x)
    got = to_host(gb.scan_inclusive(xd, op))
    assert_scan_matches(got, as3(x, 1, n, 1), op, True, what="seg %s %s incl n=%d" % (dt, op, n))
    init = x[0] if op != "add" else None
    got = to_host(gb.scan_exclusive(xd, op, init=init))
    assert_scan_matches(got, as3(x, 1, n, 1), op, False, init, what="seg %s %s excl n=%d" % (dt, op, n))
    assert gb.device_error() == gb.OK


@pytest.mark.parametrize("dt,n", [("f32", 10_000_019), ("i32", 25_165_824), ("f32", 25_165_824),
                                  ("u64", 12_582_912), ("i64", 7_000_003), ("f64", 10_000_019),
                                  ("f64", 12_582_912)])
def test_segment_path_large(dt, n):
    """Up to the 96 MiB limit, where every warp takes several chunks."""
    if dt not in DTYPES:
        pytest.skip("no torch dtype")
    x = make(dt, n, n % 1000)
    xd = to_dev(x)
    for op in ("add", "max"):
        got = to_host(gb.scan_inclusive(xd, op))
        assert_scan_matches(got, as3(x, 1, n, 1), op, True, what="seg %s %s n=%d" % (dt, op, n))
    got = to_host(gb.scan_exclusive(xd, "add"))
    assert_scan_matches(got, as3(x, 1, n, 1), "add", False, what="seg %s excl n=%d" % (dt, n))
    assert gb.device_error() == gb.OK


@pytest.mark.parametrize("dt", [np.float32, np.float64])
def test_segment_path_reproducible_and_in_place(dt):
    """The segment kernels combine in a fixed order: float sums repeat bit for bit."""
    x = workloads.normal(10_000_000, dt, 21)
    xd = to_dev(x)
    first = to_host(gb.scan_inclusive(xd))
    for _ in range(3):
        assert np.array_equal(to_host(gb.scan_inclusive(xd)), first)
    y = to_dev(x)
    gb.scan_inclusive(y, out=y)
    assert np.array_equal(to_host(y), first)
    assert gb.device_error() == gb.OK


def test_segment_fp64_integer_valued_exact():
    """Integer-valued doubles sum exactly in any order: the fp64 segment kernel must
    then agree with the oracle bit for bit, and with the row kernel (unaligned view)."""
    n = 3_000_017
    x = workloads.small_ints(n + 1, 4, -50, 51).astype(np.float64)
    got = to_host(gb.scan_inclusive(to_dev(x[1:])))
    assert np.array_equal(got, oracle.scan(x[1:]))
    rows = to_host(gb.scan_inclusive(to_dev(x)[1:]))
    assert np.array_equal(rows, got)
    got = to_host(gb.scan_exclusive(to_dev(x[1:]), init=np.float64(7)))
    assert np.array_equal(got, oracle.scan(x[1:], inclusive=False, init=np.float64(7)))


# ---- the L2-resident single-pass path (one long aligned row above 96 MiB) ------------

@pytest.mark.parametrize("dt,n", [("f32", 25_165_824 + 77), ("f32", 33_554_432 + 5), ("i32", 30_000_001),
                                  ("u32", 26_000_000), ("i64", 13_000_003), ("u64", 12_582_912 + 8)])
@pytest.mark.parametrize("op", ["add", "max", "min"])
def test_l2_resident_path(dt, n, op):
    if dt not in DTYPES:
        pytest.skip("no torch dtype")
    x = make(dt, n, n % 1000)
    xd = to_dev(x)
    got = to_host(gb.scan_inclusive(xd, op))
    assert_scan_matches(got, as3(x, 1, n, 1), op, True, what="%s %s incl n=%d" % (dt, op, n))
    init = x[0] if op != "add" else None
    got = to_host(gb.scan_exclusive(xd, op, init=init))
    assert_scan_matches(got, as3(x, 1, n, 1), op, False, init, what="%s %s excl n=%d" % (dt, op, n))
    assert gb.device_error() == gb.OK


def test_l2_resident_path_repeated_in_place():
    x = workloads.small_ints(30_000_000, 5, -3, 4)
    want = oracle.scan(x)
    for _ in range(5):
        y = to_dev(x)
        gb.scan_inclusive(y, out=y)
        assert np.array_equal(to_host(y), want)
    assert gb.device_error() == gb.OK


# ---- the row kernel on one row (unaligned views never take the other kernels) ---------

@pytest.mark.parametrize("dt", ["i32", "f32", "f64", "i64"])
@pytest.mark.parametrize("n", [4097, 1_000_003, 10_000_001])
def test_row_kernel_single_row(dt, n):
    base = make(dt, n + 1, 3 + n % 100)
    xd = to_dev(base)[1:]
    got = to_host(gb.scan_inclusive(xd))
    assert_scan_matches(got, as3(base[1:], 1, n, 1), "add", True, what="rows %s n=%d" % (dt, n))
    got = to_host(gb.scan_inclusive(xd, "min"))
    assert_scan_matches(got, as3(base[1:], 1, n, 1), "min", True, what="rows %s min n=%d" % (dt, n))
    assert gb.device_error() == gb.OK
