"""GPU parity: a seeded random sweep over the API, against the CPU oracle.

Each case draws a dtype, an operator, inclusive or exclusive, a size, a lane count or
an axis, and an element offset (0 gives 16-byte aligned data, 1..3 an unaligned view),
so that the dispatch between the kernel families (segment, L2-resident, row, lane and
reduce-then-scan kernels; the segment and tile compaction kernels) is crossed at
random as well as at the boundaries the other test files pin.  Sizes are drawn around
those boundaries: chunk (512 elements), tile (4096) and run (3 tiles) sizes, the size
at which every warp of every CTA has a chunk (2,490,368), and log-uniform in between.
Packing by counts and the host-array scan are swept the same way.  The bars are the
usual ones (tests/parity.py): bit-exact for integers, max/min, indices, partitions
and records; the stated tolerance for float add; the product bound for float
multiply (whose factors here are +-2^k, so exact).
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
DTS = list(NP)
EDGES = [1, 2, 31, 32, 33, 511, 512, 513, 4095, 4096, 4097, 12_287, 12_288, 12_289, 65_535, 65_537,
         2_490_368, 2_490_369]
MAX_VALUES = 4_000_000  # elements x lanes per case


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    gb.load()
    yield
    torch.cuda.synchronize()


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def draw_n(r, cap=MAX_VALUES):
    u = r.random()
    if u < 0.3:
        n = int(r.choice(EDGES))
    elif u < 0.6:
        n = int(r.integers(1, 3000))
    else:
        n = int(np.exp(r.uniform(np.log(3000), np.log(3_000_000))))
    return max(1, min(n, cap))


def scan_values(dt, op, n, seed):
    if op == "mul":
        if dt[0] == "f":
            return workloads.signs_pow2(n, NP[dt], seed)
        return workloads.odd_ints(n, seed, np.int64).astype(NP[dt])
    if dt[0] == "f":
        return workloads.normal(n, NP[dt], seed)
    if dt[0] == "u":  # the whole range: max/min must compare as unsigned, add wraps
        return workloads.full_range_uints(n, seed, NP[dt])
    return workloads.small_ints(n, seed, -1000, 1000, dtype=np.int64).astype(NP[dt])


def draw_init(r, x, op, inclusive):
    """A scalar initial value for an exclusive scan (max/min need one)."""
    if inclusive:
        return None
    if op in ("max", "min"):
        return x[int(r.integers(0, x.size))] if x.size else 0
    if r.random() < 0.5:
        return None
    return 1 if op == "mul" else 3


@pytest.mark.parametrize("case", range(400))
def test_fuzz_scan(case):
    r = np.random.default_rng(7_000 + case)
    dt = str(r.choice(DTS))
    op = str(r.choice(["add", "max", "min", "mul"]))
    inclusive = bool(r.random() < 0.5)
    lanes = 1
    if r.random() < 0.25:
        lanes = int(r.choice([2, 3, 4, 8, 16, 24] + ([17] if dt == "f64" else [])))
    n = draw_n(r, MAX_VALUES // lanes)
    off = 0 if r.random() < 0.6 else int(r.integers(1, 4))
    x = scan_values(dt, op, n * lanes + off, 7_000 + case)
    xv = x[off:]
    xd = dev(x)[off:]
    init = draw_init(r, xv, op, inclusive)
    what = "case %d: %s %s %s n=%d lanes=%d off=%d init=%r" % (
        case, dt, op, "incl" if inclusive else "excl", n, lanes, off, init)
    if inclusive:
        got = gb.scan_inclusive(xd, op, lanes=lanes)
    else:
        got = gb.scan_exclusive(xd, op, init=init, lanes=lanes)
    assert_scan_matches(got.cpu().numpy(), as3(xv, 1, n, lanes), op, inclusive, init, what=what)
    assert gb.device_error() == gb.OK, what


# Past the segment kernels' 96 MiB: aligned rows take the L2-resident kernel (fp64:
# the row kernel's chunked variant), unaligned views the row kernel.
@pytest.mark.parametrize("case", range(12))
def test_fuzz_scan_large(case):
    r = np.random.default_rng(12_000 + case)
    dt = str(r.choice(DTS))
    op = str(r.choice(["add", "max", "min"]))
    inclusive = bool(r.random() < 0.5)
    size = NP[dt]().itemsize
    n = int(r.integers((96 << 20) // size + 1, (160 << 20) // size))
    off = 0 if r.random() < 0.6 else int(r.integers(1, 4))
    x = scan_values(dt, op, n + off, 12_000 + case)
    xv = x[off:]
    xd = dev(x)[off:]
    init = draw_init(r, xv, op, inclusive)
    what = "case %d: %s %s %s n=%d off=%d init=%r" % (case, dt, op, "incl" if inclusive else "excl", n, off, init)
    got = gb.scan_inclusive(xd, op) if inclusive else gb.scan_exclusive(xd, op, init=init)
    assert_scan_matches(got.cpu().numpy(), as3(xv, 1, n, 1), op, inclusive, init, what=what)
    assert gb.device_error() == gb.OK, what


@pytest.mark.parametrize("case", range(200))
def test_fuzz_batched(case):
    r = np.random.default_rng(8_000 + case)
    dt = str(r.choice(DTS))
    op = str(r.choice(["add", "max", "min", "mul"]))
    inclusive = bool(r.random() < 0.5)
    axis = int(r.integers(0, 2))
    lanes = 1 if r.random() < 0.8 else int(r.choice([2, 3]))
    rows = int(r.choice([1, 2, 3, 7, 64, 65, 300, 1000])) if r.random() < 0.5 else int(r.integers(1, 400))
    cols = draw_n(r, max(1, MAX_VALUES // (rows * lanes)))
    x = scan_values(dt, op, rows * cols * lanes, 8_000 + case)
    shape = (rows, cols) if lanes == 1 else (rows, cols, lanes)
    xd = dev(x).reshape(shape)
    init = draw_init(r, x, op, inclusive)
    what = "case %d: %s %s %s axis %d rows=%d cols=%d lanes=%d init=%r" % (
        case, dt, op, "incl" if inclusive else "excl", axis, rows, cols, lanes, init)
    got = gb.scan_batched(xd, axis=axis, op=op, inclusive=inclusive, init=init, lanes=lanes).cpu().numpy()
    x3 = as3(x, rows, cols, lanes) if axis == 1 else as3(x, 1, rows, cols * lanes)
    assert_scan_matches(got, x3, op, inclusive, init, what=what)
    assert gb.device_error() == gb.OK, what


PREDS = ["lt", "le", "gt", "ge", "eq", "ne"]


def select_values(dt, n, seed):
    if dt[0] == "f":
        return workloads.uniform01(n, NP[dt], seed)
    if dt[0] == "u" and seed % 2:  # the whole range: comparisons must be unsigned
        return workloads.full_range_uints(n, seed, NP[dt])
    return workloads.small_ints(n, seed, 0, 100, dtype=np.int64).astype(NP[dt])


def draw_threshold(r, dt, x, pred):
    if (pred in ("eq", "ne") or (dt[0] == "u" and x.size and int(x.max()) > 100)) and x.size:
        return x[int(r.integers(0, x.size))]
    return float(r.random()) if dt[0] == "f" else int(r.integers(0, 101))


@pytest.mark.parametrize("case", range(150))
def test_fuzz_compact(case):
    r = np.random.default_rng(9_000 + case)
    dt = str(r.choice(DTS))
    pred = str(r.choice(PREDS))
    n = draw_n(r)
    off = 0 if r.random() < 0.6 else int(r.integers(1, 4))
    x = select_values(dt, n + off, 9_000 + case)
    xv = x[off:]
    thr = draw_threshold(r, dt, xv, pred)
    what = "case %d: %s %s %r n=%d off=%d" % (case, dt, pred, thr, n, off)
    idx, cnt = gb.compact(dev(x)[off:], pred, thr)
    want = oracle.compact(xv, pred, thr)
    c = int(cnt.item())
    assert c == want.size, "%s: count %d, oracle %d" % (what, c, want.size)
    assert np.array_equal(idx[:c].cpu().numpy().astype(np.int64), want), "%s: indices differ" % what
    assert gb.device_error() == gb.OK, what


BITS = {np.dtype(np.float32): np.uint32, np.dtype(np.float64): np.uint64}


@pytest.mark.parametrize("case", range(150))
def test_fuzz_partition(case):
    r = np.random.default_rng(10_000 + case)
    dt = str(r.choice(DTS))
    bit_split = dt[0] != "f" and r.random() < 0.3
    pred = "bit_clear" if bit_split else str(r.choice(PREDS))
    n = draw_n(r)
    off = 0 if r.random() < 0.6 else int(r.integers(1, 4))
    x = select_values(dt, n + off, 10_000 + case)
    xv = x[off:]
    thr = int(r.integers(0, 7)) if bit_split else draw_threshold(r, dt, xv, pred)
    with_idx = bool(r.random() < 0.8)
    what = "case %d: %s %s %r n=%d off=%d idx=%s" % (case, dt, pred, thr, n, off, with_idx)
    out, out_idx, cnt = gb.partition(dev(x)[off:], pred, thr, with_idx=with_idx)
    vals, idx, m = oracle.partition(xv, pred, thr)
    assert int(cnt.cpu().item()) == m, "%s: count %d, want %d" % (what, int(cnt.cpu().item()), m)
    got = out.cpu().numpy()[:n]
    bits = BITS.get(got.dtype)
    same = np.array_equal(got.view(bits), vals.view(bits)) if bits else np.array_equal(got, vals)
    assert same, "%s: values differ" % what
    if with_idx:
        assert np.array_equal(out_idx.cpu().numpy()[:n], idx), "%s: indices differ" % what
    assert gb.device_error() == gb.OK, what


@pytest.mark.parametrize("case", range(150))
def test_fuzz_segmented(case):
    r = np.random.default_rng(11_000 + case)
    dt = str(r.choice(DTS))
    op = str(r.choice(["add", "max", "min", "mul"]))
    inclusive = bool(r.random() < 0.5)
    n = draw_n(r)
    off = 0 if r.random() < 0.6 else int(r.integers(1, 4))
    x = scan_values(dt, op, n + off, 11_000 + case)
    fl = workloads.head_flags(n + off, float(r.choice([0.0, 0.001, 0.05, 0.5])), 11_000 + case)
    xv, fv = x[off:], fl[off:]
    init = draw_init(r, xv, op, inclusive)
    what = "case %d: %s %s %s n=%d off=%d init=%r" % (case, dt, op, "incl" if inclusive else "excl", n, off, init)
    got = gb.scan_segmented(dev(x)[off:], dev(fl)[off:], op=op, inclusive=inclusive, init=init).cpu().numpy()
    want = oracle.scan_segmented(xv, fv, op, inclusive, init)
    if xv.dtype.kind != "f" or op != "add":
        ok = got.astype(want.dtype) == want
    else:
        mag = oracle.scan_segmented(np.abs(xv.astype(np.float64)), fv, "add")
        if not inclusive:  # the exclusive value covers the elements before i in its segment
            mag = np.where(np.r_[True, fv[1:] != 0], 0.0, np.r_[0.0, mag[:-1]])
            if init is not None:
                mag = mag + abs(float(init))
        ok = np.abs(got.astype(np.float64) - want) <= 1e-5 * mag + 1e-6
    if not ok.all():
        i = int(np.flatnonzero(~ok)[0])
        raise AssertionError("%s: %d mismatches, first at %d: got %r want %r" % (
            what, int((~ok).sum()), i, got[i], want[i]))
    assert gb.device_error() == gb.OK, what


@pytest.mark.parametrize("case", range(80))
def test_fuzz_pack(case):
    r = np.random.default_rng(13_000 + case)
    n = draw_n(r, 1_000_000)
    lam = float(r.choice([0.0, 0.05, 1.0, 4.0, 20.0]))
    k = workloads.poisson_counts(n, lam, 13_000 + case)
    total = int(k.astype(np.int64).sum())
    cap = total + int(r.choice([0, 1, 1000]))
    with_offsets = bool(r.random() < 0.8)
    what = "case %d: n=%d lambda=%g cap=%d offsets=%s" % (case, n, lam, cap, with_offsets)
    offs, recs, tot = gb.pack_by_counts(dev(k), cap, offsets=with_offsets)
    w_offs, w_recs, w_total = oracle.pack_by_counts(k, capacity=cap)
    assert int(tot.item()) == w_total, what
    if with_offsets:
        assert np.array_equal(offs.cpu().numpy()[:n].astype(np.int64), w_offs), what + ": offsets"
    assert np.array_equal(recs.cpu().numpy()[:total], w_recs[:total]), what + ": records"
    assert gb.device_error() == gb.OK, what


@pytest.mark.parametrize("case", range(40))
def test_fuzz_host_scan(case):
    r = np.random.default_rng(14_000 + case)
    dt = str(r.choice(["i32", "i64", "f32", "f64"]))
    op = str(r.choice(["add", "max", "min"]))
    n = draw_n(r)
    chunk = int(r.choice([0, 4096, 65_536, 1 << 20] + ([16] if n < 5000 else [])))
    pinned = bool(r.random() < 0.7)
    x = scan_values(dt, op, n, 14_000 + case)
    xh = torch.from_numpy(x)
    if pinned:
        xh = xh.pin_memory()
    what = "case %d: %s %s n=%d chunk=%d pinned=%s" % (case, dt, op, n, chunk, pinned)
    out = gb.scan_inclusive_host(xh, op, chunk_elems=chunk)
    torch.cuda.current_stream().synchronize()
    assert_scan_matches(out.numpy(), as3(x, 1, n, 1), op, True, what=what)
    assert gb.device_error() == gb.OK, what


@pytest.mark.parametrize("case", range(120))
def test_fuzz_affine(case):
    """Composition of affine maps (two lanes of an integer type): sizes around the
    segment kernel's chunks and past the point where every warp has one, views 0 to 3
    maps off alignment (32-bit maps are 8 bytes: odd offsets take the look-back tile
    kernel), inclusive and exclusive with and without an initial map; bit for bit."""
    r = np.random.default_rng(15_000 + case)
    dt = str(r.choice(["i32", "u32", "i64", "u64"]))
    npt = NP[dt]
    n = draw_n(r, 2_000_000)
    off = 0 if r.random() < 0.5 else int(r.integers(1, 4))
    inclusive = bool(r.random() < 0.5)
    bits = 8 * np.dtype(npt).itemsize
    init = None
    if not inclusive and r.random() < 0.6:  # a full-range initial map (a, b)
        init = workloads.full_range_uints(2, 16_000 + case, np.uint32 if bits == 32 else np.uint64).view(npt)
    x = workloads.full_range_uints(2 * (n + off), 15_000 + case, np.uint32 if bits == 32 else np.uint64)
    x = x.view(npt) if np.dtype(npt).kind == "i" else x
    xv = x[2 * off:]
    xd = dev(x)[2 * off:]
    what = "case %d: %s n=%d off=%d %s init=%r" % (case, dt, n, off, "incl" if inclusive else "excl", init)
    got = (gb.scan_inclusive(xd, "affine", lanes=2) if inclusive
           else gb.scan_exclusive(xd, "affine", init=init, lanes=2)).cpu().numpy()
    want = oracle.scan_affine(xv, inclusive, init)
    ok = got == want
    if not ok.all():
        i = int(np.flatnonzero(~ok)[0])
        raise AssertionError("%s: %d values differ, first at map %d: got %s want %s" % (
            what, int((~ok).sum()), i // 2, got[i // 2 * 2: i // 2 * 2 + 2], want[i // 2 * 2: i // 2 * 2 + 2]))
    assert gb.device_error() == gb.OK, what
