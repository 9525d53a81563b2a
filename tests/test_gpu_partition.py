"""GPU parity: stable partition (and its one-bit split) against the CPU oracle.

The values, the input indices and the count are compared bit for bit (floats by their
bit patterns, so NaNs compare too).
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
BITS = {np.dtype(np.float32): np.uint32, np.dtype(np.float64): np.uint64}


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    gb.load()
    yield
    torch.cuda.synchronize()


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def make(dt, n, seed):
    if dt[0] == "f":
        return workloads.uniform01(n, NP[dt], seed)
    return workloads.small_ints(n, seed, 0, 1000, dtype=np.int64).astype(NP[dt])


def make_full(dt, n, seed):
    """Unsigned values over the whole range (about half with the top bit set)."""
    return workloads.full_range_uints(n, seed, NP[dt])


def check(x, pred, thr, res, what, with_idx=True):
    out, out_idx, cnt = res
    vals, idx, m = oracle.partition(x, pred, thr)
    n = x.size
    got_m = int(cnt.cpu().item())
    assert got_m == m, "%s: count %d, want %d" % (what, got_m, m)
    got = out.cpu().numpy()[:n]
    bits = BITS.get(got.dtype)
    same = np.array_equal(got.view(bits), vals.view(bits)) if bits else np.array_equal(got, vals)
    if not same:
        bad = np.flatnonzero(got.view(bits) != vals.view(bits)) if bits else np.flatnonzero(got != vals)
        raise AssertionError("%s: %d values differ, first at %d (m=%d): got %r want %r" % (
            what, bad.size, bad[0], m, got[bad[0]], vals[bad[0]]))
    if with_idx:
        gi = out_idx.cpu().numpy()[:n]
        assert np.array_equal(gi, idx), "%s: indices differ at %d" % (what, int(np.flatnonzero(gi != idx)[0]))
    assert gb.device_error() == gb.OK


SIZES = [1, 2, 31, 513, 16_389, 1_000_003, 3_000_017]


@pytest.mark.parametrize("dt", ["i32", "u32", "i64", "u64", "f32", "f64"])
@pytest.mark.parametrize("n", SIZES)
def test_partition_lt(dt, n):
    x = make(dt, n, n % 1000)
    thr = 0.5 if dt[0] == "f" else 500
    check(x, "lt", thr, gb.partition(dev(x), "lt", thr), "%s lt n=%d" % (dt, n))


@pytest.mark.parametrize("dt", ["i32", "f32", "i64", "f64"])
@pytest.mark.parametrize("pred,thr", [("le", 0), ("gt", 990), ("ge", 1), ("eq", 7), ("ne", 7), ("lt", -1),
                                      ("ge", -1)])
def test_partition_predicates_and_selectivity(dt, pred, thr):
    n = 777_777
    x = make(dt, n, 3)
    if dt[0] == "f":
        x = np.floor(x * 1000).astype(x.dtype)  # integral values so eq / ne select some
    check(x, pred, thr, gb.partition(dev(x), pred, thr), "%s %s %s" % (dt, pred, thr))


@pytest.mark.parametrize("dt", ["u32", "u64"])
@pytest.mark.parametrize("pred", ["lt", "ge", "gt"])
@pytest.mark.parametrize("n", [4097, 1_000_003])
def test_partition_unsigned_full_range(dt, pred, n):
    """Unsigned comparisons on values with the top bit set, against a threshold that
    has it too (a signed comparison would put them on the wrong side)."""
    if not hasattr(torch, "uint32"):
        pytest.skip("no torch unsigned dtypes")
    x = make_full(dt, n, 40 + n % 7)
    thr = NP[dt](3 * (int(np.iinfo(NP[dt]).max) // 4))
    check(x, pred, thr, gb.partition(dev(x), pred, thr), "%s %s full range n=%d" % (dt, pred, n))


@pytest.mark.parametrize("dt", ["i32", "u32", "i64", "u64"])
@pytest.mark.parametrize("bit", [0, 3, 9, 31])
def test_partition_bit_split(dt, bit):
    n = 1_234_567
    x = workloads.rng(bit).integers(-2**31, 2**31, n).astype(NP[dt])
    check(x, "bit_clear", bit, gb.partition(dev(x), "bit_clear", bit), "%s bit %d" % (dt, bit))


def test_radix_sort_by_bit_splits():
    """32 stable one-bit splits from the lowest bit up sort uint32 keys, with their
    original positions carried along through the indices."""
    n = 1_000_003
    keys = workloads.rng(77).integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32)
    cur = dev(keys.view(np.int32))
    perm = torch.arange(n, dtype=torch.int64, device="cuda")
    for b in range(32):
        out, idx, _ = gb.partition(cur, "bit_clear", b)
        cur = out[:n].clone()
        perm = perm[idx[:n].long()]
    got = cur.cpu().numpy().view(np.uint32)
    assert np.array_equal(got, np.sort(keys))
    assert np.array_equal(perm.cpu().numpy(), np.argsort(keys, kind="stable"))


@pytest.mark.parametrize("dt,off", [("f32", 1), ("f32", 2), ("f32", 3), ("i32", 1), ("f64", 1), ("i64", 1)])
@pytest.mark.parametrize("n", [5, 4099, 2_000_001])
def test_partition_unaligned_views(dt, off, n):
    base = make(dt, n + off, off * 7 + n % 13)
    x = base[off:]
    xd = dev(base)[off:]
    thr = 0.3 if dt[0] == "f" else 300
    check(x, "lt", thr, gb.partition(xd, "lt", thr), "%s +%d n=%d" % (dt, off, n))


def test_partition_nan_and_no_indices():
    x = workloads.normal(2_000_003, np.float32, 5)
    x[::97] = np.nan
    xd = dev(x)
    check(x, "lt", 0.0, gb.partition(xd, "lt", 0.0), "nan lt")
    check(x, "ne", 0.0, gb.partition(xd, "ne", 0.0), "nan ne")
    check(x, "gt", 0.25, gb.partition(xd, "gt", 0.25, with_idx=False), "no idx", with_idx=False)


def test_partition_above_l2():
    """26e6 fp32 (104 MB): the same launch; its second read comes from HBM."""
    x = workloads.uniform01(26_000_003, np.float32, 8)
    check(x, "lt", 0.5, gb.partition(dev(x), "lt", 0.5), "26e6")


def test_partition_empty_and_errors():
    x = dev(np.arange(10, dtype=np.int32))
    _, _, cnt = gb.partition(x[:0], "lt", 3)
    assert int(cnt.item()) == 0
    with pytest.raises(gb.GbError) as e:
        gb.partition(dev(np.arange(10, dtype=np.float32)), "bit_clear", 1)
    assert e.value.code == gb.ERR_UNSUPPORTED
    with pytest.raises(gb.GbError) as e:
        gb.partition(x, "bit_clear", 32)
    assert e.value.code == gb.ERR_INVALID


def test_partition_full_size_workload():
    w = workloads.BY_NAME["partition_p0.5"]
    x = w.make()
    check(x, "lt", w.extra["p"], gb.partition(dev(x), "lt", w.extra["p"]), w.name)
