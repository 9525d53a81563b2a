"""GPU parity: stream compaction and packing by counts against the CPU oracle
(bit-exact: indices, order, counts, offsets, records)."""
import numpy as np
import pytest
import torch

import oracle
import stream_compaction_decoupled_gb300 as gb
from stream_compaction_decoupled_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    gb.load()
    yield
    torch.cuda.synchronize()


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def check_compact(x, pred, thr, what=""):
    idx, cnt = gb.compact(dev(x), pred, thr)
    want = oracle.compact(x, pred, thr)
    c = int(cnt.item())
    assert c == want.size, "%s: count %d, oracle %d" % (what, c, want.size)
    got = idx[:c].cpu().numpy().astype(np.int64)
    assert np.array_equal(got, want), "%s: indices differ" % what


@pytest.mark.parametrize("dt", [np.float32, np.float64, np.int32, np.int64])
@pytest.mark.parametrize("n", [1, 2, 33, 2047, 2048, 2049, 4095, 4096, 4097, 3 * 4096 + 77, 100_003])
@pytest.mark.parametrize("pred", ["lt", "le", "gt", "ge", "eq", "ne"])
def test_compact_small(dt, n, pred):
    if np.dtype(dt).kind == "f":
        x = workloads.uniform01(n, dt, n + 1)
        x[::7] = x[0]  # repeated values for eq / ne
        thr = x[0] if pred in ("eq", "ne") else 0.5
    else:
        x = workloads.small_ints(n, n + 1, -10, 10, dtype=dt)
        thr = 0
    check_compact(x, pred, thr, "%s n=%d %s" % (np.dtype(dt).name, n, pred))


@pytest.mark.parametrize("dt", [np.uint32, np.uint64])
@pytest.mark.parametrize("n", [4097, 1_000_003])
@pytest.mark.parametrize("pred", ["lt", "gt", "le"])
def test_compact_unsigned_full_range(dt, n, pred):
    """Unsigned comparisons on values with the top bit set, against a threshold that
    has it too: a signed comparison would select the complement of the right set."""
    if not hasattr(torch, "uint32"):
        pytest.skip("no torch unsigned dtypes")
    x = workloads.full_range_uints(n, n + 3, dt)
    thr = dt(3 * (int(np.iinfo(dt).max) // 4))
    check_compact(x, pred, thr, "%s n=%d %s full range" % (np.dtype(dt).name, n, pred))


def test_compact_none_all_and_empty():
    x = workloads.uniform01(3 * 4096 + 5, np.float32, 3)
    check_compact(x, "lt", 0.0, "none")
    check_compact(x, "lt", 2.0, "all")
    idx, cnt = gb.compact(torch.empty(0, dtype=torch.float32, device="cuda"), "lt", 1.0)
    assert int(cnt.item()) == 0


@pytest.mark.parametrize("dt", [np.float32, np.float64, np.int32])
@pytest.mark.parametrize("n", [2, 4097, 5 * 4096 + 3, 1_000_003])
@pytest.mark.parametrize("pred", ["lt", "ne"])
def test_compact_unaligned(dt, n, pred):
    """An input that is not 16-byte aligned takes the tile kernel (decoupled look-back)."""
    if np.dtype(dt).kind == "f":
        x = workloads.uniform01(n + 1, dt, n + 8)
        thr = 0.3
    else:
        x = workloads.small_ints(n + 1, n + 8, -10, 10, dtype=dt)
        thr = 0
    xd = dev(x)[1:]
    idx, cnt = gb.compact(xd, pred, thr)
    want = oracle.compact(x[1:], pred, thr)
    c = int(cnt.item())
    assert c == want.size and np.array_equal(idx[:c].cpu().numpy(), want)


@pytest.mark.parametrize("n", [511, 512, 513, 16_384 + 5, 2_490_368, 2_490_368 + 1, 25_165_824])
def test_compact_segment_sizes(n):
    """Chunk, CTA and warp-saturation boundaries of the segment kernel, up to 96 MiB."""
    x = workloads.uniform01(n, np.float32, n % 977)
    check_compact(x, "lt", 0.5, "seg n=%d" % n)
    check_compact(x, "ge", 0.999, "seg sparse n=%d" % n)
    assert gb.device_error() == gb.OK


def test_compact_above_segment_limit():
    """Above 96 MiB the tile kernel runs even for aligned inputs."""
    x = workloads.uniform01(26_000_003, np.float32, 11)
    check_compact(x, "lt", 0.25, "tile kernel n=26e6")
    assert gb.device_error() == gb.OK


def test_compact_nan():
    x = workloads.uniform01(10_000, np.float32, 4)
    x[::13] = np.nan
    for pred in ("lt", "ne", "ge"):
        check_compact(x, pred, 0.5, "nan " + pred)


@pytest.mark.parametrize("p", [0.01, 0.5, 0.99])
def test_compact_full_size(p):
    w = workloads.BY_NAME["compact_p%s" % p]
    x = w.make()
    check_compact(x, "lt", p, w.name)
    assert gb.device_error() == gb.OK


# ---- packing -----------------------------------------------------------------------

def check_pack(k, what="", capacity=None):
    total = int(k.astype(np.int64).sum())
    cap = total if capacity is None else capacity
    offs, recs, tot = gb.pack_by_counts(dev(k), cap)
    w_offs, w_recs, w_total = oracle.pack_by_counts(k, capacity=cap)
    assert int(tot.item()) == w_total, what
    assert np.array_equal(offs.cpu().numpy()[: k.size].astype(np.int64), w_offs), what + " offsets"
    assert np.array_equal(recs.cpu().numpy()[:cap], w_recs[:cap]), what + " records"


def test_pack_golden(golden):
    g = golden("merry_output_format_example.txt")
    k = np.array(g["counts"], dtype=np.int32)
    offs, recs, tot = gb.pack_by_counts(dev(k), 8)
    assert list(offs.cpu().numpy()) == g["offsets"]
    assert list(recs.cpu().numpy()) == g["records"]
    assert int(tot.item()) == g["total"][0]


@pytest.mark.parametrize("n", [1, 5, 4095, 4096, 4097, 3 * 4096 + 77, 200_001])
def test_pack_small(n):
    k = workloads.poisson_counts(n, 4.0, n)
    check_pack(k, "poisson n=%d" % n)
    z = np.zeros(n, dtype=np.int32)
    z[::97] = 300  # long runs, most objects empty
    check_pack(z, "sparse n=%d" % n)


def test_pack_full_size():
    w = workloads.BY_NAME["pack_poisson4_1e6"]
    check_pack(w.make(), w.name)
    assert gb.device_error() == gb.OK


def test_pack_capacity_and_negative_counts():
    k = workloads.poisson_counts(10_000, 4.0, 3)
    total = int(k.sum())
    offs, recs, tot = gb.pack_by_counts(dev(k), total // 2)
    assert int(tot.item()) == total
    _, w_recs, _ = oracle.pack_by_counts(k, capacity=total // 2)
    assert np.array_equal(recs.cpu().numpy(), w_recs)
    assert gb.device_error() == gb.ERR_RANGE          # over capacity is reported
    assert gb.device_error() == gb.OK                 # and cleared once read
    kn = k.copy()
    kn[17] = -3
    ref = kn.copy()
    ref[17] = 0                                       # a negative count counts as zero
    offs, recs, tot = gb.pack_by_counts(dev(kn), total)
    assert gb.device_error() == gb.ERR_INVALID
    w_offs, w_recs, w_total = oracle.pack_by_counts(ref, capacity=total)
    assert int(tot.item()) == w_total
    assert np.array_equal(offs.cpu().numpy().astype(np.int64), w_offs)
    assert np.array_equal(recs.cpu().numpy()[:w_total], w_recs[:w_total])


@pytest.mark.parametrize("n", [511, 512, 513, 16_385, 2_490_368 + 1, 3_000_017])
def test_pack_segment_sizes(n):
    """Chunk (512 counts), CTA and warp-saturation boundaries of the segment kernel."""
    check_pack(workloads.poisson_counts(n, 4.0, n % 991), "seg poisson n=%d" % n)
    z = np.zeros(n, dtype=np.int32)
    z[n // 3] = 1000   # one object owns many slots and blocks of slots
    z[-1] = 3
    check_pack(z, "seg sparse n=%d" % n)
    assert gb.device_error() == gb.OK


@pytest.mark.parametrize("n", [2, 4097, 100_003])
def test_pack_unaligned_counts(n):
    """Counts that are not 16-byte aligned take the tile kernel."""
    k = workloads.poisson_counts(n + 1, 3.0, 5)
    total = int(k[1:].astype(np.int64).sum())
    offs, recs, tot = gb.pack_by_counts(dev(k)[1:], total)
    w_offs, w_recs, w_total = oracle.pack_by_counts(k[1:], capacity=total)
    assert int(tot.item()) == w_total
    assert np.array_equal(offs.cpu().numpy().astype(np.int64), w_offs)
    assert np.array_equal(recs.cpu().numpy()[:total], w_recs[:total])


@pytest.mark.parametrize("aligned", [True, False])
def test_pack_saturation(aligned):
    """Offsets saturate at 2^31: exact below it, 2^31 - 1 from there on; the total is
    reported as 2^31 - 1 with GB_ERR_RANGE, and records stop at the capacity."""
    n = 100_000
    k = np.zeros(n + 1, dtype=np.int32)
    k[50_001] = 2**30
    k[70_001] = 2**30
    k[70_002] = 7
    kd = dev(k)[1:] if not aligned else dev(k[1:])
    offs, recs, tot = gb.pack_by_counts(kd, 1000)
    w_offs, w_recs, w_total = oracle.pack_by_counts(k[1:], capacity=1000)
    assert w_total == 2**31 + 7
    assert int(tot.item()) == 2**31 - 1
    assert np.array_equal(offs.cpu().numpy().astype(np.int64), np.minimum(w_offs, 2**31 - 1))
    assert np.array_equal(recs.cpu().numpy()[:1000], w_recs[:1000])
    assert gb.device_error() == gb.ERR_RANGE


@pytest.mark.parametrize("shift", [0, 1, 3, 4, 8])
@pytest.mark.parametrize("cap_frac", [1.0, 0.37])
def test_pack_record_alignment(shift, cap_frac):
    """Records written into a view that starts `shift` words into its buffer (32-byte
    vector stores only where the view allows them), at full capacity and cut short:
    the records match the oracle and no word outside [0, capacity) of the view is
    touched."""
    n = 200_003
    rng = np.random.default_rng(shift * 7 + int(cap_frac * 10))
    k = rng.poisson(4.0, n).astype(np.int32)
    k[rng.integers(0, n, 40)] = rng.integers(250, 2000, 40).astype(np.int32)  # runs over whole blocks
    k[rng.random(n) < 0.3] = 0
    total = int(k.astype(np.int64).sum())
    cap = int(total * cap_frac)
    guard = -7
    buf = torch.full((cap + shift + 64,), guard, dtype=torch.int32, device="cuda")
    recs_view = buf[shift: shift + cap]
    offs, recs, tot = gb.pack_by_counts(dev(k), cap, out_records=recs_view)
    w_offs, w_recs, w_total = oracle.pack_by_counts(k, capacity=cap)
    assert int(tot.item()) == w_total
    assert np.array_equal(offs.cpu().numpy().astype(np.int64), w_offs)
    b = buf.cpu().numpy()
    assert np.array_equal(b[shift: shift + cap], w_recs[:cap])
    assert (b[:shift] == guard).all() and (b[shift + cap:] == guard).all()
    assert gb.device_error() == (gb.OK if cap >= total else gb.ERR_RANGE)
    assert gb.device_error() == gb.OK
