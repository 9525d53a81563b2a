"""Pins for the CPU oracle: it is checked against things other than itself.

Every pin below rests on the pages or on mathematics, never on the oracle:
worked examples printed on the pages (tests/golden/), closed forms, invariants,
wraparound arithmetic done with Python's unbounded integers, and brute-force
O(n^2) prefix sums computed from scratch on tiny inputs.  The same pin suite is
run against a set of deliberately broken scans (a dropped term, a wrong sign, an
off-by-one shift, a reversed or transposed walk, the wrong operator...) to show
that a plausible mistake anywhere fails at least one pin.
"""
import math

import numpy as np
import pytest

import oracle

GOLDEN_DEF = "merry_definitions_example.txt"
GOLDEN_KS = "merry_kogge_stone_example.txt"
GOLDEN_KARY = "merry_kary_brent_kung_example.txt"
GOLDEN_PACK = "merry_output_format_example.txt"


def oracle_scan3(x, op, inclusive, init=None):
    return oracle.scan3(x, op, inclusive, init)


def one_d(scan3, x, op="add", inclusive=True, init=None):
    return scan3(np.asarray(x).reshape(1, -1, 1), op, inclusive, init).reshape(-1)


# ---------------------------------------------------------------- the pins --

def pin_golden_definitions(scan3, golden):
    g = golden(GOLDEN_DEF)
    for dt in (np.int32, np.int64, np.float32, np.float64):
        x = np.array(g["input"], dtype=dt)
        assert list(one_d(scan3, x)) == g["inclusive"]
        assert list(one_d(scan3, x, inclusive=False)) == g["exclusive"]


def pin_golden_kogge_stone(scan3, golden):
    g = golden(GOLDEN_KS)
    x = np.array(g["input"], dtype=np.int32)
    assert list(one_d(scan3, x)) == g["inclusive"]


def pin_golden_kary(scan3, golden):
    g = golden(GOLDEN_KARY)
    x = np.array(g["input"], dtype=np.int32)
    inc = [int(v) for v in one_d(scan3, x)]
    exc = [int(v) for v in one_d(scan3, x, inclusive=False)]
    b = g["block_size"][0]
    assert inc == g["inclusive"]
    assert inc[-1] == g["total"][0]
    # Block sums and the exclusive block bases of the 4-ary down-sweep.
    ends = [inc[k * b + b - 1] for k in range(len(x) // b)]
    assert [ends[0]] + [ends[k] - ends[k - 1] for k in range(1, len(ends))] == g["block_sums"]
    assert [exc[k * b] for k in range(len(x) // b)] == g["block_bases"]


def pin_all_ones(scan3, golden=None):
    for dt, n in ((np.int32, 100_003), (np.int64, 4097), (np.float32, 70_000), (np.float64, 5000)):
        x = np.ones(n, dtype=dt)
        assert np.array_equal(one_d(scan3, x), np.arange(1, n + 1))
        assert np.array_equal(one_d(scan3, x, inclusive=False), np.arange(0, n))


def pin_last_is_reduction(scan3, golden=None):
    r = np.random.default_rng(101)
    xi = r.integers(-2**31, 2**31, 5000, dtype=np.int64).astype(np.int32)
    total = sum(int(v) for v in xi) % 2**32
    total = total - 2**32 if total >= 2**31 else total
    assert int(one_d(scan3, xi)[-1]) == total
    xf = r.standard_normal(20_000)
    bound = 2 * len(xf) * np.finfo(np.float64).eps * np.abs(xf).sum()
    assert abs(float(one_d(scan3, xf)[-1]) - math.fsum(xf)) <= bound
    xm = r.standard_normal(3000).astype(np.float32)
    assert float(one_d(scan3, xm, "max")[-1]) == float(xm.max())
    assert float(one_d(scan3, xm, "min")[-1]) == float(xm.min())


def pin_max_min_monotone(scan3, golden=None):
    up = np.arange(-500, 500, dtype=np.int32)
    down = up[::-1].copy()
    assert np.array_equal(one_d(scan3, up, "max"), up)
    assert np.array_equal(one_d(scan3, down, "max"), np.full(down.size, down[0]))
    assert np.array_equal(one_d(scan3, down, "min"), down)
    assert np.array_equal(one_d(scan3, up, "min"), np.full(up.size, up[0]))
    upf = np.linspace(-3, 3, 777).astype(np.float32)
    assert np.array_equal(one_d(scan3, upf, "max"), upf.astype(np.float64))


def pin_exclusive_relations(scan3, golden=None):
    r = np.random.default_rng(7)
    x = r.integers(-1000, 1000, 4000).astype(np.int32)
    s = one_d(scan3, x).astype(np.int64)
    e = one_d(scan3, x, inclusive=False).astype(np.int64)
    assert np.array_equal(e, s - x)           # e = s - x for (invertible) add
    assert e[0] == 0 and np.array_equal(e[1:], s[:-1])
    xf = r.standard_normal(3000).astype(np.float32)
    sm = one_d(scan3, xf, "max")
    em = one_d(scan3, xf, "max", inclusive=False, init=xf[0])
    assert em[0] == xf[0] and np.array_equal(em[1:], sm[:-1])   # e_i = s_{i-1}
    e5 = one_d(scan3, x, inclusive=False, init=5).astype(np.int64)
    assert np.array_equal(e5, e + 5)          # init folds in on the left


def pin_wraparound(scan3, golden=None):
    x = np.array([2**31 - 1, 1, 2**31 - 1, 2**31 - 1, -5, 7], dtype=np.int32)
    acc, want = 0, []
    for v in x:
        acc = (acc + int(v)) % 2**32
        want.append(acc - 2**32 if acc >= 2**31 else acc)
    assert [int(v) for v in one_d(scan3, x)] == want
    xu = np.array([2**32 - 1, 2, 2**32 - 3], dtype=np.uint32)
    acc, wantu = 0, []
    for v in xu:
        acc = (acc + int(v)) % 2**32
        wantu.append(acc)
    assert [int(v) for v in one_d(scan3, xu)] == wantu


def pin_wraparound_64(scan3, golden=None):
    """64-bit add keeps the low 64 bits of the exact sum (Python integers)."""
    x = np.array([2**63 - 1, 1, 2**63 - 1, -2**63, -5, 7, 2**62, 2**62], dtype=np.int64)
    acc, want = 0, []
    for v in x:
        acc = _wrap(acc + int(v), 64)
        want.append(acc)
    assert [int(v) for v in one_d(scan3, x)] == want
    r = np.random.default_rng(404)
    xu = r.integers(0, 2**64, 700, dtype=np.uint64)
    acc, wantu = 0, []
    for v in xu:
        acc = (acc + int(v)) % 2**64
        wantu.append(acc)
    assert [int(v) for v in one_d(scan3, xu)] == wantu
    e = one_d(scan3, xu, inclusive=False, init=xu[3])
    assert [int(v) for v in e] == [(int(xu[3]) + (w - int(v))) % 2**64 for w, v in zip(wantu, xu)]


def pin_unsigned_max_min(scan3, golden=None):
    """Unsigned max and min order values as unsigned integers: a value with the top
    bit set is larger than any without it.  Full-range values (about half with the
    top bit set) and a head whose signed and unsigned orders differ, inclusive and
    exclusive, against Python integers."""
    r = np.random.default_rng(303)
    for dt, bits in ((np.uint32, 32), (np.uint64, 64)):
        x = r.integers(0, 2**bits, 600, dtype=dt)
        x[:3] = np.array([2**bits - 1, 1, 2**(bits - 1)], dtype=dt)
        xs = [int(v) for v in x]
        for op, f in (("max", max), ("min", min)):
            acc, want = None, []
            for v in xs:
                acc = v if acc is None else f(acc, v)
                want.append(acc)
            assert [int(v) for v in one_d(scan3, x, op)] == want, (dt, op)
            acc, want = xs[5], []
            for v in xs:
                want.append(acc)
                acc = f(acc, v)
            assert [int(v) for v in one_d(scan3, x, op, False, init=x[5])] == want, (dt, op, "excl")


def _brute(x, op, inclusive, init):
    """Every prefix recomputed from scratch: O(n^2)."""
    n = len(x)
    out = []
    for i in range(n):
        terms = list(x[: i + 1]) if inclusive else list(x[:i])
        if not inclusive and init is not None:
            terms = [init] + terms
        if op == "add":
            out.append(math.fsum(terms) if isinstance(terms[0] if terms else 0.0, float) else sum(terms))
        elif op == "max":
            out.append(max(terms))
        else:
            out.append(min(terms))
    return out


def pin_bruteforce(scan3, golden=None):
    r = np.random.default_rng(2024)
    for n in (1, 2, 31, 33, 257):
        xi = r.integers(-50, 50, n).astype(np.int64)
        for op in ("add", "max", "min"):
            got = [int(v) for v in one_d(scan3, xi, op)]
            assert got == _brute([int(v) for v in xi], op, True, None)
            got = [int(v) for v in one_d(scan3, xi, op, False, init=3)]
            assert got == _brute([int(v) for v in xi], op, False, 3)
        xf = r.standard_normal(n)
        tol = 2 * n * np.finfo(np.float64).eps * np.cumsum(np.abs(xf))
        got = one_d(scan3, xf, "add")
        want = np.array(_brute([float(v) for v in xf], "add", True, None))
        assert np.all(np.abs(got - want) <= tol)
        for op in ("max", "min"):
            assert list(one_d(scan3, xf, op)) == _brute([float(v) for v in xf], op, True, None)


def pin_axes_and_lanes(scan3, golden=None):
    """A (B, R, C) scan is B*C independent 1-D scans along R."""
    r = np.random.default_rng(5)
    B, R, C = 3, 41, 5
    x = r.integers(-9, 9, (B, R, C)).astype(np.int32)
    got = scan3(x, "add", True)
    for b in range(B):
        for c in range(C):
            want = _brute([int(v) for v in x[b, :, c]], "add", True, None)
            assert [int(v) for v in got[b, :, c]] == want
    got = scan3(x, "add", False, [1, 2, 3, 4, 5])
    for c in range(C):
        want = _brute([int(v) for v in x[0, :, c]], "add", False, c + 1)
        assert [int(v) for v in got[0, :, c]] == want


def _wrap(v, bits, signed=True):
    v %= 2**bits
    return v - 2**bits if signed and v >= 2**(bits - 1) else v


def pin_mul_closed_forms(scan3, golden=None):
    """Multiply (cumprod): factorials, powers of two, exact sign/power-of-two
    products, wraparound to the low bits, and the neutral element 1."""
    x = np.arange(1, 21, dtype=np.int64)                 # 20! < 2^63
    assert [int(v) for v in one_d(scan3, x, "mul")] == [math.factorial(k) for k in range(1, 21)]
    xf = np.arange(1, 19, dtype=np.float64)              # 18! < 2^53: exact in fp64
    assert [float(v) for v in one_d(scan3, xf, "mul")] == [float(math.factorial(k)) for k in range(1, 19)]
    p = np.full(40, 2, dtype=np.int32)                   # 2^k keeps its low 32 bits
    assert [int(v) for v in one_d(scan3, p, "mul")] == [_wrap(2**k, 32) for k in range(1, 41)]
    e = one_d(scan3, np.array([3, 4, 5], dtype=np.int32), "mul", inclusive=False)
    assert [int(v) for v in e] == [1, 3, 12]             # no init: starts from 1
    e7 = one_d(scan3, np.array([3, 4, 5], dtype=np.int32), "mul", inclusive=False, init=7)
    assert [int(v) for v in e7] == [7, 21, 84]           # init folds in on the left
    r = np.random.default_rng(33)
    xo = (r.integers(-999, 1000, 300) | 1).astype(np.int32)   # odd: never 0 mod 2^32
    acc, want = 1, []
    for v in xo:
        acc *= int(v)
        want.append(_wrap(acc, 32))
    assert [int(v) for v in one_d(scan3, xo, "mul")] == want
    xs = r.choice(np.array([1.0, -1.0, 2.0, 0.5], dtype=np.float32), 2000, p=[0.4, 0.3, 0.15, 0.15])
    acc, wantf = 1, []
    for v in xs:                                         # products of +-2^k are exact
        acc = acc * float(v)
        wantf.append(acc)
    assert [float(v) for v in one_d(scan3, xs, "mul")] == wantf


def pin_mul_bruteforce(scan3, golden=None):
    r = np.random.default_rng(77)
    for n in (1, 2, 33, 200):
        xi = r.integers(-50, 50, n).astype(np.int64)
        got = [int(v) for v in one_d(scan3, xi, "mul")]
        assert got == [_wrap(math.prod(int(v) for v in xi[: i + 1]), 64) for i in range(n)]
        xf = np.exp(r.standard_normal(n) * 0.3)
        got = one_d(scan3, xf, "mul")
        want = np.array([math.prod(float(v) for v in xf[: i + 1]) for i in range(n)])
        eps = np.finfo(np.float64).eps
        assert np.all(np.abs(got - want) <= 2 * (np.arange(n) + 1) * eps * np.abs(want))


PINS = [pin_golden_definitions, pin_golden_kogge_stone, pin_golden_kary, pin_all_ones,
        pin_last_is_reduction, pin_max_min_monotone, pin_exclusive_relations,
        pin_wraparound, pin_wraparound_64, pin_unsigned_max_min, pin_bruteforce, pin_axes_and_lanes,
        pin_mul_closed_forms, pin_mul_bruteforce]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_scan_pins(pin, golden):
    pin(oracle_scan3, golden)


def test_exclusive_max_needs_init():
    with pytest.raises(oracle.NoIdentity):
        oracle.scan(np.arange(5, dtype=np.float32), "max", inclusive=False)
    with pytest.raises(oracle.NoIdentity):
        oracle.scan(np.arange(5, dtype=np.int32), "min", inclusive=False)


def test_oracle_wrapper_axes(golden):
    """scan_batched's axis mapping: axis 1 = rows, axis 0 = columns (row-major)."""
    r = np.random.default_rng(9)
    m = r.integers(-5, 5, (7, 11)).astype(np.int32)
    rows = oracle.scan_batched(m, axis=1)
    cols = oracle.scan_batched(m, axis=0)
    for i in range(7):
        assert np.array_equal(rows[i], oracle.scan(m[i]))
    for j in range(11):
        assert np.array_equal(cols[:, j], oracle.scan(np.ascontiguousarray(m[:, j])))


# ------------------------------------------ the pins catch planted mistakes --

def _numpy_scan3(mistake):
    """A scan3 built from numpy with one plausible mistake planted in it."""
    def scan3(x, op, inclusive, init=None):
        x = np.asarray(x)
        acc_t = np.float64 if x.dtype.kind == "f" else x.dtype
        if mistake == "fp32_accumulate" and x.dtype.kind == "f":
            acc_t = np.float32
        a = x.astype(acc_t)
        axis = 2 if mistake == "transposed_axis" else 1
        if mistake == "reversed":
            a = np.flip(a, axis=axis)
        use = op
        if mistake == "max_is_min":
            use = {"max": "min", "min": "max"}.get(op, op)
        if mistake == "mul_is_add":
            use = {"mul": "add"}.get(op, op)
        signed_view = None
        if mistake == "signed_compare" and x.dtype.kind == "u" and use in ("max", "min"):
            signed_view = np.dtype("i%d" % x.dtype.itemsize)   # compares as if signed
            a = a.view(signed_view)
            acc_t = signed_view
        if mistake == "drop_first_term":
            a = a.copy()
            idx = [slice(None)] * 3
            idx[axis] = 0
            if use == "add":
                a[tuple(idx)] = 0
            if use == "mul":
                a[tuple(idx)] = 1
        if use == "mul":
            s = np.cumprod(a, axis=axis, dtype=acc_t)
        elif use == "add":
            if mistake == "wrong_sign":
                s = np.cumsum(-a, axis=axis) + 2 * np.take(a, [0], axis=axis)
            else:
                s = np.cumsum(a, axis=axis, dtype=acc_t)
        elif use == "max":
            s = np.maximum.accumulate(a, axis=axis)
        else:
            s = np.minimum.accumulate(a, axis=axis)
        if mistake == "reversed":
            s = np.flip(s, axis=axis)
        if signed_view is not None:
            s = s.view(x.dtype)
            acc_t = x.dtype
        if mistake == "off_by_one":
            inclusive = not inclusive
        if inclusive:
            return s
        first = np.zeros_like(np.take(s, [0], axis=axis))
        if use == "mul" and mistake != "mul_identity_zero":
            first = first + 1
        if init is not None and mistake != "init_ignored":
            first = first * 0 + np.asarray(init, dtype=acc_t).reshape(1, 1, -1)
            if use == "mul":
                s = s * np.asarray(init, dtype=acc_t).reshape(1, 1, -1)
            elif use == "add":
                s = s + np.asarray(init, dtype=acc_t).reshape(1, 1, -1)
            elif use == "max":
                s = np.maximum(s, np.asarray(init, dtype=acc_t).reshape(1, 1, -1))
            else:
                s = np.minimum(s, np.asarray(init, dtype=acc_t).reshape(1, 1, -1))
        shifted = np.concatenate([first, np.delete(s, -1, axis=axis)], axis=axis)
        return shifted
    return scan3


MISTAKES = ["drop_first_term", "wrong_sign", "off_by_one", "reversed", "transposed_axis",
            "max_is_min", "init_ignored", "fp32_accumulate", "mul_is_add", "mul_identity_zero",
            "signed_compare"]


def test_reference_numpy_scan_passes(golden):
    """The numpy stand-in without a planted mistake passes every pin."""
    for pin in PINS:
        pin(_numpy_scan3("none"), golden)


@pytest.mark.parametrize("mistake", MISTAKES)
def test_pins_catch_planted_mistake(mistake, golden):
    failures = 0
    for pin in PINS:
        try:
            pin(_numpy_scan3(mistake), golden)
        except (AssertionError, ValueError, IndexError):
            failures += 1
    assert failures >= 1, "no pin caught the planted mistake %r" % mistake


# ------------------------------------------------------------- compaction --

def test_compact_invariants_and_bruteforce():
    r = np.random.default_rng(55)
    x = r.random(50_001, dtype=np.float32)
    for pred, p in (("lt", 0.01), ("lt", 0.5), ("lt", 0.99), ("ge", 0.5), ("eq", float(x[17])),
                    ("ne", float(x[3])), ("le", 0.25), ("gt", 0.75)):
        idx = oracle.compact(x, pred, p)
        t = np.float32(p)
        mask = {"lt": x < t, "le": x <= t, "gt": x > t, "ge": x >= t, "eq": x == t, "ne": x != t}[pred]
        assert idx.size == int(mask.sum())                     # count = sum of predicate bits
        assert np.all(np.diff(idx) > 0)                        # stable, strictly ascending
        assert np.array_equal(idx, np.nonzero(mask)[0])        # brute force
        assert np.all(mask[idx])


def test_compact_special_cases():
    x = np.linspace(0, 1, 1000, endpoint=False).astype(np.float32)
    assert oracle.compact(x, "lt", 0.0).size == 0              # selects none
    assert np.array_equal(oracle.compact(x, "lt", 2.0), np.arange(1000))   # selects all
    assert oracle.compact(np.zeros(0, np.float32), "lt", 1.0).size == 0
    nan = np.array([np.nan, 1.0, np.nan], dtype=np.float32)
    assert list(oracle.compact(nan, "ne", 1.0)) == [0, 2]      # NaN != t holds
    assert list(oracle.compact(nan, "lt", 5.0)) == [1]         # NaN < t does not
    xi = np.array([5, -3, 7, 0], dtype=np.int32)
    assert list(oracle.compact(xi, "gt", 0)) == [0, 2]


# ---------------------------------------------------------------- packing --

def test_pack_golden(golden):
    g = golden(GOLDEN_PACK)
    offs, recs, total = oracle.pack_by_counts(np.array(g["counts"], dtype=np.int32))
    assert list(offs) == g["offsets"]
    assert list(recs) == g["records"]
    assert total == g["total"][0]


def test_pack_invariants():
    r = np.random.default_rng(6)
    k = r.poisson(4.0, 20_000).astype(np.int32)
    offs, recs, total = oracle.pack_by_counts(k)
    assert total == int(k.astype(np.int64).sum())
    assert np.array_equal(offs, np.concatenate([[0], np.cumsum(k, dtype=np.int64)[:-1]]))
    assert np.array_equal(recs, np.repeat(np.arange(k.size, dtype=np.int32), k))
    # capacity truncates the records but not the total
    offs2, recs2, total2 = oracle.pack_by_counts(k, capacity=1000)
    assert total2 == total and np.array_equal(recs2, recs[:1000])
    # empty input and all-zero counts
    assert oracle.pack_by_counts(np.zeros(0, np.int32))[2] == 0
    assert oracle.pack_by_counts(np.zeros(10, np.int32))[2] == 0


# -------------------------------------------------------------- partition --

_PYPRED = {"lt": lambda v, t: v < t, "le": lambda v, t: v <= t, "gt": lambda v, t: v > t,
           "ge": lambda v, t: v >= t, "eq": lambda v, t: v == t, "ne": lambda v, t: not (v == t)}


def test_partition_against_the_definition():
    """Selected elements in input order, then the rest in input order (list comprehensions)."""
    r = np.random.default_rng(61)
    for dt in (np.int32, np.uint32, np.int64, np.uint64, np.float32, np.float64):
        x = r.integers(0, 100, 3001).astype(dt)
        for pred, f in _PYPRED.items():
            vals, idx, m = oracle.partition(x, pred, 37)
            sel = [i for i in range(x.size) if f(x[i], dt(37))]
            rest = [i for i in range(x.size) if not f(x[i], dt(37))]
            assert [int(i) for i in idx] == sel + rest and m == len(sel)
            assert np.array_equal(vals, x[idx])


def test_partition_bit_split_and_radix_sort():
    """The one-bit split equals numpy's stable argsort of that bit, and 32 splits from
    the lowest bit up (an LSD radix sort) sort unsigned keys like numpy.sort."""
    r = np.random.default_rng(62)
    x = r.integers(-2**31, 2**31, 5000).astype(np.int32)
    for b in (0, 7, 31):
        vals, idx, m = oracle.partition(x, "bit_clear", b)
        key = (x.view(np.uint32) >> np.uint32(b)) & np.uint32(1)
        assert np.array_equal(idx, np.argsort(key, kind="stable"))
        assert m == int((key == 0).sum()) and np.array_equal(vals, x[idx])
    xu = r.integers(0, 2**32, 3000, dtype=np.uint64).astype(np.uint32)
    y = xu.copy()
    for b in range(32):
        y, _, _ = oracle.partition(y, "bit_clear", b)
    assert np.array_equal(y, np.sort(xu))
    x64 = r.integers(-2**62, 2**62, 2000).astype(np.int64)
    _, idx, _ = oracle.partition(x64, "bit_clear", 40)
    assert np.array_equal(idx, np.argsort((x64.view(np.uint64) >> np.uint64(40)) & np.uint64(1), kind="stable"))


def test_partition_special_cases():
    x = np.array([3.0, np.nan, -1.0, np.nan, 2.0], dtype=np.float32)
    vals, idx, m = oracle.partition(x, "lt", 2.5)      # NaN fails <: it goes with the rest
    assert list(idx) == [2, 4, 0, 1, 3] and m == 2
    _, idx, m = oracle.partition(x, "ne", 3.0)          # ... and passes !=
    assert list(idx) == [1, 2, 3, 4, 0] and m == 4
    y = np.arange(10, dtype=np.int32)
    assert oracle.partition(y, "lt", 0)[2] == 0 and list(oracle.partition(y, "lt", 0)[1]) == list(range(10))
    assert oracle.partition(y, "ge", 0)[2] == 10
    assert oracle.partition(np.zeros(0, np.int32), "lt", 1)[2] == 0
    with pytest.raises(ValueError):
        oracle.partition(y, "bit_clear", 32)             # no bit 32 in int32
    with pytest.raises(ValueError):
        oracle.partition(x, "bit_clear", 1)              # floats have no bit split


# ------------------------------------------------------------ segmented scan --

def _numpy_segments(x, flags, op, inclusive, init):
    """Each segment scanned on its own with numpy's accumulate (a library routine)."""
    heads = np.flatnonzero(flags)
    heads = np.union1d([0], heads).astype(np.int64)
    out = []
    for a, b in zip(heads, list(heads[1:]) + [x.size]):
        seg = x[a:b]
        if x.dtype.kind == "f":
            seg = seg.astype(np.float64)
        acc = {"add": np.add, "max": np.maximum, "min": np.minimum, "mul": np.multiply}[op].accumulate(seg, dtype=seg.dtype)
        if inclusive:
            out.append(acc)
        else:
            first = np.asarray([init], dtype=acc.dtype)
            body = {"add": np.add, "max": np.maximum, "min": np.minimum, "mul": np.multiply}[op](
                np.asarray(init, dtype=acc.dtype), acc[:-1])
            out.append(np.concatenate([first, body]))
    return np.concatenate(out) if out else np.zeros(0, x.dtype)


def test_segmented_against_numpy_per_segment():
    r = np.random.default_rng(63)
    for dt in (np.int32, np.int64, np.uint32, np.float64):
        for p in (0.0, 0.01, 0.3, 1.0):
            x = r.integers(-50 if dt != np.uint32 else 0, 50, 2000).astype(dt)
            fl = (r.random(2000) < p).astype(np.uint8)
            for op in ("add", "max", "min", "mul"):
                got = oracle.scan_segmented(x, fl, op)
                assert np.array_equal(got, _numpy_segments(x, fl, op, True, None)), (dt, p, op)
                init = 7 if op in ("add", "mul") else 3
                got = oracle.scan_segmented(x, fl, op, False, init)
                assert np.array_equal(got, _numpy_segments(x, fl, op, False, init)), (dt, p, op, "excl")


def test_segmented_closed_forms_and_rows():
    r = np.random.default_rng(64)
    x = r.integers(-9, 9, 4096).astype(np.int32)
    assert np.array_equal(oracle.scan_segmented(x, np.ones(4096, np.uint8)), x)          # every element a head
    assert np.array_equal(oracle.scan_segmented(x, np.ones(4096, np.uint8), inclusive=False), np.zeros(4096))
    ones = np.ones(5000, np.float32)
    assert np.array_equal(oracle.scan_segmented(ones, np.zeros(5000, np.uint8)), np.arange(1, 5001))
    rows = x.reshape(64, 64)                                                             # equal segments = rows
    fl = np.zeros(4096, np.uint8)
    fl[::64] = 1
    assert np.array_equal(oracle.scan_segmented(x, fl).reshape(64, 64), np.cumsum(rows, axis=1, dtype=np.int32))
    with pytest.raises(oracle.NoIdentity):
        oracle.scan_segmented(x, fl, "max", inclusive=False)


# -------------------------------------------- composition of affine maps --
# Element i is the map y -> a_i*y + b_i; the operator applies the earlier map first:
# (a1, b1) (+) (a2, b2) = (a1*a2, a2*b1 + b2).  Pins in Python integers, wrapped to
# the type's width: the recurrence y_i = a_i*y_{i-1} + b_i, maps applied one by one
# to a start value, the closed form for equal maps, a worked pair whose two orders
# differ, and O(n^2) brute force.

def oracle_affine(x, inclusive=True, init=None):
    return oracle.scan_affine(x, inclusive, init)


def _pairs(x):
    return [(int(x[2 * i]), int(x[2 * i + 1])) for i in range(x.size // 2)]


def _out_pairs(y, bits):
    return [(int(a) % 2**bits, int(b) % 2**bits) for a, b in _pairs(np.asarray(y))]


def apin_worked_pair(scan_affine):
    """y -> 2y + 3 then y -> 5y + 1 is y -> 10y + 16; the other order is y -> 10y + 5."""
    x = np.array([2, 3, 5, 1], dtype=np.int32)
    assert _out_pairs(scan_affine(x), 32) == [(2, 3), (10, 16)]
    x = np.array([5, 1, 2, 3], dtype=np.int32)
    assert _out_pairs(scan_affine(x), 32) == [(5, 1), (10, 5)]
    assert _out_pairs(scan_affine(np.array([5, 1, 2, 3], dtype=np.int64), False), 64) == [(1, 0), (5, 1)]


def apin_recurrence(scan_affine):
    """s_i = (a_0 ... a_i, y_i) with y_i = a_i y_{i-1} + b_i and y_{-1} = 0."""
    r = np.random.default_rng(501)
    for dt, bits in ((np.int32, 32), (np.uint32, 32), (np.int64, 64), (np.uint64, 64)):
        x = r.integers(0, 2**bits, 2 * 700, dtype=np.uint64).astype(dt) if bits == 64 else \
            r.integers(0, 2**bits, 2 * 700, dtype=np.uint64).astype(np.uint32).astype(dt)
        prod, y, want = 1, 0, []
        for a, b in _pairs(x):
            prod = prod * a % 2**bits
            y = (a * y + b) % 2**bits
            want.append((prod, y))
        assert _out_pairs(scan_affine(x), bits) == want, dt


def apin_apply_to_start(scan_affine):
    """The scanned map s_i sends any start value y0 where the maps f_0 .. f_i,
    applied one after the other, send it."""
    r = np.random.default_rng(502)
    x = r.integers(-50, 50, 2 * 300).astype(np.int64)
    got = _out_pairs(scan_affine(x), 64)
    for y0 in (0, 1, -7, 123456789):
        y = y0
        for i, (a, b) in enumerate(_pairs(x)):
            y = (a * y + b) % 2**64
            ga, gb = got[i]
            assert (ga * y0 + gb) % 2**64 == y, (y0, i)


def apin_equal_maps(scan_affine):
    """All maps equal to (a, b): s_i = (a^(i+1), b (1 + a + ... + a^i))."""
    for a, b, dt, bits in ((3, 5, np.int32, 32), (-2, 7, np.int64, 64), (1, 9, np.uint32, 32)):
        n = 1000
        x = np.tile(np.array([a, b], dtype=np.int64), n).astype(dt)
        want = [(a**(i + 1) % 2**bits, b * sum(a**k for k in range(i + 1)) % 2**bits) for i in range(n)]
        assert _out_pairs(scan_affine(x), bits) == want, (a, b)


def apin_exclusive(scan_affine):
    """e_0 = init and e_i = init (+) s_{i-1}; no init: the identity map (1, 0)."""
    r = np.random.default_rng(503)
    x = r.integers(-1000, 1000, 2 * 500).astype(np.int32)
    s = _out_pairs(scan_affine(x), 32)
    e = _out_pairs(scan_affine(x, False), 32)
    assert e == [(1, 0)] + s[:-1]
    ia, ib = 7, -3
    e = _out_pairs(scan_affine(x, False, (ia, ib)), 32)
    want = [(ia % 2**32, ib % 2**32)] + [(ia * a % 2**32, (a * ib + b) % 2**32) for a, b in s[:-1]]
    assert e == want


def apin_bruteforce(scan_affine):
    """Each prefix composed from scratch, as a Python function applied to 0 and 1."""
    r = np.random.default_rng(504)
    for n in (1, 2, 31, 33, 150):
        x = r.integers(-9, 9, 2 * n).astype(np.int64)
        ps = _pairs(x)
        got = _out_pairs(scan_affine(x), 64)
        for i in range(n):
            def f(y, i=i):
                for a, b in ps[: i + 1]:
                    y = a * y + b
                return y % 2**64
            b0, b1 = f(0), f(1)
            assert got[i] == ((b1 - b0) % 2**64, b0), (n, i)


APINS = [apin_worked_pair, apin_recurrence, apin_apply_to_start, apin_equal_maps, apin_exclusive,
         apin_bruteforce]


@pytest.mark.parametrize("pin", APINS, ids=lambda p: p.__name__)
def test_oracle_affine_pins(pin):
    pin(oracle_affine)


def test_oracle_affine_rejects_floats_and_odd_sizes():
    with pytest.raises(ValueError):
        oracle.scan_affine(np.ones(4, np.float32))
    with pytest.raises(ValueError):
        oracle.scan_affine(np.ones(3, np.int32))
    assert oracle.scan_affine(np.zeros(0, np.int32)).size == 0


def _python_affine(mistake):
    """A Python stand-in for the affine scan with one plausible mistake planted."""
    def scan_affine(x, inclusive=True, init=None):
        x = np.asarray(x)
        bits = 8 * x.dtype.itemsize
        m = 2**bits

        def comb(l, r_):
            (a1, b1), (a2, b2) = l, r_
            if mistake == "swapped_order":
                return (a2 * a1 % m, (a1 * b2 + b1) % m)
            if mistake == "b_unscaled":
                return (a1 * a2 % m, (b1 + b2) % m)
            if mistake == "scaled_by_first":
                return (a1 * a2 % m, (a1 * b1 + b2) % m)
            return (a1 * a2 % m, (a2 * b1 + b2) % m)
        acc = (1, 0) if (inclusive or init is None) else (int(init[0]) % m, int(init[1]) % m)
        if mistake == "identity_zero" and not inclusive and init is None:
            acc = (0, 0)
        out = []
        for i, p in enumerate(_pairs(x)):
            p = (p[0] % m, p[1] % m)
            if inclusive:
                acc = p if i == 0 else comb(acc, p)
                out.append(acc)
            else:
                out.append(acc)
                acc = comb(acc, p)
        flat = [v for pair in out for v in pair]
        return np.array(flat, dtype=np.uint64 if bits == 64 else np.uint32).astype(x.dtype) if flat else \
            np.zeros(0, x.dtype)
    return scan_affine


AFFINE_MISTAKES = ["swapped_order", "b_unscaled", "scaled_by_first", "identity_zero"]


def test_affine_stand_in_passes():
    for pin in APINS:
        pin(_python_affine("none"))


@pytest.mark.parametrize("mistake", AFFINE_MISTAKES)
def test_affine_pins_catch_planted_mistake(mistake):
    failures = 0
    for pin in APINS:
        try:
            pin(_python_affine(mistake))
        except (AssertionError, ValueError, OverflowError):
            failures += 1
    assert failures >= 1, "no pin caught the planted mistake %r" % mistake
