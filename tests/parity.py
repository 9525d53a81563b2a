"""Comparison helpers for the GPU parity tests (GPU result vs the CPU oracle).

Bars:
  - integers, max/min, compaction indices, packing: bit-exact (max/min on floats:
    exact value equality, since they never round);
  - float add: |gpu - oracle_fp64| <= 1e-5 * (prefix sum of |x|) + 1e-6, element
    by element and lane by lane, the prefix sum of |x| taken along the scanned axis
    over the terms the output combines (for an exclusive scan: the elements before
    it and the initial value);
  - float multiply: |gpu - oracle_fp64| <= gamma_k * |oracle_fp64| with k the number
    of factors at that position (plus init) and gamma_k = k u / (1 - k u), u the unit
    roundoff of the element type: the rounding bound of a product of k floats in any
    bracketing (each multiplication adds a relative error of at most u).
"""
import numpy as np

import oracle

REL, ABS = 1e-5, 1e-6


def abs_prefix(x3: np.ndarray) -> np.ndarray:
    """Prefix sums of |x| along axis 1 of a (B, R, C) array, in fp64."""
    return np.cumsum(np.abs(x3.astype(np.float64)), axis=1)


def assert_scan_matches(got: np.ndarray, x3: np.ndarray, op: str, inclusive: bool, init=None,
                        what: str = ""):
    """got and x3 are (B, R, C) arrays; the oracle scans x3 along axis 1."""
    want = oracle.scan3(x3, op, inclusive, init)
    got = got.reshape(x3.shape)
    if op == "mul" and x3.dtype.kind == "f":
        u = 2.0 ** -24 if x3.dtype == np.float32 else 2.0 ** -53
        k = np.arange(1, x3.shape[1] + 1, dtype=np.float64).reshape(1, -1, 1)
        if not inclusive:
            k = k - 1 + (0 if init is None else 1)
        ku = k * u
        gamma = np.where(ku < 0.5, ku / (1 - ku), np.inf)
        err = np.abs(got.astype(np.float64) - want)
        ok = err <= gamma * np.abs(want)
        if not ok.all():
            bad = np.argwhere(~ok)[:5]
            b0 = tuple(bad[0])
            raise AssertionError("%s: %d products out of tolerance, first at %s: got %r want %r" % (
                what, int((~ok).sum()), list(b0), float(got[b0]), float(want[b0])))
        return
    if x3.dtype.kind in "iu" or op != "add":
        if x3.dtype.kind == "f":
            ok = got.astype(np.float64) == want
        else:
            ok = got == want
        if not ok.all():
            bad = np.argwhere(~ok)[:5]
            raise AssertionError("%s: %d mismatches, first at %s: got %s want %s" % (
                what, int((~ok).sum()), bad[0].tolist(), got[tuple(bad[0])], want[tuple(bad[0])]))
        return
    mag = abs_prefix(x3)
    if not inclusive:
        # the exclusive value at i covers the elements before i, plus init
        shifted = np.zeros_like(mag)
        shifted[:, 1:, :] = mag[:, :-1, :]
        mag = shifted
        if init is not None:
            mag = mag + np.abs(np.asarray(init, dtype=np.float64)).reshape(1, 1, -1)
    bound = REL * mag + ABS
    err = np.abs(got.astype(np.float64) - want)
    ok = err <= bound
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        b0 = tuple(bad[0])
        raise AssertionError("%s: %d elements out of tolerance, first at %s: got %r want %r (bound %g)" % (
            what, int((~ok).sum()), list(b0), float(got[b0]), float(want[b0]), float(bound[b0])))


def as3(x: np.ndarray, B: int, R: int, C: int) -> np.ndarray:
    return np.ascontiguousarray(x).reshape(B, R, C)
