"""Seeded synthetic inputs for the scan and compaction workloads.

This module only draws random numbers (numpy PCG64 through ``default_rng``); it
holds none of the scan or compaction arithmetic.  The tests, the smoke check, the
benchmark and the oracle all take their inputs from here, so the GPU path and the
CPU oracle always see the same bytes.

The workload shapes, sizes and value distributions are those of the kernel-time
table in AcceleratedKernels.jl PR #208 ("Fit the scans' tiles in local memory for
large element types"): cumsum of 1e6/1e8 fp32, 1e7 fp64, 1e7 fp32 with an operator
that has no neutral element, scans along either axis of 4096x4096, 2x1e7, 1e6x8
and 1000x1e4 arrays, findall over 1e7 fp32, and 96-byte / 136-byte element types.
Arrays are row-major here (the PR's Julia arrays are column-major).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def normal(n: int, dtype, seed: int) -> np.ndarray:
    """n values ~ N(0, 1) in fp32 or fp64."""
    return rng(seed).standard_normal(n, dtype=np.dtype(dtype).type)


def uniform01(n: int, dtype, seed: int) -> np.ndarray:
    """n values uniform in [0, 1) in fp32 or fp64."""
    return rng(seed).random(n, dtype=np.dtype(dtype).type)


def uniform_pm1(n: int, dtype, seed: int) -> np.ndarray:
    """n values uniform in [-1, 1)."""
    return rng(seed).uniform(-1.0, 1.0, n).astype(dtype)


def small_ints(n: int, seed: int, lo: int = 0, hi: int = 100, dtype=np.int32) -> np.ndarray:
    """n integers uniform in [lo, hi)."""
    return rng(seed).integers(lo, hi, n, dtype=dtype)


def full_range_uints(n: int, seed: int, dtype=np.uint32) -> np.ndarray:
    """n unsigned integers uniform over the whole range of the type: about half of
    them have the top bit set, where signed and unsigned comparisons disagree."""
    bits = 8 * np.dtype(dtype).itemsize
    return rng(seed).integers(0, 2 ** bits, n, dtype=np.dtype(dtype).type)


def lognormal(n: int, dtype, seed: int, sigma: float) -> np.ndarray:
    """n factors exp(sigma * N(0, 1)): products of many stay within the type's range."""
    return np.exp(sigma * rng(seed).standard_normal(n)).astype(dtype)


def odd_ints(n: int, seed: int, dtype=np.int32) -> np.ndarray:
    """n odd integers in [-999, 999]: their products never reach 0 modulo 2^32."""
    return (rng(seed).integers(-999, 1000, n) | 1).astype(dtype)


def signs_pow2(n: int, dtype, seed: int, span: int = 30) -> np.ndarray:
    """n factors +-2^k whose running products are +-2^e with |e| <= span: every
    partial product is exact in fp32 and fp64, in any bracketing.  The exponent
    path is a lazy random walk folded into [-span, span] (steps of -1, 0, +1)."""
    r = rng(seed)
    walk = np.cumsum(r.choice(np.array([-1, 0, 1]), n, p=[0.1, 0.8, 0.1]))
    e = span - np.abs(np.mod(walk + span, 4 * span) - 2 * span)   # folded, unit steps
    step = np.diff(np.concatenate([[0], e]))
    sign = r.choice(np.array([1.0, -1.0]), n, p=[0.7, 0.3])
    return (sign * np.exp2(step)).astype(dtype)


def head_flags(n: int, p: float, seed: int) -> np.ndarray:
    """n uint8 head flags, each 1 with probability p (segments of mean length 1/p)."""
    return (rng(seed).random(n) < p).astype(np.uint8)


def poisson_counts(n: int, lam: float, seed: int) -> np.ndarray:
    """n int32 record counts k_i ~ Poisson(lam)."""
    return rng(seed).poisson(lam, n).astype(np.int32)


def values(kind: str, n: int, dtype, seed: int, extra: dict | None = None) -> np.ndarray:
    """Dispatch on a distribution name: normal, uniform01, uniform_pm1, ints, ones,
    lognormal (extra["sigma"]), odd_ints, signs_pow2."""
    if kind == "normal":
        return normal(n, dtype, seed)
    if kind == "uniform01":
        return uniform01(n, dtype, seed)
    if kind == "uniform_pm1":
        return uniform_pm1(n, dtype, seed)
    if kind == "ints":
        return small_ints(n, seed, dtype=dtype)
    if kind == "ones":
        return np.ones(n, dtype=dtype)
    if kind == "lognormal":
        return lognormal(n, dtype, seed, (extra or {}).get("sigma", 0.005))
    if kind == "odd_ints":
        return odd_ints(n, seed, dtype)
    if kind == "signs_pow2":
        return signs_pow2(n, dtype, seed)
    raise ValueError(kind)


@dataclass(frozen=True)
class Workload:
    """One benchmark configuration: what to scan or compact, and its seed."""
    name: str
    kind: str            # "scan", "batched", "compact", "pack", "partition", "segmented"
    dtype: str           # numpy dtype name of one lane
    shape: tuple         # (n,) or (rows, cols)
    dist: str
    seed: int
    op: str = "add"
    lanes: int = 1
    axis: int = -1       # batched: 0 (down columns) or 1 (along rows)
    inclusive: bool = True
    extra: dict = field(default_factory=dict)

    @property
    def elems(self) -> int:
        n = 1
        for s in self.shape:
            n *= s
        return n

    def make(self) -> np.ndarray:
        """Generate the input (lane values flattened in row-major order)."""
        if self.kind == "pack":
            return poisson_counts(self.elems, self.extra.get("lam", 4.0), self.seed)
        return values(self.dist, self.elems * self.lanes, self.dtype, self.seed, self.extra)


# The configurations, each with a fixed seed.  The headline is "fp32_1e8".
WORKLOADS = [
    Workload("i32_1e6", "scan", "int32", (1_000_000,), "ints", 1),
    Workload("i32_1e6_excl", "scan", "int32", (1_000_000,), "ints", 1, inclusive=False),
    Workload("fp32_1e8", "scan", "float32", (100_000_000,), "normal", 2),
    Workload("fp32_1e8_excl", "scan", "float32", (100_000_000,), "normal", 2, inclusive=False),
    Workload("fp64_1e7", "scan", "float64", (10_000_000,), "uniform_pm1", 3),
    Workload("fp32_1e7_max", "scan", "float32", (10_000_000,), "normal", 4, op="max"),
    Workload("compact_p0.01", "compact", "float32", (10_000_000,), "uniform01", 5, extra={"p": 0.01}),
    Workload("compact_p0.5", "compact", "float32", (10_000_000,), "uniform01", 5, extra={"p": 0.5}),
    Workload("compact_p0.99", "compact", "float32", (10_000_000,), "uniform01", 5, extra={"p": 0.99}),
    Workload("pack_poisson4_1e6", "pack", "int32", (1_000_000,), "poisson", 6, extra={"lam": 4.0}),
    Workload("fp32_4096x4096_axis0", "batched", "float32", (4096, 4096), "normal", 7, axis=0),
    Workload("fp32_4096x4096_axis1", "batched", "float32", (4096, 4096), "normal", 8, axis=1),
    Workload("fp32_2x1e7_axis1", "batched", "float32", (2, 10_000_000), "normal", 9, axis=1),
    Workload("fp32_1e6x8_axis0", "batched", "float32", (1_000_000, 8), "normal", 10, axis=0),
    Workload("fp64_1000x1e4_axis0", "batched", "float64", (1000, 10_000), "normal", 11, axis=0),
    Workload("struct96_1e6", "scan", "float32", (1_000_000,), "normal", 12, lanes=24),
    Workload("struct96_3x1e5_axis1", "batched", "float32", (3, 100_000), "normal", 13, lanes=24, axis=1),
    Workload("dual16_1e6", "scan", "float64", (1_000_000,), "uniform_pm1", 14, lanes=17),
    Workload("dual16_3x1e5_axis1", "batched", "float64", (3, 100_000), "uniform_pm1", 15, lanes=17, axis=1),
    # Beyond the kernel-time table: cumprod (the accumulate API's other reduction),
    # the 32-byte struct the PR also measures, and its largest element (2080 bytes)
    # with and without a neutral element.
    Workload("fp32_1e7_cumprod", "scan", "float32", (10_000_000,), "lognormal", 16, op="mul",
             extra={"sigma": 0.005}),
    Workload("i32_1e6_cumprod", "scan", "int32", (1_000_000,), "odd_ints", 17, op="mul"),
    Workload("struct32_1e6", "scan", "float32", (1_000_000,), "normal", 18, lanes=8),
    Workload("elem2080_2e4", "scan", "float32", (20_000,), "normal", 19, lanes=520),
    Workload("elem2080_2e4_max", "scan", "float32", (20_000,), "normal", 20, lanes=520, op="max"),
    # Segmented scan by head flags: segments of mean length 1000.
    Workload("fp32_1e7_segmented", "segmented", "float32", (10_000_000,), "normal", 22,
             extra={"p_head": 0.001, "flag_seed": 23}),
    # Stable partition (x < 0.5 first) of the compaction input's shape, values and indices.
    Workload("partition_p0.5", "partition", "float32", (10_000_000,), "uniform01", 21, extra={"p": 0.5}),
    # An operator that is not commutative: 1e7 affine maps (a, b) of int32 under
    # composition (the first-order recurrence y_i = a_i y_{i-1} + b_i), 80 MB each way.
    Workload("i32_1e7_affine", "scan", "int32", (10_000_000,), "ints", 24, op="affine", lanes=2),
]

BY_NAME = {w.name: w for w in WORKLOADS}
HEADLINE = "fp32_1e8"
