"""Seeded synthetic inputs for the five workload families.

This module draws random numbers and nothing else: it holds none of the
library's arithmetic, and both the CUDA path's tests and the CPU oracle take
their inputs from here.  Generator: numpy ``default_rng(seed)`` (PCG64); values
are drawn before indices; an f32 input is the f64 draw rounded to nearest.

Workloads (shapes and distributions of the pages' use cases; no public dataset
is involved):

* sum -- ``uniform[0, 12)`` values, seed 0 (inexact values that round, as the
  Day 68 page asks of a determinism test, section "Pitfalls").
* scatter -- N(0,1) values, int32 bins uniform over ``num_bins`` (or all in bin
  0), seed 2: the ``atomic_add(out, bins[tid], values[tid])`` kernel of the Warp
  "Deterministic Execution" guide, section "Pattern A: Accumulation Atomics".
* skewed scatter -- N(0,1) values, bins from a bounded Zipf(s) law over
  ``num_bins`` ranks by inverse CDF (rank r -> bin r-1, so hot bins are low
  indices), then about 5 % of the indices moved out of range (half negative,
  half >= num_bins), seed 3; out-of-range destinations are skipped as in
  "warp.tile_atomic_add_indexed".
* scan -- lognormal(0, 1) values, an area-CDF-like input (drjit-core pull
  request "Make CUDA floating-point prefix sums deterministic", "Root cause"),
  seed 4; segment lengths geometric with the given mean, the last one cut to
  fit, as int64 CSR offsets.
* row scatter -- N(0,1) source rows and destination rows, int32 row indices
  uniform over the destination rows, seed 5 ("warp.tile_atomic_add_indexed").
"""
from __future__ import annotations

import numpy as np

SUM_N = 1 << 20
SCATTER_N = 1 << 24
SCATTER_BINS = 1024
SKEW_N = 1 << 26
SKEW_BINS = 1 << 20
SKEW_S = 1.1
SKEW_OOR = 0.05
SCAN_SMALL_N = 164_738
SCAN_N = 1 << 28
SCAN_SEG_MEAN = 4096
ROWS_SRC = 1 << 20
ROWS_DST = 1 << 16
ROWS_LEN = 64


def _cast(x: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(x.astype(dtype, copy=False))


def sum_input(n: int = SUM_N, dtype=np.float32, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return _cast(rng.uniform(0.0, 12.0, n), dtype)


def scatter_input(n: int = SCATTER_N, num_bins: int = SCATTER_BINS, dtype=np.float32,
                  seed: int = 2, all_in_bin0: bool = False):
    """Returns (values, bins, out0) with out0 zero-initialised."""
    rng = np.random.default_rng(seed)
    values = _cast(rng.standard_normal(n), dtype)
    if all_in_bin0:
        bins = np.zeros(n, dtype=np.int32)
    else:
        bins = rng.integers(0, num_bins, n, dtype=np.int32)
    return values, bins, np.zeros(num_bins, dtype=dtype)


def zipf_bins(rng, n: int, num_bins: int, s: float) -> np.ndarray:
    ranks = np.arange(1, num_bins + 1, dtype=np.float64)
    p = ranks ** (-s)
    cdf = np.cumsum(p / p.sum())
    cdf[-1] = 1.0
    u = rng.random(n)
    b = np.searchsorted(cdf, u, side="right")
    return np.minimum(b, num_bins - 1).astype(np.int32)


def skewed_scatter_input(n: int = SKEW_N, num_bins: int = SKEW_BINS, dtype=np.float64,
                         seed: int = 3, s: float = SKEW_S, oor: float = SKEW_OOR):
    """Returns (values, bins, out0)."""
    rng = np.random.default_rng(seed)
    values = _cast(rng.standard_normal(n), dtype)
    bins = zipf_bins(rng, n, num_bins, s)
    move = rng.random(n) < oor
    negative = rng.random(n) < 0.5
    low = rng.integers(-(1 << 31), 0, n, dtype=np.int64)
    high = rng.integers(num_bins, 1 << 31, n, dtype=np.int64)
    bins = np.where(move, np.where(negative, low, high), bins).astype(np.int32)
    return values, bins, np.zeros(num_bins, dtype=dtype)


def scan_input(n: int = SCAN_SMALL_N, dtype=np.float32, seed: int = 4) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return _cast(rng.lognormal(0.0, 1.0, n), dtype)


def segment_offsets(n: int, mean: int = SCAN_SEG_MEAN, seed: int = 4) -> np.ndarray:
    """int64 CSR offsets [0, ..., n] with geometric lengths; last one truncated."""
    rng = np.random.default_rng(seed + 1000)
    lens = []
    total = 0
    while total < n:
        chunk = rng.geometric(1.0 / mean, max(16, (n - total) // mean + 16)).astype(np.int64)
        lens.append(chunk)
        total += int(chunk.sum())
    lens = np.concatenate(lens) if lens else np.zeros(0, dtype=np.int64)
    offsets = np.concatenate([[0], np.cumsum(lens)])
    cut = int(np.searchsorted(offsets, n, side="left"))
    offsets = offsets[: cut + 1].copy()
    offsets[-1] = n
    return offsets.astype(np.int64)


def fixed_segment_offsets(n: int, length: int) -> np.ndarray:
    """Segments of a constant length (the drjit block prefix sum case)."""
    return np.unique(np.concatenate([np.arange(0, n, length, dtype=np.int64), [n]]))


def rows_input(src_rows: int = ROWS_SRC, dst_rows: int = ROWS_DST, row_len: int = ROWS_LEN,
               dtype=np.float32, seed: int = 5):
    """Returns (src, idx, dst0)."""
    rng = np.random.default_rng(seed)
    src = _cast(rng.standard_normal((src_rows, row_len)), dtype)
    idx = rng.integers(0, dst_rows, src_rows, dtype=np.int32)
    dst = _cast(rng.standard_normal((dst_rows, row_len)), dtype)
    return src, idx, dst


VEC_WIDTH = 3


def vec_scatter_input(n: int = SCATTER_N, width: int = VEC_WIDTH, num_bins: int = SCATTER_BINS, dtype=np.float32,
                      seed: int = 6):
    """Composite scatter records (vec3 by default): returns (values n x width, bins, out0 num_bins x width),
    values N(0,1), bins uniform, out0 zero-initialised like the scalar scatter's."""
    rng = np.random.default_rng(seed)
    values = _cast(rng.standard_normal((n, width)), dtype)
    bins = rng.integers(0, num_bins, n, dtype=np.int32)
    out0 = np.zeros((num_bins, width), dtype=dtype)
    return values, bins, out0
