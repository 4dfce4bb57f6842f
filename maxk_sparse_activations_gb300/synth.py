"""Seeded synthetic inputs shaped like the pages' workloads.

This module generates numbers only: it holds none of the selection arithmetic,
and both the CUDA path's tests and the oracle draw their inputs from it.

The pages measure on hidden-feature matrices of GNN layers (Reddit, Flickr,
Ogbn-products, Yelp at hidden size 256, k = 32) and study early stopping on
normally distributed synthetic vectors ("RTop-K ..." summary, "Limitations";
"MaxK-GNN ...", "One layer, one epoch, on Reddit"). Those datasets are not
available, so i.i.d. N(0, 1) rows of the same shape stand in for them, plus
the adversarial value sets of the long-row cases.

All generators return C-contiguous numpy arrays: float32 for fp32 inputs and
uint16 bit patterns for bf16 inputs.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "normal_f32", "uniform_pm1_f32", "int_ties_f32", "all_equal_rows_f32",
    "outliers_f32", "subnormals_f32", "wide_range_f32", "dense_bucket_f32", "negative_f32",
    "signed_zeros_f32", "f32_to_bf16_bits", "normal_bf16",
    "make", "VALUE_SETS", "power_law_graph", "transpose_graph",
]


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def normal_f32(N: int, M: int, seed: int = 0) -> np.ndarray:
    """i.i.d. standard normal, generated directly in float32."""
    return _rng(seed).standard_normal((N, M), dtype=np.float32)


def uniform_pm1_f32(N: int, M: int, seed: int = 0) -> np.ndarray:
    """U(-1, 1): 24-bit uniform integers scaled by 2^-23 and shifted (exact)."""
    u = _rng(seed).integers(0, 1 << 24, size=(N, M), dtype=np.int64)
    return (u.astype(np.float32) * np.float32(2.0 ** -23)) - np.float32(1.0)


def int_ties_f32(N: int, M: int, seed: int = 0) -> np.ndarray:
    """Heavy ties: integers 0..15 stored as float32."""
    return _rng(seed).integers(0, 16, size=(N, M), dtype=np.int32).astype(np.float32)


def all_equal_rows_f32(N: int, M: int, seed: int = 0) -> np.ndarray:
    """Row r is the constant c_r, c_r ~ N(0, 1)."""
    c = _rng(seed).standard_normal((N, 1), dtype=np.float32)
    return np.ascontiguousarray(np.broadcast_to(c, (N, M)))


def outliers_f32(N: int, M: int, seed: int = 0, p: float = 0.01, mag: float = 1e30) -> np.ndarray:
    """N(0, 1) with each entry replaced by +-mag (fair sign) with probability p."""
    g = _rng(seed)
    x = g.standard_normal((N, M), dtype=np.float32)
    hit = g.random((N, M)) < p
    sign = np.where(g.random((N, M)) < 0.5, np.float32(-mag), np.float32(mag))
    x[hit] = sign[hit]
    return x


def subnormals_f32(N: int, M: int, seed: int = 0) -> np.ndarray:
    """Mixed-sign subnormals: exponent field 0, mantissa uniform in [1, 2^23 - 1]."""
    g = _rng(seed)
    mant = g.integers(1, 1 << 23, size=(N, M), dtype=np.uint32)
    sign = (g.integers(0, 2, size=(N, M), dtype=np.uint32) << np.uint32(31))
    return (mant | sign).view(np.float32)


def wide_range_f32(N: int, M: int, seed: int = 0) -> np.ndarray:
    """Random sign times 10^U(-40, 37.5): magnitudes from binary32 subnormals to
    3e37, across the range of every 16-bit format."""
    g = _rng(seed)
    mag = np.power(10.0, g.uniform(-40.0, 37.5, size=(N, M)))
    sign = np.where(g.random((N, M)) < 0.5, -1.0, 1.0)
    return (sign * mag).astype(np.float32)


def dense_bucket_f32(N: int, M: int, seed: int = 0) -> np.ndarray:
    """Every row a shuffle of 1 + j * 2^-23 for j = 0..M-1 (M <= 2^23): distinct
    binary32 values, all within a few binary16 or bf16 spacings of 1."""
    g = _rng(seed)
    j = np.argsort(g.random((N, M)), axis=1).astype(np.float64)
    return (1.0 + j * 2.0 ** -23).astype(np.float32)


def negative_f32(N: int, M: int, seed: int = 0) -> np.ndarray:
    """-|N(0, 1)|: every value negative."""
    return -np.abs(_rng(seed).standard_normal((N, M), dtype=np.float32))


def signed_zeros_f32(N: int, M: int, seed: int = 0) -> np.ndarray:
    """Mostly -0.0 and +0.0 (fair sign), about one entry in eight N(0, 1)."""
    g = _rng(seed)
    x = np.where(g.random((N, M)) < 0.5, np.float32(-0.0), np.float32(0.0)).astype(np.float32)
    hit = g.random((N, M)) < 0.125
    x[hit] = g.standard_normal((N, M), dtype=np.float32)[hit]
    return x


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even) and return the 16-bit patterns.

    Inputs are finite (the generators never produce NaN or infinity).
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def normal_bf16(N: int, M: int, seed: int = 0) -> np.ndarray:
    """i.i.d. N(0, 1) rounded to bf16, as uint16 bit patterns."""
    return f32_to_bf16_bits(normal_f32(N, M, seed))


VALUE_SETS = {
    "normal": normal_f32,
    "uniform": uniform_pm1_f32,
    "int_ties": int_ties_f32,
    "all_equal": all_equal_rows_f32,
    "outliers": outliers_f32,
    "subnormal": subnormals_f32,
    "wide_range": wide_range_f32,
    "dense_bucket": dense_bucket_f32,
    "negative": negative_f32,
    "signed_zeros": signed_zeros_f32,
}


def make(value_set: str, N: int, M: int, seed: int = 0, dtype: str = "f32") -> np.ndarray:
    """Generate one of VALUE_SETS as float32 ('f32') or bf16 bit patterns ('bf16')."""
    x = VALUE_SETS[value_set](N, M, seed)
    if dtype == "f32":
        return x
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    raise ValueError(dtype)


def power_law_graph(n_dst: int, n_src: int, avg_degree: float, seed: int = 0, alpha: float = 2.2,
                    max_degree: int | None = None):
    """Synthetic GNN graph in CSR over destination rows (stand-in for the pages'
    Reddit / Flickr / Ogbn-products / Yelp graphs, which are not available).

    In-degrees follow a Pareto tail with exponent ``alpha`` scaled to the mean
    ``avg_degree`` (at least 1, at most ``max_degree`` or ``n_src``); sources
    are uniform. Edge weights are 1 / in-degree (mean aggregation).
    Returns (row_ptr int64 [n_dst + 1], col int32 [E], w float32 [E]).
    """
    g = _rng(seed)
    raw = g.pareto(alpha - 1.0, size=n_dst) + 1.0
    deg = np.maximum(1, np.rint(raw * (avg_degree / raw.mean()))).astype(np.int64)
    deg = np.minimum(deg, max_degree if max_degree is not None else n_src)
    row_ptr = np.zeros(n_dst + 1, dtype=np.int64)
    np.cumsum(deg, out=row_ptr[1:])
    col = g.integers(0, n_src, size=int(row_ptr[-1]), dtype=np.int64).astype(np.int32)
    w = np.repeat((1.0 / deg).astype(np.float32), deg)
    return row_ptr, col, w


def transpose_graph(row_ptr, col, w, n_src: int):
    """The same edges grouped by source row: (t_ptr int64 [n_src + 1],
    t_row int32 [E] = destination of each edge, t_w float32 [E]). Within a source
    the edges keep their forward order (ascending destination)."""
    row_ptr = np.asarray(row_ptr, dtype=np.int64)
    n_dst = row_ptr.shape[0] - 1
    dst = np.repeat(np.arange(n_dst, dtype=np.int32), np.diff(row_ptr))
    order = np.argsort(np.asarray(col), kind="stable")
    t_ptr = np.zeros(n_src + 1, dtype=np.int64)
    np.cumsum(np.bincount(np.asarray(col), minlength=n_src), out=t_ptr[1:])
    return t_ptr, np.ascontiguousarray(dst[order]), np.ascontiguousarray(np.asarray(w, dtype=np.float32)[order])
