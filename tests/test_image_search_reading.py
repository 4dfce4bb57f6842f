"""CPU check of the reading behind the packed exact search.

In exact mode the result is one set -- the k largest values, ties at the k-th
value to the lowest index ("RTop-K ..." summary, "Problem") -- so the bisection
may count on any monotone image h of the row (x <= y implies h(x) <= h(y)):

* a threshold t with #{h(x) >= t} == k gives exactly the top-k set;
* when no image value is left strictly inside the bracket [lo, hi), the k-th
  value lies in the bucket {lo <= h(x) < hi}, and a binary32 bisection started
  from [min of the bucket, next binary32 above its max] finishes it.

This test replays that search step by step in numpy on binary16 images of fp32
rows (nearest, saturated at +-65504) and on bf16 rows themselves, and compares
the kept index sets with the definition (oracle.sort_topk) on every value set,
including the ones built to defeat a 16-bit image. It checks the mathematics of
the reading, not the CUDA kernel (the GPU tests compare that one).
"""
import numpy as np
import pytest

import oracle
from maxk_sparse_activations_gb300 import synth

F32 = np.float32


def _f16_image(x):
    return np.clip(x.astype(F32), F32(-65504), F32(65504)).astype(np.float16).astype(F32)


def _bf16_round(x):
    b = np.asarray(x, dtype=F32).reshape(-1).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(F32).reshape(np.shape(x))


def _next_up(v):
    v = F32(v)
    if v == 0:
        return np.array([1], np.uint32).view(F32)[0]
    b = np.array([v], F32).view(np.int32)[0]
    return np.array([b + 1 if v > 0 else b - 1], np.int32).view(F32)[0]


def _binary32_finish(x, lo, hi, k):
    """Bisection with binary32 midpoints from a valid bracket, then the fill
    (keep x >= hi, fill from [lo, hi) by ascending index)."""
    while True:
        mid = F32(F32(lo + hi) * F32(0.5))
        if not (lo < mid < hi):
            break
        c = int((x >= mid).sum())
        if c == k:
            lo = mid
            break
        if c > k:
            lo = mid
        else:
            hi = mid
    keep_s = np.flatnonzero(x >= hi)
    fill = np.flatnonzero((x >= lo) & (x < hi))[: k - keep_s.size]
    return np.sort(np.concatenate([keep_s, fill]))


def _image_search(x, k, bf16):
    """The coarse search on the image h, then the bucket finish."""
    h = x.copy() if bf16 else _f16_image(x)
    rnd = (lambda v: _bf16_round(np.array([v], F32))[0]) if bf16 else (lambda v: _f16_image(np.array([v], F32))[0])
    lo, hi = rnd(x.min()), rnd(x.max())
    if int((h >= hi).sum()) >= k:  # ties at the top image
        b_lo, b_hi = hi, F32(np.inf)
    else:
        while True:
            m = rnd(F32(F32(lo + hi) * F32(0.5)))
            if not (lo < m < hi):
                break
            c = int((h >= m).sum())
            if c == k:
                return np.flatnonzero(h >= m)
            if c > k:
                lo = m
            else:
                hi = m
        b_lo, b_hi = lo, hi
    bucket = (h >= b_lo) & ~(h >= b_hi)
    return _binary32_finish(x, F32(x[bucket].min()), _next_up(x[bucket].max()), k)


VALUE_SETS = ["normal", "uniform", "int_ties", "all_equal", "outliers", "subnormal", "wide_range",
              "dense_bucket", "negative", "signed_zeros"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("value_set", VALUE_SETS)
def test_image_search_is_the_definition(value_set, dtype):
    M = 128
    x = synth.make(value_set, 40, M, seed=3, dtype=dtype)
    xf = oracle.widen_bf16(x) if dtype == "bf16" else x
    for k in (1, 7, 32, 33, 100, M):
        _, want = oracle.sort_topk(x, k)
        for r in range(x.shape[0]):
            got = _image_search(xf[r], k, dtype == "bf16")
            np.testing.assert_array_equal(got, want[r], err_msg=f"{value_set} {dtype} k={k} row {r}")


def test_bucket_finish_is_needed():
    """The binary32 finish carries weight: ending the search on the collapsed
    binary16 bracket and filling its bucket by lowest index (no finish) gives a
    different set on rows whose values sit inside one binary16 bucket."""
    x = synth.make("dense_bucket", 20, 128, seed=3)
    _, want = oracle.sort_topk(x, 32)
    wrong = 0
    for r in range(x.shape[0]):
        h = _f16_image(x[r])
        lo, hi = F32(h.min()), F32(h.max())
        if int((h >= hi).sum()) >= 32:
            lo, hi = hi, F32(np.inf)
        keep = np.flatnonzero(h >= hi)
        fill = np.flatnonzero((h >= lo) & (h < hi))[: 32 - keep.size]
        wrong += not np.array_equal(np.sort(np.concatenate([keep, fill])), want[r])
        assert np.array_equal(_image_search(x[r], 32, False), want[r])
    assert wrong > 0


def test_sign_of_the_rounded_difference_decides_the_compare():
    """The 16-bit search counts h >= t as "RN(h - t) has its sign bit clear".
    That holds for every finite binary16 image h other than -0 (images are
    canonicalised by adding +0) and every threshold t, zeros and subnormals
    included: checked exhaustively over all finite images against thresholds
    spread over the whole range (numpy's binary16 subtraction rounds once, to
    nearest even)."""
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
    h = h[np.isfinite(h)]
    h = h[h.view(np.uint16) != 0x8000]          # canonical: no -0
    rng = np.random.default_rng(0)
    special = np.array([0.0, -0.0, 6e-8, -6e-8, 6.1e-5, -6.1e-5, 1.0, -1.0, 65504.0, -65504.0],
                       dtype=np.float16)
    t = np.concatenate([special, rng.choice(h, size=1500, replace=False)])
    with np.errstate(over="ignore", invalid="ignore"):
        for chunk in np.array_split(t, 10):
            d = h[None, :] - chunk[:, None]
            sign_clear = (d.view(np.uint16) & 0x8000) == 0
            assert np.array_equal(sign_clear, h[None, :] >= chunk[:, None])


def test_binary32_difference_sign_decides_the_compare():
    """The binary32 counting pass reads x >= t off the sign bit of the rounded
    difference x - t. For x without -0 and finite t this holds for every pair:
    equal values give +0 (x - x rounds to +0 in round-to-nearest), and a nonzero
    difference of binary32 values never rounds to zero with gradual underflow
    (it is at least the smallest subnormal). Checked over zeros of both signs
    as t, subnormals, values around the extremes, and random bit patterns."""
    rng = np.random.default_rng(11)
    special = np.array([0.0, -0.0, 1e-45, -1e-45, 2e-45, -2e-45, 1.1754942e-38, -1.1754942e-38,
                        1.1754944e-38, -1.1754944e-38, 1.0, -1.0, 1e38, -1e38, 3.0e38, -3.0e38],
                       dtype=F32)
    bits = rng.integers(0, 1 << 32, size=4000, dtype=np.uint64).astype(np.uint32)
    rand = bits.view(F32)
    rand = rand[np.isfinite(rand) & (np.abs(rand) <= F32(1e38))]
    subn = (rng.integers(1, 1 << 23, size=500, dtype=np.uint32)
            | (rng.integers(0, 2, size=500, dtype=np.uint32) << np.uint32(31))).view(F32)
    vals = np.concatenate([special, rand, subn]).astype(F32)
    x = vals + F32(0.0)  # canonical: -0 -> +0
    assert not np.any((x == 0) & np.signbit(x))
    with np.errstate(over="ignore"):
        for t in vals:
            d = (x - t).astype(F32)
            got = ~np.signbit(d)
            np.testing.assert_array_equal(got, x >= t, err_msg=f"t={t!r}")
