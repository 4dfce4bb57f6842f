"""Accuracy of early-stopped top-k against exact top-k (host-side reporting).

The RTop-K summary ("Key results") reports, for early stopping, a hit rate and
"max and min relative errors" without defining them. This module uses:

* hit rate   = |I_approx intersect I_exact| / k per row;
* r_max      = |max(v_approx) - max(v_exact)| / |max(v_exact)|;
* r_min      = |min(v_approx) - min(v_exact)| / |min(v_exact)|;
  a zero denominator falls back to the absolute difference;
* r_sum      = |sum(v_approx) - sum(v_exact)| / |sum(v_exact)| (supplementary).

All quantities are computed in float64 per row and summarised as mean and worst
over rows. This is reporting, not a step of the selection, and runs on the host.
"""
from __future__ import annotations

import numpy as np


def _to_f64(v: np.ndarray) -> np.ndarray:
    if v.dtype == np.uint16:  # bf16 bit patterns
        return (v.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return v.astype(np.float64)


def _rel(a: np.ndarray, e: np.ndarray) -> np.ndarray:
    d = np.abs(a - e)
    den = np.abs(e)
    out = d.copy()
    nz = den > 0
    out[nz] = d[nz] / den[nz]
    return out


def compare(vals_a, idx_a, vals_e, idx_e) -> dict:
    """Per-row accuracy of (vals_a, idx_a) against exact (vals_e, idx_e), N x k each."""
    idx_a = np.asarray(idx_a).astype(np.int64)
    idx_e = np.asarray(idx_e).astype(np.int64)
    N, k = idx_e.shape
    if N == 0:
        return {"rows": 0}
    # rows are sets of distinct indices: count common members via sorted merge
    sa = np.sort(idx_a, axis=1)
    se = np.sort(idx_e, axis=1)
    M = int(max(sa.max(), se.max())) + 1
    hit = np.zeros(N, dtype=np.int64)
    offs = (np.arange(N, dtype=np.int64) * M)[:, None]
    inter = np.intersect1d((sa + offs).ravel(), (se + offs).ravel(), assume_unique=True)
    np.add.at(hit, inter // M, 1)
    hit_rate = hit / float(k)
    va, ve = _to_f64(np.asarray(vals_a)), _to_f64(np.asarray(vals_e))
    r_max = _rel(va.max(axis=1), ve.max(axis=1))
    r_min = _rel(va.min(axis=1), ve.min(axis=1))
    r_sum = _rel(va.sum(axis=1), ve.sum(axis=1))
    return {
        "rows": int(N),
        "hit_rate_mean": float(hit_rate.mean()), "hit_rate_worst": float(hit_rate.min()),
        "r_max_mean": float(r_max.mean()), "r_max_worst": float(r_max.max()),
        "r_min_mean": float(r_min.mean()), "r_min_worst": float(r_min.max()),
        "r_sum_mean": float(r_sum.mean()), "r_sum_worst": float(r_sum.max()),
    }
