"""Helpers for the GPU parity tests: move seeded numpy inputs to the device,
run the CUDA path through the binding, bring results back as numpy."""
import numpy as np
import torch


def to_dev(x: np.ndarray, device="cuda") -> torch.Tensor:
    if x.dtype == np.float32:
        return torch.from_numpy(np.ascontiguousarray(x)).to(device)
    if x.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(device)
    raise TypeError(x.dtype)


def vals_np(t: torch.Tensor) -> np.ndarray:
    """Device values as raw bit patterns (uint32 for fp32, uint16 for bf16)."""
    if t.dtype == torch.float32:
        return t.cpu().numpy().view(np.uint32)
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def ref_bits(v: np.ndarray) -> np.ndarray:
    return v.view(np.uint32) if v.dtype == np.float32 else v.view(np.uint16)


def assert_same_selection(gv, gi, ov, oi, rows=None, what=""):
    """Bit-exact equality of values and indices (optionally on a row subset)."""
    gv = vals_np(gv) if isinstance(gv, torch.Tensor) else gv
    gi = gi.cpu().numpy() if isinstance(gi, torch.Tensor) else gi
    if rows is not None:
        gv, gi = gv[rows], gi[rows]
    gi = gi.astype(np.int64)
    oi = oi.astype(np.int64)
    bad = np.flatnonzero((gi != oi).any(axis=1) | (gv != ref_bits(ov)).any(axis=1))
    assert bad.size == 0, (f"{what}: {bad.size} rows differ; first row {bad[0]}: "
                           f"gpu idx {gi[bad[0]][:16]} oracle idx {oi[bad[0]][:16]}")


def oracle_rows(fn, x, *args, threads=None):
    """Run an oracle function over contiguous row blocks of x on every host
    core and stack the per-block results (the oracle's C code releases the GIL
    inside ctypes calls, so the blocks run in parallel). Results are the same
    as one call over all rows: every oracle function works row by row."""
    import concurrent.futures as cf
    import os

    n = x.shape[0]
    threads = threads or min(32, os.cpu_count() or 1)
    if n < 4096 or threads == 1:
        return fn(x, *args)
    bounds = np.linspace(0, n, threads + 1).astype(np.int64)
    blocks = [(int(a), int(b)) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
    with cf.ThreadPoolExecutor(max_workers=len(blocks)) as ex:
        parts = list(ex.map(lambda ab: fn(x[ab[0]:ab[1]], *args), blocks))
    if isinstance(parts[0], tuple):
        return tuple(np.concatenate([p[j] for p in parts]) for j in range(len(parts[0])))
    return np.concatenate(parts)
