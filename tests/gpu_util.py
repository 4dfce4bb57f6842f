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
