"""CPU oracle for row-wise top-k (RTop-K) and the MaxK layer.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product path
(``maxk_sparse_activations_gb300``) never imports it, and the two share no code:
the arithmetic lives in ``rtopk_oracle.c`` (plain C, binary32, no FMA
contraction), which this module compiles with gcc and calls through ctypes.
Inputs come from the seeded generators in ``maxk_sparse_activations_gb300.synth``,
a module that holds none of the method's arithmetic.

Functions (each follows the page and section named in ``rtopk_oracle.c``):

* ``sort_topk(x, k)`` -- the definition of exact top-k: order the row by value
  descending then index ascending, take the first k, list them by index.
  ("RTop-K ..." summary, "Problem".)
* ``brute_topk(x, k)`` -- the same result found by enumerating every k-subset
  of a tiny row (M <= 20); an independent pin of ``sort_topk``.
* ``replay(x, k, max_iter, eps)`` -- the method step by step: min/max range,
  bisection on the binary32 midpoint with ``>=`` counting, ``max_iter`` early
  stop, ``eps`` stop, and the fill pass of borderline ties by lowest index.
  ("RTop-K ..." summary, "Approach".)
* ``maxk_backward(dy, idx, M)`` -- the MaxK backward scatter: the gradient row
  is zero except at the kept positions. ("MaxK-GNN ...", "How MaxK-GNN works",
  "Asymmetric passes, one mask".)
* ``bucketed_topk(x, k, buckets, max_iter, eps)`` -- bucketed approximate top-k:
  the replay above applied to each of ``buckets`` contiguous column blocks of
  every row with k / buckets kept per block, indices shifted to the row.
  ("Approximate Top-k for Increased Parallelism", abstract.)
* ``spgemm_cbsr(graph, sp_data, sp_index, M)`` -- MaxK-GNN forward aggregation:
  each destination row sums its neighbours' CBSR rows, scattered to their
  columns, in edge order (binary32, no FMA). ("MaxK-GNN ...", "How MaxK-GNN
  works", "Why it works".)
* ``sspmm_cbsr(tgraph, dout, sp_index, n_dst)`` -- the backward sampled product:
  the gradient of each CBSR value sums, over the source row's out-edges in
  order, the edge weight times dout at (destination, sp_index).
* ``round_bf16(x)`` -- binary32 to the nearest bf16, ties to an even last bit,
  chosen by comparing the exact distances to the two neighbouring bf16 values.
* ``sspmm_scatter(tgraph, dout, sp_index, n_dst, M)`` -- the backward sampled
  product followed by the MaxK backward scatter of its bf16-rounded values:
  the dense gradient of the MaxK input. ("MaxK-GNN ...", "Asymmetric passes,
  one mask".)

bf16 inputs are widened exactly to binary32 (the 16 bits become the top half of
the word) and run through the same functions; kept values are the original
16-bit patterns gathered at the kept indices.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rtopk_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, EARG, EINPUT, ENOMEM = 0, -1, -2, -3


def build(force: bool = False) -> str:
    """Compile ``rtopk_oracle.c`` into ``liboracle.so`` (in-tree, git-ignored)."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
            lib.oracle_sort_topk.argtypes = [p, i64, i32, i32, p]
            lib.oracle_brute_topk.argtypes = [p, i64, i32, i32, p]
            lib.oracle_replay.argtypes = [p, i64, i32, i32, i32, f32, p, p]
            lib.oracle_maxk_backward_u16.argtypes = [p, p, i64, i32, i32, p]
            lib.oracle_spgemm_cbsr.argtypes = [p, p, p, i64, i64, p, p, i32, i32, p]
            lib.oracle_sspmm_cbsr.argtypes = [p, p, p, i64, i64, p, p, i32, i32, p]
            for f in (lib.oracle_sort_topk, lib.oracle_brute_topk, lib.oracle_replay,
                      lib.oracle_maxk_backward_u16, lib.oracle_spgemm_cbsr, lib.oracle_sspmm_cbsr):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc == EINPUT:
        raise ValueError(f"{what}: input row is non-finite or has |x| > 1e38")
    if rc != OK:
        raise ValueError(f"{what}: invalid arguments (code {rc})")


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """Exact bf16 -> binary32: the 16 bits become the high half of the word."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _as_f32_rows(x: np.ndarray):
    """Returns (fp32 view used for the arithmetic, original array for values)."""
    if x.dtype == np.float32:
        return np.ascontiguousarray(x), np.ascontiguousarray(x)
    if x.dtype == np.uint16:  # raw bf16 bit patterns
        return widen_bf16(x), np.ascontiguousarray(x)
    raise TypeError("oracle inputs are float32 or uint16 (bf16 bit patterns)")


def _gather(orig: np.ndarray, idx: np.ndarray) -> np.ndarray:
    return np.take_along_axis(orig, idx.astype(np.int64), axis=1)


def sort_topk(x: np.ndarray, k: int):
    """Exact top-k by the definition. Returns (values, int32 indices), N x k."""
    xf, orig = _as_f32_rows(x)
    N, M = xf.shape
    idx = np.empty((N, k), dtype=np.int32)
    _check(_load().oracle_sort_topk(_ptr(xf), N, M, k, _ptr(idx)), "sort_topk")
    return _gather(orig, idx), idx


def brute_topk(x: np.ndarray, k: int):
    """Exact top-k by enumerating all k-subsets (M <= 20)."""
    xf, orig = _as_f32_rows(x)
    N, M = xf.shape
    idx = np.empty((N, k), dtype=np.int32)
    _check(_load().oracle_brute_topk(_ptr(xf), N, M, k, _ptr(idx)), "brute_topk")
    return _gather(orig, idx), idx


def replay(x: np.ndarray, k: int, max_iter: int = -1, eps: float = 0.0):
    """Step-by-step replay of the bisection. Returns (values, idx, iters)."""
    xf, orig = _as_f32_rows(x)
    N, M = xf.shape
    idx = np.empty((N, k), dtype=np.int32)
    iters = np.empty((N,), dtype=np.int32)
    rc = _load().oracle_replay(_ptr(xf), N, M, k, int(max_iter), float(np.float32(eps)),
                               _ptr(idx), _ptr(iters))
    _check(rc, "replay")
    return _gather(orig, idx), idx, iters


def maxk_backward(dy_bits: np.ndarray, idx: np.ndarray, M: int) -> np.ndarray:
    """MaxK backward scatter of bf16 bit patterns into a zero N x M row block."""
    dy = np.ascontiguousarray(dy_bits, dtype=np.uint16)
    ix = np.ascontiguousarray(idx, dtype=np.int16)
    N, k = dy.shape
    grad = np.empty((N, M), dtype=np.uint16)
    _check(_load().oracle_maxk_backward_u16(_ptr(dy), _ptr(ix), N, M, k, _ptr(grad)),
           "maxk_backward")
    return grad


def spgemm_cbsr(row_ptr, col, w, n_src: int, sp_data_bits, sp_index, M: int) -> np.ndarray:
    """Forward aggregation over CBSR: dense (n_dst x M) float32."""
    rp = np.ascontiguousarray(row_ptr, dtype=np.int64)
    cl = np.ascontiguousarray(col, dtype=np.int32)
    wt = None if w is None else np.ascontiguousarray(w, dtype=np.float32)
    sd = np.ascontiguousarray(sp_data_bits, dtype=np.uint16)
    si = np.ascontiguousarray(sp_index, dtype=np.int16)
    n_dst = rp.shape[0] - 1
    k = sd.shape[1]
    out = np.empty((n_dst, M), dtype=np.float32)
    rc = _load().oracle_spgemm_cbsr(_ptr(rp), _ptr(cl), None if wt is None else _ptr(wt), n_dst, n_src,
                                    _ptr(sd), _ptr(si), M, k, _ptr(out))
    _check(rc, "spgemm_cbsr")
    return out


def sspmm_cbsr(t_ptr, t_row, t_w, n_dst: int, dout, sp_index) -> np.ndarray:
    """Backward sampled product: float32 (n_src x k) gradient of the CBSR values."""
    tp = np.ascontiguousarray(t_ptr, dtype=np.int64)
    tr = np.ascontiguousarray(t_row, dtype=np.int32)
    tw = None if t_w is None else np.ascontiguousarray(t_w, dtype=np.float32)
    do = np.ascontiguousarray(dout, dtype=np.float32)
    si = np.ascontiguousarray(sp_index, dtype=np.int16)
    n_src, k = si.shape
    M = do.shape[1]
    out = np.empty((n_src, k), dtype=np.float32)
    rc = _load().oracle_sspmm_cbsr(_ptr(tp), _ptr(tr), None if tw is None else _ptr(tw), n_src, n_dst,
                                   _ptr(do), _ptr(si), M, k, _ptr(out))
    _check(rc, "sspmm_cbsr")
    return out


def bucketed_topk(x: np.ndarray, k: int, buckets: int, max_iter: int = -1, eps: float = 0.0):
    """Bucketed top-k: per row, each of `buckets` column blocks keeps its
    top-(k / buckets) by the replay; returns (values, int32 indices), N x k."""
    N, M = x.shape
    if M % buckets or k % buckets:
        raise ValueError("buckets must divide M and k")
    mb, kb = M // buckets, k // buckets
    xb = np.ascontiguousarray(x).reshape(N * buckets, mb)
    vals, idx, _ = replay(xb, kb, max_iter, eps)
    offset = (np.arange(N * buckets) % buckets * mb).astype(np.int32)[:, None]
    return vals.reshape(N, k), (idx + offset).reshape(N, k)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Finite binary32 -> nearest bf16 bit pattern, ties to an even last bit.

    The two candidates are the bf16 values that bracket x: its top 16 bits
    (toward zero) and the next bf16 away from zero. Their distances to x are
    exact in float64, so the nearer one is picked exactly.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lo = (b >> np.uint32(16)).astype(np.uint32)          # toward zero
    hi = lo + np.uint32(1)                                # one bf16 step away from zero
    xv = b.view(np.float32).astype(np.float64)
    lv = (lo << np.uint32(16)).view(np.float32).astype(np.float64)
    hv = (hi << np.uint32(16)).view(np.float32).astype(np.float64)
    dl, dh = np.abs(xv - lv), np.abs(hv - xv)
    pick_hi = (dh < dl) | ((dh == dl) & ((lo & np.uint32(1)) == 1))
    return np.where(pick_hi, hi, lo).astype(np.uint16)


def sspmm_scatter(t_ptr, t_row, t_w, n_dst: int, dout, sp_index, M: int) -> np.ndarray:
    """Backward sampled product, rounded to bf16 and scattered to a dense
    n_src x M bf16 (bit pattern) gradient of the MaxK input."""
    d_sp = sspmm_cbsr(t_ptr, t_row, t_w, n_dst, dout, sp_index)
    return maxk_backward(round_bf16(d_sp), sp_index, M)
