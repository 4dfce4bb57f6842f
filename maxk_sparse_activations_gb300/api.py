"""Python binding of the C ABI (argument marshalling only).

Every function here checks shapes and dtypes, allocates outputs with torch when
the caller passes none, and calls the same-named entry point of librtopk.so on
the current CUDA stream. All selection and scatter work runs in the library's
CUDA kernels; nothing here computes on the host. Tensors may live in device
memory or in pinned host memory: on a Grace-Blackwell node the kernels then
read and write the host buffers directly over NVLink-C2C, with no staging copy.
"""
from __future__ import annotations

import contextlib
import ctypes

from typing import Optional

import torch

from . import _lib


def _stream_ptr(stream: Optional[torch.cuda.Stream], device: torch.device) -> int:
    if stream is not None:
        return stream.cuda_stream
    if device.type != "cuda":  # pinned host tensors: the current CUDA device's stream
        device = torch.device("cuda", torch.cuda.current_device())
    return torch.cuda.current_stream(device).cuda_stream


def _need_cuda_2d(t: torch.Tensor, name: str) -> None:
    """Device tensors, or pinned host tensors that the GPU reads and writes in
    place (over NVLink-C2C / PCIe, no staging copy)."""
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or a pinned host tensor")
    if t.dim() != 2 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D tensor")


def _empty_like_home(shape, dtype, x: torch.Tensor) -> torch.Tensor:
    """Output in the same memory as the input: device memory, or pinned host memory."""
    if x.is_cuda:
        return torch.empty(shape, dtype=dtype, device=x.device)
    return torch.empty(shape, dtype=dtype).pin_memory()


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _same_home(t: torch.Tensor, x: torch.Tensor) -> bool:
    """t lives where the kernels launched for x can address it: on x's GPU when x
    is a device tensor; in pinned host memory (or on the current GPU) when x is
    a pinned host tensor."""
    if x.is_cuda:
        return t.is_cuda and t.device == x.device
    return t.is_pinned() or (t.is_cuda and t.device.index == torch.cuda.current_device())


def _check_out(t: torch.Tensor, shape, dtype, x: torch.Tensor, name: str) -> None:
    """A caller-supplied output must be exactly what the kernel writes: the
    kernels write every element of `shape`, so a smaller, strided or misplaced
    tensor would take writes past its storage."""
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch.Tensor")
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype:
        raise ValueError(f"{name} must have shape {tuple(shape)} and dtype {dtype}, "
                         f"got {tuple(t.shape)} {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not _same_home(t, x):
        raise ValueError(f"{name} must live on the same device as the input "
                         f"(or in pinned host memory for pinned inputs)")


def _check_status(t: Optional[torch.Tensor], x: torch.Tensor) -> None:
    if t is None:
        return
    if t.numel() != 1 or t.element_size() != 4 or t.dtype.is_floating_point or not t.is_contiguous():
        raise ValueError("status must be a one-element 32-bit integer tensor")
    if not _same_home(t, x):
        raise ValueError("status must live on the same device as the input (or in pinned host memory)")


def _on(x: torch.Tensor):
    """Makes x's GPU the current device for the call: the library sizes its grids
    and launches on the current device, and the stream is taken from x's device."""
    return torch.cuda.device(x.device) if x.is_cuda else contextlib.nullcontext()


def rtopk_select(x: torch.Tensor, k: int, max_iter: int = -1, eps: float = 0.0, *,
                 vals: Optional[torch.Tensor] = None, idx: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None):
    """Row-wise top-k of x (N x M, fp32 or bf16) -> (vals N x k, idx N x k int32)."""
    vals, idx, _, _ = rtopk_select_stats(x, k, max_iter, eps, vals=vals, idx=idx, stats=False,
                                         stream=stream)
    return vals, idx


def rtopk_select_stats(x: torch.Tensor, k: int, max_iter: int = -1, eps: float = 0.0, *,
                       vals: Optional[torch.Tensor] = None, idx: Optional[torch.Tensor] = None,
                       iters: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                       stats: bool = True, stream: Optional[torch.cuda.Stream] = None):
    """rtopk_select plus per-row pass counts and the device status word.

    Returns (vals, idx, iters, status); iters is int32 of length N and status a
    one-element int32 tensor holding the OR of the STATUS_* bits (zeroed here
    before the launch when this function allocates it).
    """
    _need_cuda_2d(x, "x")
    if x.dtype == torch.float32:
        dtype = _lib.RTOPK_F32
    elif x.dtype == torch.bfloat16:
        dtype = _lib.RTOPK_BF16
    else:
        raise ValueError("x must be float32 or bfloat16")
    N, M = x.shape
    k = int(k)
    if not 1 <= k <= M:
        raise ValueError(f"k must be in [1, M] = [1, {M}], got {k}")
    if vals is None:
        vals = _empty_like_home((N, k), x.dtype, x)
    else:
        _check_out(vals, (N, k), x.dtype, x, "vals")
    if idx is None:
        idx = _empty_like_home((N, k), torch.int32, x)
    else:
        _check_out(idx, (N, k), torch.int32, x, "idx")
    if stats:
        if iters is None:
            iters = _empty_like_home((N,), torch.int32, x)
        else:
            _check_out(iters, (N,), torch.int32, x, "iters")
        if status is None:
            status = _empty_like_home((1,), torch.int32, x).zero_()
        else:
            _check_status(status, x)
    lib = _lib.load()
    with _on(x):
        if stats:
            rc = lib.rtopk_select_stats(x.data_ptr(), N, M, k, int(max_iter), float(eps), dtype,
                                        vals.data_ptr(), idx.data_ptr(), _ptr(iters), _ptr(status),
                                        _stream_ptr(stream, x.device))
        else:
            rc = lib.rtopk_select(x.data_ptr(), N, M, k, int(max_iter), float(eps), dtype,
                                  vals.data_ptr(), idx.data_ptr(), _stream_ptr(stream, x.device))
    _lib.check(rc, "rtopk_select")
    return vals, idx, iters, status


def rtopk_select_bucketed(x: torch.Tensor, k: int, buckets: int, max_iter: int = -1, eps: float = 0.0, *,
                          vals: Optional[torch.Tensor] = None, idx: Optional[torch.Tensor] = None,
                          stream: Optional[torch.cuda.Stream] = None):
    """Bucketed approximate top-k: each row split into `buckets` column blocks,
    each keeping its top-(k / buckets). Returns (vals N x k, idx N x k int32)."""
    _need_cuda_2d(x, "x")
    if x.dtype == torch.float32:
        dtype = _lib.RTOPK_F32
    elif x.dtype == torch.bfloat16:
        dtype = _lib.RTOPK_BF16
    else:
        raise ValueError("x must be float32 or bfloat16")
    N, M = x.shape
    k = int(k)
    if not 1 <= k <= M:
        raise ValueError(f"k must be in [1, M] = [1, {M}], got {k}")
    if vals is None:
        vals = _empty_like_home((N, k), x.dtype, x)
    else:
        _check_out(vals, (N, k), x.dtype, x, "vals")
    if idx is None:
        idx = _empty_like_home((N, k), torch.int32, x)
    else:
        _check_out(idx, (N, k), torch.int32, x, "idx")
    with _on(x):
        rc = _lib.load().rtopk_select_bucketed(x.data_ptr(), N, M, k, int(buckets), int(max_iter), float(eps),
                                               dtype, vals.data_ptr(), idx.data_ptr(),
                                               _stream_ptr(stream, x.device))
    _lib.check(rc, "rtopk_select_bucketed")
    return vals, idx


def maxk_forward(x: torch.Tensor, k: int, max_iter: int = -1, eps: float = 0.0, *,
                 vals: Optional[torch.Tensor] = None, idx: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None):
    """MaxK nonlinearity: bf16 x (N x M) -> CBSR (sp_data bf16 N x k, sp_index int16 N x k)."""
    _need_cuda_2d(x, "x")
    if x.dtype != torch.bfloat16:
        raise ValueError("maxk_forward takes bfloat16 input")
    N, M = x.shape
    k = int(k)
    if not 1 <= k <= M:
        raise ValueError(f"k must be in [1, M] = [1, {M}], got {k}")
    if vals is None:
        vals = _empty_like_home((N, k), torch.bfloat16, x)
    else:
        _check_out(vals, (N, k), torch.bfloat16, x, "vals")
    if idx is None:
        idx = _empty_like_home((N, k), torch.int16, x)
    else:
        _check_out(idx, (N, k), torch.int16, x, "idx")
    with _on(x):
        rc = _lib.load().maxk_forward(x.data_ptr(), N, M, k, int(max_iter), float(eps),
                                      vals.data_ptr(), idx.data_ptr(), _stream_ptr(stream, x.device))
    _lib.check(rc, "maxk_forward")
    return vals, idx


def maxk_backward_scatter(dy: torch.Tensor, idx: torch.Tensor, M: int, *,
                          grad: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                          stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """MaxK backward: dense N x M bf16 gradient, dy at idx and zero elsewhere."""
    _need_cuda_2d(dy, "dy")
    _need_cuda_2d(idx, "idx")
    if dy.dtype != torch.bfloat16 or idx.dtype != torch.int16:
        raise ValueError("dy must be bfloat16 and idx int16")
    if dy.shape != idx.shape:
        raise ValueError("dy and idx must have the same N x k shape")
    if not _same_home(idx, dy):
        raise ValueError("dy and idx must live on the same device")
    N, k = dy.shape
    M = int(M)
    if grad is None:
        grad = _empty_like_home((N, M), torch.bfloat16, dy)
    else:
        _check_out(grad, (N, M), torch.bfloat16, dy, "grad")
    _check_status(status, dy)
    with _on(dy):
        rc = _lib.load().maxk_backward_scatter(dy.data_ptr(), idx.data_ptr(), N, M, int(k),
                                               grad.data_ptr(), _ptr(status), _stream_ptr(stream, dy.device))
    _lib.check(rc, "maxk_backward_scatter")
    return grad


class MaxK(torch.autograd.Function):
    """Autograd wrapper: forward keeps the top-k of each row (CBSR), backward
    scatters the gradient of the kept values back to their recorded positions."""

    @staticmethod
    def forward(ctx, x: torch.Tensor, k: int):
        vals, idx = maxk_forward(x.contiguous(), k)
        ctx.save_for_backward(idx)
        ctx.M = x.shape[1]
        ctx.mark_non_differentiable(idx)
        return vals, idx

    @staticmethod
    def backward(ctx, dvals: torch.Tensor, _didx):
        (idx,) = ctx.saved_tensors
        return maxk_backward_scatter(dvals.contiguous(), idx, ctx.M), None


def _need_1d(t: torch.Tensor, name: str, dtype) -> None:
    if not (t.is_cuda or t.is_pinned()) or t.dim() != 1 or not t.is_contiguous() or t.dtype != dtype:
        raise ValueError(f"{name} must be a contiguous 1-D {dtype} tensor on the GPU (or pinned)")


def maxk_spgemm_forward(row_ptr: torch.Tensor, col_idx: torch.Tensor, edge_w: Optional[torch.Tensor],
                        sp_data: torch.Tensor, sp_index: torch.Tensor, M: int, *,
                        out: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                        stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """MaxK-GNN forward aggregation: dense fp32 (n_dst x M) = graph (CSR over
    destination rows) times the CBSR feature rows (bf16 sp_data, int16 sp_index)."""
    _need_1d(row_ptr, "row_ptr", torch.int64)
    _need_1d(col_idx, "col_idx", torch.int32)
    if edge_w is not None:
        _need_1d(edge_w, "edge_w", torch.float32)
    _need_cuda_2d(sp_data, "sp_data")
    _need_cuda_2d(sp_index, "sp_index")
    if sp_data.dtype != torch.bfloat16 or sp_index.dtype != torch.int16 or sp_data.shape != sp_index.shape:
        raise ValueError("sp_data must be bf16 and sp_index int16, both n_src x k")
    for t, name in ((row_ptr, "row_ptr"), (col_idx, "col_idx"), (edge_w, "edge_w"), (sp_index, "sp_index")):
        if t is not None and not _same_home(t, sp_data):
            raise ValueError(f"{name} must live on the same device as sp_data")
    n_dst = row_ptr.numel() - 1
    n_src, k = sp_data.shape
    M = int(M)
    if out is None:
        out = _empty_like_home((n_dst, M), torch.float32, sp_data)
    else:
        _check_out(out, (n_dst, M), torch.float32, sp_data, "out")
    _check_status(status, sp_data)
    with _on(sp_data):
        rc = _lib.load().maxk_spgemm_forward(row_ptr.data_ptr(), col_idx.data_ptr(), _ptr(edge_w), n_dst, n_src,
                                             sp_data.data_ptr(), sp_index.data_ptr(), M, int(k), out.data_ptr(),
                                             _ptr(status), _stream_ptr(stream, sp_data.device))
    _lib.check(rc, "maxk_spgemm_forward")
    return out


def maxk_sspmm_backward(t_row_ptr: torch.Tensor, t_dst: torch.Tensor, t_edge_w: Optional[torch.Tensor],
                        dout: torch.Tensor, sp_index: torch.Tensor, *, d_sp: Optional[torch.Tensor] = None,
                        status: Optional[torch.Tensor] = None,
                        stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """MaxK-GNN backward of the aggregation: fp32 gradient of the CBSR values
    (n_src x k), sampled at the forward sp_index. The graph is given transposed
    (CSR over source rows: offsets, destination of each edge, edge weights)."""
    _need_1d(t_row_ptr, "t_row_ptr", torch.int64)
    _need_1d(t_dst, "t_dst", torch.int32)
    if t_edge_w is not None:
        _need_1d(t_edge_w, "t_edge_w", torch.float32)
    _need_cuda_2d(dout, "dout")
    _need_cuda_2d(sp_index, "sp_index")
    if dout.dtype != torch.float32 or sp_index.dtype != torch.int16:
        raise ValueError("dout must be float32 and sp_index int16")
    n_dst, M = dout.shape
    n_src, k = sp_index.shape
    if t_row_ptr.numel() != n_src + 1:
        raise ValueError("t_row_ptr must have n_src + 1 entries")
    for t, name in ((t_row_ptr, "t_row_ptr"), (t_dst, "t_dst"), (t_edge_w, "t_edge_w"), (sp_index, "sp_index")):
        if t is not None and not _same_home(t, dout):
            raise ValueError(f"{name} must live on the same device as dout")
    if d_sp is None:
        d_sp = _empty_like_home((n_src, k), torch.float32, dout)
    else:
        _check_out(d_sp, (n_src, k), torch.float32, dout, "d_sp")
    _check_status(status, dout)
    with _on(dout):
        rc = _lib.load().maxk_sspmm_backward(t_row_ptr.data_ptr(), t_dst.data_ptr(), _ptr(t_edge_w), n_src, n_dst,
                                             dout.data_ptr(), sp_index.data_ptr(), int(M), int(k), d_sp.data_ptr(),
                                             _ptr(status), _stream_ptr(stream, dout.device))
    _lib.check(rc, "maxk_sspmm_backward")
    return d_sp


def maxk_sspmm_backward_scatter(t_row_ptr: torch.Tensor, t_dst: torch.Tensor, t_edge_w: Optional[torch.Tensor],
                                dout: torch.Tensor, sp_index: torch.Tensor, M: Optional[int] = None, *,
                                grad: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                                stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """maxk_sspmm_backward with the MaxK backward scatter fused in: the dense
    bf16 gradient of the MaxK input (n_src x M), the CBSR-value gradient
    rounded to bf16 at the forward sp_index and +0 elsewhere. M defaults to
    the width of dout."""
    _need_1d(t_row_ptr, "t_row_ptr", torch.int64)
    _need_1d(t_dst, "t_dst", torch.int32)
    if t_edge_w is not None:
        _need_1d(t_edge_w, "t_edge_w", torch.float32)
    _need_cuda_2d(dout, "dout")
    _need_cuda_2d(sp_index, "sp_index")
    if dout.dtype != torch.float32 or sp_index.dtype != torch.int16:
        raise ValueError("dout must be float32 and sp_index int16")
    n_dst, Md = dout.shape
    M = Md if M is None else int(M)
    if M != Md:
        raise ValueError("M must equal the width of dout")
    n_src, k = sp_index.shape
    if t_row_ptr.numel() != n_src + 1:
        raise ValueError("t_row_ptr must have n_src + 1 entries")
    for t, name in ((t_row_ptr, "t_row_ptr"), (t_dst, "t_dst"), (t_edge_w, "t_edge_w"), (sp_index, "sp_index")):
        if t is not None and not _same_home(t, dout):
            raise ValueError(f"{name} must live on the same device as dout")
    if grad is None:
        grad = _empty_like_home((n_src, M), torch.bfloat16, dout)
    else:
        _check_out(grad, (n_src, M), torch.bfloat16, dout, "grad")
    _check_status(status, dout)
    with _on(dout):
        rc = _lib.load().maxk_sspmm_backward_scatter(t_row_ptr.data_ptr(), t_dst.data_ptr(), _ptr(t_edge_w), n_src,
                                                     n_dst, dout.data_ptr(), sp_index.data_ptr(), int(M), int(k),
                                                     grad.data_ptr(), _ptr(status),
                                                     _stream_ptr(stream, dout.device))
    _lib.check(rc, "maxk_sspmm_backward_scatter")
    return grad


def read_status(status: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> int:
    """Waits for the stream and returns the device status word's bits
    (0 = every row valid; see the RTOPK_STATUS_* bits in include/rtopk.h)."""
    if status.numel() != 1 or status.element_size() != 4:
        raise ValueError("status must be a one-element 32-bit tensor")
    bits = ctypes.c_uint32(0)
    dev = status.device if status.is_cuda else torch.device("cuda", torch.cuda.current_device())
    with _on(status):
        rc = _lib.load().rtopk_status_read(status.data_ptr(), ctypes.addressof(bits), _stream_ptr(stream, dev))
    if rc not in (0, -7):
        _lib.check(rc, "rtopk_status_read")
    return int(bits.value)
