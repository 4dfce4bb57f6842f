"""GPU parity of the MaxK-GNN aggregation over CBSR (forward SpGEMM, backward
sampled product) against the oracle: bit-exact, since both add in edge order
with one binary32 rounding per product and per sum (forward rows with more than
512 edges are summed in chunks and compared within the binary32 bound). CBSR inputs come from the
oracle's own selection, so no oracle input comes from the CUDA path.
("MaxK-GNN: Extremely Fast GPU Kernel Design for Accelerating Graph Neural
Networks Training", "How MaxK-GNN works", "Asymmetric passes, one mask".)
"""
import numpy as np
import pytest
import torch

import oracle
from maxk_sparse_activations_gb300 import api, synth

from gpu_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    oracle.build()


def _cbsr(n, M, k, seed):
    x = synth.normal_bf16(n, M, seed=seed)
    _, idx, _ = oracle.replay(x, k)
    return np.take_along_axis(x, idx.astype(np.int64), 1), idx.astype(np.int16)


def _t(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.cuda() if dtype is None else t.to(dtype).cuda()


def _run_fwd(row_ptr, col, w, sp_data, sp_index, M):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = api.maxk_spgemm_forward(_t(row_ptr), _t(col), None if w is None else _t(w), to_dev(sp_data),
                                  _t(sp_index), M, status=st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("M,k,weighted", [(256, 32, True), (256, 32, False), (128, 16, True),
                                          (512, 64, True), (1024, 128, True), (2048, 256, True),
                                          (100, 7, True), (8192, 64, True)])
def test_forward_bit_exact(M, k, weighted):
    n_src, n_dst = 3000, 2500
    sp_data, sp_index = _cbsr(n_src, M, k, seed=M + k)
    # in-degree <= 512: every row takes the sequential single-warp path
    row_ptr, col, w = synth.power_law_graph(n_dst, n_src, 16.0, seed=1, max_degree=512)
    w = w if weighted else None
    got, st = _run_fwd(row_ptr, col, w, sp_data, sp_index, M)
    want = oracle.spgemm_cbsr(row_ptr, col, w, n_src, sp_data, sp_index, M)
    assert st == 0
    np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))


def test_forward_large_graph_and_empty_rows():
    n_src, n_dst, M, k = 1 << 16, 1 << 17, 256, 32
    sp_data, sp_index = _cbsr(n_src, M, k, seed=3)
    row_ptr, col, w = synth.power_law_graph(n_dst, n_src, 48.0, seed=4)
    # give every 97th destination row no edges at all
    deg = np.diff(row_ptr)
    keep = np.ones(col.shape[0], dtype=bool)
    for i in range(0, n_dst, 97):
        keep[row_ptr[i]:row_ptr[i + 1]] = False
    deg[::97] = 0
    row_ptr2 = np.zeros_like(row_ptr)
    np.cumsum(deg, out=row_ptr2[1:])
    col2, w2 = col[keep], w[keep]
    got, st = _run_fwd(row_ptr2, col2, w2, sp_data, sp_index, M)
    want = oracle.spgemm_cbsr(row_ptr2, col2, w2, n_src, sp_data, sp_index, M)
    assert st == 0
    assert np.all(got[::97] == 0)
    deg = np.diff(row_ptr2)
    light = deg <= 512
    assert (~light).sum() > 10  # the power-law tail exercises the chunked path
    np.testing.assert_array_equal(got[light].view(np.uint32), want[light].view(np.uint32))
    # chunked rows: both sums are within (deg + 1) 2^-24 sum|terms| of the exact sum
    H = np.zeros((n_src, M))
    vals = (sp_data.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    np.put_along_axis(H, sp_index.astype(np.int64), vals, axis=1)
    for i in np.flatnonzero(~light):
        e = slice(row_ptr2[i], row_ptr2[i + 1])
        absref = np.abs(w2[e].astype(np.float64)) @ np.abs(H[col2[e]])
        bound = 2 * (deg[i] + 1) * 2.0 ** -24 * absref * 1.0001
        assert np.all(np.abs(got[i].astype(np.float64) - want[i]) <= bound), i


@pytest.mark.parametrize("M,k", [(256, 32), (512, 64), (1024, 256), (100, 7)])
def test_backward_bit_exact(M, k):
    n_src, n_dst = 2000, 3000
    _, sp_index = _cbsr(n_src, M, k, seed=11)
    row_ptr, col, w = synth.power_law_graph(n_dst, n_src, 16.0, seed=12)
    t_ptr, t_row, t_w = synth.transpose_graph(row_ptr, col, w, n_src)
    dout = synth.normal_f32(n_dst, M, seed=13)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = api.maxk_sspmm_backward(_t(t_ptr), _t(t_row), _t(t_w), _t(dout), _t(sp_index), status=st)
    torch.cuda.synchronize()
    want = oracle.sspmm_cbsr(t_ptr, t_row, t_w, n_dst, dout, sp_index)
    assert int(st.item()) == 0
    np.testing.assert_array_equal(got.cpu().numpy().view(np.uint32), want.view(np.uint32))


def test_bad_edges_and_indices_are_flagged():
    n_src, n_dst, M, k = 50, 40, 64, 8
    sp_data, sp_index = _cbsr(n_src, M, k, seed=21)
    row_ptr, col, w = synth.power_law_graph(n_dst, n_src, 5.0, seed=22)
    col = col.copy()
    col[3] = n_src + 5  # out of range: skipped
    sp_index = sp_index.copy()
    sp_index[7, 2] = 999
    got, st = _run_fwd(row_ptr, col, w, sp_data, sp_index, M)
    assert st & 0x10 and st & 0x8


def test_fused_maxk_layer_chain():
    """maxk_forward -> aggregation -> backward sampled product -> MaxK scatter,
    against the same chain on the oracle."""
    n, M, k = 4096, 256, 32
    xb = synth.normal_bf16(n, M, seed=31)
    row_ptr, col, w = synth.power_law_graph(n, n, 24.0, seed=32, max_degree=512)
    t_ptr, t_row, t_w = synth.transpose_graph(row_ptr, col, w, n)
    dout = synth.normal_f32(n, M, seed=33)
    fv, fi = api.maxk_forward(to_dev(xb), k)
    out = api.maxk_spgemm_forward(_t(row_ptr), _t(col), _t(w), fv, fi, M)
    dsp = api.maxk_sspmm_backward(_t(t_ptr), _t(t_row), _t(t_w), _t(dout), fi)
    dx = api.maxk_backward_scatter(dsp.to(torch.bfloat16), fi, M)
    torch.cuda.synchronize()
    ov, oi, _ = oracle.replay(xb, k)
    o_out = oracle.spgemm_cbsr(row_ptr, col, w, n, ov, oi.astype(np.int16), M)
    o_dsp = oracle.sspmm_cbsr(t_ptr, t_row, t_w, n, dout, oi.astype(np.int16))
    o_dx = oracle.maxk_backward(synth.f32_to_bf16_bits(o_dsp), oi.astype(np.int16), M)
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32), o_out.view(np.uint32))
    np.testing.assert_array_equal(dsp.cpu().numpy().view(np.uint32), o_dsp.view(np.uint32))
    np.testing.assert_array_equal(dx.cpu().view(torch.int16).numpy().view(np.uint16), o_dx)


@pytest.mark.parametrize("M,k,weighted", [(256, 32, True), (512, 64, False), (100, 7, True), (2048, 256, True),
                                          (8192, 64, True), (36, 4, True)])
def test_fused_backward_scatter_bit_exact(M, k, weighted):
    """maxk_sspmm_backward_scatter against the oracle's backward product,
    rounded to bf16 and scattered (the composition it replaces)."""
    n_src, n_dst = 1500, 1200
    _, sp_index = _cbsr(n_src, M, k, seed=41 + M)
    row_ptr, col, w = synth.power_law_graph(n_dst, n_src, 12.0, seed=42)
    t_ptr, t_row, t_w = synth.transpose_graph(row_ptr, col, w, n_src)
    t_w = t_w if weighted else None
    dout = synth.normal_f32(n_dst, M, seed=43)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = api.maxk_sspmm_backward_scatter(_t(t_ptr), _t(t_row), None if t_w is None else _t(t_w), _t(dout),
                                          _t(sp_index), M, status=st)
    torch.cuda.synchronize()
    want = oracle.sspmm_scatter(t_ptr, t_row, t_w, n_dst, dout, sp_index, M)
    assert int(st.item()) == 0
    np.testing.assert_array_equal(got.cpu().view(torch.int16).numpy().view(np.uint16), want)


def test_fused_backward_scatter_flags_bad_index():
    n_src, n_dst, M, k = 64, 50, 64, 8
    _, sp_index = _cbsr(n_src, M, k, seed=51)
    sp_index = sp_index.copy()
    sp_index[5, 3] = 300
    row_ptr, col, w = synth.power_law_graph(n_dst, n_src, 4.0, seed=52)
    t_ptr, t_row, t_w = synth.transpose_graph(row_ptr, col, w, n_src)
    dout = synth.normal_f32(n_dst, M, seed=53)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = api.maxk_sspmm_backward_scatter(_t(t_ptr), _t(t_row), _t(t_w), _t(dout), _t(sp_index), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 0x8
    # every other row is exact (the oracle gets an in-range stand-in for the bad entry)
    g = got.cpu().view(torch.int16).numpy().view(np.uint16)
    ok_rows = np.r_[0:5, 6:n_src]
    want = oracle.sspmm_scatter(t_ptr, t_row, t_w, n_dst, dout, np.where(sp_index == 300, 0, sp_index), M)
    np.testing.assert_array_equal(g[ok_rows], want[ok_rows])


def test_fused_backward_scatter_flags_bad_edge():
    n_src, n_dst, M, k = 60, 40, 64, 8
    _, sp_index = _cbsr(n_src, M, k, seed=61)
    row_ptr, col, w = synth.power_law_graph(n_dst, n_src, 4.0, seed=62)
    t_ptr, t_row, t_w = synth.transpose_graph(row_ptr, col, w, n_src)
    t_row = t_row.copy()
    t_row[0] = n_dst + 3  # destination out of range: skipped and flagged
    dout = synth.normal_f32(n_dst, M, seed=63)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = api.maxk_sspmm_backward_scatter(_t(t_ptr), _t(t_row), _t(t_w), _t(dout), _t(sp_index), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 0x10
    # the source row owning edge 0 sums its other edges; every other row is exact
    src0 = int(np.searchsorted(t_ptr, 0, side="right") - 1)
    keep = np.ones(t_row.shape[0], dtype=bool)
    keep[0] = False
    deg = np.diff(t_ptr)
    deg[src0] -= 1
    t_ptr2 = np.zeros_like(t_ptr)
    np.cumsum(deg, out=t_ptr2[1:])
    want = oracle.sspmm_scatter(t_ptr2, t_row[keep], t_w[keep], n_dst, dout, sp_index, M)
    np.testing.assert_array_equal(got.cpu().view(torch.int16).numpy().view(np.uint16), want)
