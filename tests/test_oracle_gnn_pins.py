"""Pins of the oracle's MaxK-GNN aggregation (forward SpGEMM over CBSR) and its
backward sampled product, against facts that do not come from the oracle:
a hand-worked graph, the float64 dense product within the binary32 rounding
bound, and the adjoint identity <A H, G> = <H, A^T G> restricted to the CBSR
entries ("MaxK-GNN: Extremely Fast GPU Kernel Design for Accelerating Graph
Neural Networks Training", "How MaxK-GNN works", "Asymmetric passes, one mask").
"""
import numpy as np
import pytest

from maxk_sparse_activations_gb300 import synth


def _bf16(x):
    return synth.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def test_hand_worked_aggregation(oracle_mod):
    # 2 source rows with k = 2 of M = 4 columns, 2 destination rows
    sp_data = _bf16([[1.0, 2.0], [3.0, -1.0]])
    sp_index = np.array([[0, 2], [2, 3]], dtype=np.int16)
    # dst 0 <- src 0 (w 0.5), src 1 (w 0.5);  dst 1 <- src 1 (w 2)
    row_ptr = np.array([0, 2, 3]); col = np.array([0, 1, 1]); w = np.array([0.5, 0.5, 2.0], np.float32)
    out = oracle_mod.spgemm_cbsr(row_ptr, col, w, 2, sp_data, sp_index, 4)
    # dst 0: col0 = 0.5*1, col2 = 0.5*2 + 0.5*3 = 2.5, col3 = 0.5*-1 ; dst 1: col2 = 6, col3 = -2
    np.testing.assert_array_equal(out, np.array([[0.5, 0, 2.5, -0.5], [0, 0, 6, -2]], np.float32))
    # backward with dout = ones: d_sp[j, t] = sum of the weights of j's out-edges
    t_ptr, t_row, t_w = synth.transpose_graph(row_ptr, col, w, 2)
    d = oracle_mod.sspmm_cbsr(t_ptr, t_row, t_w, 2, np.ones((2, 4), np.float32), sp_index)
    np.testing.assert_array_equal(d, np.array([[0.5, 0.5], [2.5, 2.5]], np.float32))


def _dense_H(sp_data, sp_index, M):
    H = np.zeros((sp_data.shape[0], M))
    vals = (sp_data.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    np.put_along_axis(H, sp_index.astype(np.int64), vals, axis=1)
    return H


@pytest.mark.parametrize("M,k", [(256, 32), (128, 16), (512, 64)])
def test_forward_matches_float64_product(oracle_mod, M, k):
    n = 3000
    x = synth.normal_bf16(n, M, seed=2)
    _, idx, _ = oracle_mod.replay(x, k)
    sp_data = np.take_along_axis(x, idx.astype(np.int64), 1)
    sp_index = idx.astype(np.int16)
    row_ptr, col, w = synth.power_law_graph(n, n, 12.0, seed=3)
    out = oracle_mod.spgemm_cbsr(row_ptr, col, w, n, sp_data, sp_index, M)
    H = _dense_H(sp_data, sp_index, M)
    ref = np.zeros((n, M))
    absref = np.zeros((n, M))
    for i in range(n):
        e = slice(row_ptr[i], row_ptr[i + 1])
        ref[i] = w[e].astype(np.float64) @ H[col[e]]
        absref[i] = np.abs(w[e].astype(np.float64)) @ np.abs(H[col[e]])
    deg = np.diff(row_ptr)[:, None]
    # binary32 running sum of deg rounded products: |err| <= (deg + 1) u sum|terms|, u = 2^-24
    bound = (deg + 1) * 2.0 ** -24 * absref * 1.0001
    assert np.all(np.abs(out - ref) <= bound)


def test_backward_is_the_adjoint(oracle_mod):
    n_dst, n_src, M, k = 1500, 2000, 256, 32
    x = synth.normal_bf16(n_src, M, seed=5)
    _, idx, _ = oracle_mod.replay(x, k)
    sp_data = np.take_along_axis(x, idx.astype(np.int64), 1)
    sp_index = idx.astype(np.int16)
    row_ptr, col, w = synth.power_law_graph(n_dst, n_src, 20.0, seed=6)
    G = synth.normal_f32(n_dst, M, seed=7)
    out = oracle_mod.spgemm_cbsr(row_ptr, col, w, n_src, sp_data, sp_index, M).astype(np.float64)
    t_ptr, t_row, t_w = synth.transpose_graph(row_ptr, col, w, n_src)
    dsp = oracle_mod.sspmm_cbsr(t_ptr, t_row, t_w, n_dst, G, sp_index).astype(np.float64)
    vals = (sp_data.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    lhs = float(np.sum(out * G))
    rhs = float(np.sum(vals * dsp))
    assert abs(lhs - rhs) <= 1e-4 * (abs(lhs) + float(np.sum(np.abs(out * G))) * 1e-3)


def test_transpose_graph_matches_scipy():
    sp = pytest.importorskip("scipy.sparse")
    row_ptr, col, w = synth.power_law_graph(700, 900, 9.0, seed=1)
    t_ptr, t_row, t_w = synth.transpose_graph(row_ptr, col, w, 900)
    A = sp.csr_matrix((w, col, row_ptr), shape=(700, 900))
    At = A.T.tocsr()
    At.sort_indices()
    np.testing.assert_array_equal(t_ptr, At.indptr)
    np.testing.assert_array_equal(t_row, At.indices)
    np.testing.assert_array_equal(t_w, At.data.astype(np.float32))


def test_power_law_degrees():
    row_ptr, col, w = synth.power_law_graph(20000, 20000, 30.0, seed=0)
    deg = np.diff(row_ptr)
    assert deg.min() >= 1 and abs(deg.mean() - 30.0) < 3.0
    assert deg.max() > 10 * deg.mean()  # heavy tail
    np.testing.assert_allclose(np.add.reduceat(w.astype(np.float64), row_ptr[:-1]), 1.0, rtol=1e-5)
