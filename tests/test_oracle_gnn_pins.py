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


def test_round_bf16_matches_torch_and_ties(oracle_mod):
    """The oracle's bf16 rounding against torch's conversion (a library
    routine), on normal, subnormal and huge values, plus hand-made ties."""
    torch = pytest.importorskip("torch")
    x = np.concatenate([synth.normal_f32(16, 256, seed=6).ravel(),
                        synth.subnormals_f32(4, 256, seed=7).ravel(),
                        synth.outliers_f32(4, 256, seed=8, mag=3e38).ravel()])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle_mod.round_bf16(x), ref)
    # exact halfway cases: an even last bit stays, an odd one rounds away
    ties = np.array([0x3F808000, 0x3F818000, 0xBF808000, 0xBF818000, 0x00008000, 0x00018000],
                    dtype=np.uint32).view(np.float32)
    np.testing.assert_array_equal(oracle_mod.round_bf16(ties),
                                  np.array([0x3F80, 0x3F82, 0xBF80, 0xBF82, 0x0000, 0x0002], dtype=np.uint16))


def test_fused_backward_scatter_is_the_composition(oracle_mod):
    """sspmm_scatter: at sp_index the bf16 rounding of the sampled product,
    +0 everywhere else -- checked on a graph small enough to sum by hand in
    float64 (every partial sum here is exact in binary32)."""
    # 3 source rows, 2 destination rows, M = 6, k = 2
    sp_index = np.array([[0, 4], [1, 5], [2, 3]], dtype=np.int16)
    dout = np.arange(12, dtype=np.float32).reshape(2, 6) * np.float32(0.5)  # dout[i, m] = (6 i + m) / 2
    # transposed graph: source 0 -> dst 0 (w 1), dst 1 (w 2); source 1 -> dst 1 (w 4); source 2 -> none
    t_ptr = np.array([0, 2, 3, 3], dtype=np.int64)
    t_row = np.array([0, 1, 1], dtype=np.int32)
    t_w = np.array([1.0, 2.0, 4.0], dtype=np.float32)
    g = oracle_mod.sspmm_scatter(t_ptr, t_row, t_w, 2, dout, sp_index, 6)
    want = np.zeros((3, 6), dtype=np.float64)
    want[0, 0] = 1 * 0.0 + 2 * 3.0          # dout[0,0], dout[1,0]
    want[0, 4] = 1 * 2.0 + 2 * 5.0          # dout[0,4], dout[1,4]
    want[1, 1] = 4 * 3.5
    want[1, 5] = 4 * 5.5
    np.testing.assert_array_equal(oracle_mod.widen_bf16(g).astype(np.float64), want)
    # random case: the composition, and zeros off the kept columns
    n_src, n_dst, M, k = 300, 200, 64, 8
    idx = np.stack([np.sort(np.random.default_rng(s).choice(M, k, replace=False)) for s in range(n_src)])
    idx = idx.astype(np.int16)
    row_ptr, col, w = synth.power_law_graph(n_dst, n_src, 6.0, seed=5)
    tp, tr, tw = synth.transpose_graph(row_ptr, col, w, n_src)
    do = synth.normal_f32(n_dst, M, seed=9)
    g = oracle_mod.sspmm_scatter(tp, tr, tw, n_dst, do, idx, M)
    d_sp = oracle_mod.sspmm_cbsr(tp, tr, tw, n_dst, do, idx)
    np.testing.assert_array_equal(np.take_along_axis(g, idx.astype(np.int64), 1), oracle_mod.round_bf16(d_sp))
    mask = np.zeros((n_src, M), dtype=bool)
    np.put_along_axis(mask, idx.astype(np.int64), True, 1)
    assert np.all(g[~mask] == 0)
