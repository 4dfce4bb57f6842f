"""GPU parity: the CUDA path (through the C ABI binding) against the CPU oracle.

Bar: bit-exact values (raw bits) and indices, and identical per-row pass counts,
in exact mode and in every early-stop / eps mode (the oracle replays the same
binary32 search). Workloads follow the five configurations of the method's
evaluation shape: M = 256, k = 32 normal rows; the MaxK-shaped early-stop study;
the shape sweep; long rows with adversarial values; the fused MaxK layer.
"""
import numpy as np
import pytest
import torch

import oracle
from maxk_sparse_activations_gb300 import accuracy, api, synth

from gpu_util import assert_same_selection, oracle_rows, to_dev, vals_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    oracle.build()


def _run(x, k, max_iter=-1, eps=0.0):
    xt = to_dev(x)
    v, i, it, st = api.rtopk_select_stats(xt, k, max_iter, eps)
    torch.cuda.synchronize()
    return v, i, it.cpu().numpy(), int(st.item())


def _check_full(x, k, max_iter=-1, eps=0.0, what=""):
    v, i, it, st = _run(x, k, max_iter, eps)
    ov, oi, oit = oracle.replay(x, k, max_iter, eps)
    assert st == 0, f"{what}: status {st:#x}"
    assert_same_selection(v, i, ov, oi, what=what)
    np.testing.assert_array_equal(it, oit, err_msg=f"{what}: pass counts differ")
    return v, i, ov, oi


def _sample_rows(N, n, seed=0):
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([np.arange(min(N, 64)), np.arange(max(0, N - 64), N),
                                     rng.integers(0, N, size=n)]))
    return rows


# ---- configuration 1: exact, N=4096, M=256, k=32, fp32 N(0,1) seed 0 ---------------------
def test_config1_exact_bit_identical():
    x = synth.normal_f32(4096, 256, seed=0)
    v, i, ov, oi = _check_full(x, 32, what="config1")
    _, si = oracle.sort_topk(x, 32)
    np.testing.assert_array_equal(i.cpu().numpy(), si)


# ---- configuration 2: MaxK-shaped, N=262144, exact and max_iter in {2,3,4,5,8} ------------
def test_config2_exact_and_early_stop():
    x = synth.normal_f32(262144, 256, seed=0)
    _, ie, ove, oie = _check_full(x, 32, what="config2 exact")
    for m in (2, 3, 4, 5, 8):
        v, i, _, _ = _check_full(x, 32, max_iter=m, what=f"config2 max_iter={m}")
        acc = accuracy.compare(vals_np(v).view(np.float32), i.cpu().numpy(), ove, oie)
        assert acc["r_max_worst"] == 0.0
        print(f"max_iter={m}: {acc}")


# ---- configuration 3: shape sweep (reduced N, every combination) -----------------------
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("M", [128, 256, 512, 1024])
def test_config3_sweep_reduced(M, dtype):
    x = synth.make("normal", 2048, M, seed=0, dtype=dtype)
    for k in (16, 32, 64, 128, 256):
        if k >= M:
            continue
        for eps in (0.0, 1e-4, 1e-2):
            for m in (-1, 2):
                _check_full(x, k, m, eps, what=f"sweep M={M} k={k} {dtype} eps={eps} max_iter={m}")


@pytest.mark.parametrize("N", [1 << 16, 1 << 18, 1 << 20])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_config3_full_rows(N, dtype):
    """The sweep's full batch sizes at M = 256, k = 32, compared on every row:
    exact with pass counts, the default call (no pass counts: the packed
    search), max_iter = 2 and eps = 1e-2."""
    M, k = 256, 32
    x = synth.make("normal", N, M, seed=0, dtype=dtype)
    xt = to_dev(x)
    for m, eps in ((-1, 0.0), (2, 0.0), (-1, 1e-2)):
        v, i, it, st = api.rtopk_select_stats(xt, k, m, eps)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        ov, oi, oit = oracle_rows(oracle.replay, x, k, m, eps)
        assert_same_selection(v, i, ov, oi, what=f"N={N} {dtype} max_iter={m} eps={eps}")
        np.testing.assert_array_equal(it.cpu().numpy(), oit)
        if m < 0 and eps == 0.0:
            v, i = api.rtopk_select(xt, k)
            torch.cuda.synchronize()
            assert_same_selection(v, i, ov, oi, what=f"N={N} {dtype} default path")


# ---- configuration 4: long rows, adversarial values ------------------------------------
@pytest.mark.parametrize("value_set", ["uniform", "int_ties", "all_equal", "outliers", "subnormal"])
@pytest.mark.parametrize("M", [2048, 4096, 8192])
def test_config4_long_rows_adversarial(M, value_set):
    """Every one of the 65,536 rows, k in {64, 256, 1024}, through both calls:
    rtopk_select_stats (binary32 search from [min, max], pass counts compared)
    and rtopk_select (no pass counts: the block kernel's raised lower end and
    its shared-list tail), each against the oracle's exact replay, which the
    pins tie to the definition."""
    N = 65536
    x = synth.make(value_set, N, M, seed=0)
    xt = to_dev(x)
    for k in (64, 256, 1024):
        ov, oi, oit = oracle_rows(oracle.replay, x, k)
        v, i, it, st = api.rtopk_select_stats(xt, k)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert_same_selection(v, i, ov, oi, what=f"M={M} {value_set} k={k} with pass counts")
        np.testing.assert_array_equal(it.cpu().numpy(), oit)
        v, i = api.rtopk_select(xt, k)
        torch.cuda.synchronize()
        assert_same_selection(v, i, ov, oi, what=f"M={M} {value_set} k={k} default path")
        del v, i, it, st
    rows = _sample_rows(N, 300)
    _, si = oracle.sort_topk(x[rows], 1024)
    np.testing.assert_array_equal(oi[rows], si)
    del xt
    torch.cuda.empty_cache()


# ---- configuration 5: fused MaxK layer, bf16 -> CBSR (int16) -> backward scatter ---------
def test_config5_maxk_forward_backward():
    N, M, k = 1 << 20, 256, 32
    xb = synth.normal_bf16(N, M, seed=0)
    xt = to_dev(xb)
    fv, fi = api.maxk_forward(xt, k)
    torch.cuda.synchronize()
    assert fi.dtype == torch.int16 and fv.dtype == torch.bfloat16
    # every row: values are the input at the kept indices, indices strictly ascending
    fil = fi.long()
    assert torch.equal(torch.gather(xt, 1, fil).view(torch.int16), fv.view(torch.int16))
    assert bool((fil[:, 1:] > fil[:, :-1]).all()) and int(fil.min()) >= 0 and int(fil.max()) < M
    ov, oi, _ = oracle_rows(oracle.replay, xb, k)
    assert_same_selection(fv, fi, ov, oi, what="maxk_forward")
    # backward over all rows against the oracle scatter
    dy = synth.normal_bf16(N, k, seed=1)
    g = api.maxk_backward_scatter(to_dev(dy), fi, M)
    torch.cuda.synchronize()
    want = oracle.maxk_backward(dy, fi.cpu().numpy(), M)
    np.testing.assert_array_equal(vals_np(g), want)


# ---- edge cases --------------------------------------------------------------------------
@pytest.mark.parametrize("M", [1, 2, 3, 5, 31, 33, 100, 129, 1000, 1023, 1024, 1025, 1500,
                               2047, 4095, 5000, 8191, 8192])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_edge_row_lengths(M, dtype):
    N = 300
    x = synth.make("int_ties" if M % 2 else "normal", N, M, seed=M, dtype=dtype)
    for k in sorted({1, max(1, M // 3), M}):
        for m in (-1, 0, 3):
            _check_full(x, k, m, what=f"M={M} {dtype} k={k} max_iter={m}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_misaligned_input_pointer(dtype):
    N, M, k = 257, 256, 32
    x = synth.make("normal", N, M + 1, seed=3, dtype=dtype)
    flat = to_dev(x).reshape(-1)
    xt = flat[1:1 + N * M].view(N, M)  # 4- or 2-byte offset: no 16-byte loads possible
    v, i, it, st = api.rtopk_select_stats(xt, k)
    torch.cuda.synchronize()
    host = x.reshape(-1)[1:1 + N * M].reshape(N, M)
    ov, oi, oit = oracle.replay(host, k)
    assert_same_selection(v, i, ov, oi, what="misaligned")
    np.testing.assert_array_equal(it.cpu().numpy(), oit)


def test_tiny_and_degenerate():
    for N in (1, 2, 7):
        x = synth.normal_f32(N, 256, seed=N)
        _check_full(x, 32, what=f"N={N}")
    x = synth.all_equal_rows_f32(100, 256, seed=1)
    _check_full(x, 32, what="all equal")
    x = synth.normal_f32(100, 256, seed=2)
    _check_full(x, 32, -1, 1e30, what="eps >= range")
    _check_full(x, 256, what="k == M")
    # N == 0 is a no-op
    v, i = api.rtopk_select(torch.empty((0, 256), device="cuda"), 32)
    assert v.shape == (0, 32)


def test_signed_zero_and_subnormal_bits():
    x = synth.subnormals_f32(512, 256, seed=5)
    x[:, ::7] = np.float32(-0.0)
    x[:, 3::11] = np.float32(0.0)
    _check_full(x, 40, what="zeros+subnormals")
    _check_full(x, 40, 5, what="zeros+subnormals early stop")


def test_status_word_flags_bad_rows():
    x = synth.normal_f32(64, 256, seed=0)
    x[3, 10] = np.nan
    x[9, 0] = np.inf
    x[20, 5] = np.float32(3e38)
    v, i, it, st = _run(x, 32)
    assert st & 0x1 and st & 0x2 and not st & 0x4
    # the host reader returns the same bits (RTOPK_EDEVICE underneath)
    xt = to_dev(x)
    word = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.rtopk_select_stats(xt, 32, status=word)
    assert api.read_status(word) == st
    clean = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.rtopk_select_stats(to_dev(synth.normal_f32(64, 256, seed=1)), 32, status=clean)
    assert api.read_status(clean) == 0
    good = np.setdiff1d(np.arange(64), [3, 9, 20])
    ov, oi, _ = oracle.replay(x[good], 32)
    assert_same_selection(v, i, ov, oi, rows=good, what="good rows beside bad ones")


def test_backward_bad_index_flag_and_edges():
    N, M, k = 40, 100, 10
    dy = synth.normal_bf16(N, k, seed=1)
    idx = np.tile(np.arange(0, 3 * k, 3, dtype=np.int16), (N, 1))
    idx[5, 2] = 100  # out of range
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = api.maxk_backward_scatter(to_dev(dy), torch.from_numpy(idx).cuda(), M, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 0x8
    ok = np.setdiff1d(np.arange(N), [5])
    want = oracle.maxk_backward(dy[ok], idx[ok], M)
    np.testing.assert_array_equal(vals_np(g)[ok], want)
    for M2 in (1, 7, 8, 8192):
        k2 = min(4, M2)
        dy2 = synth.normal_bf16(9, k2, seed=2)
        idx2 = np.tile(np.arange(k2, dtype=np.int16) * (M2 // k2), (9, 1))
        g2 = api.maxk_backward_scatter(to_dev(dy2), torch.from_numpy(idx2).cuda(), M2)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(vals_np(g2), oracle.maxk_backward(dy2, idx2, M2))


def test_side_stream_and_determinism():
    x = synth.normal_f32(20000, 512, seed=4)
    xt = to_dev(x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        v1, i1 = api.rtopk_select(xt, 64)
    s.synchronize()
    v2, i2 = api.rtopk_select(xt, 64)
    torch.cuda.synchronize()
    assert torch.equal(i1, i2) and torch.equal(v1.view(torch.int32), v2.view(torch.int32))


def test_autograd_maxk_layer():
    x = synth.normal_bf16(512, 256, seed=0)
    xt = to_dev(x).requires_grad_(True)
    vals, idx = api.MaxK.apply(xt, 32)
    (vals.float() * 2).sum().backward()
    g = xt.grad
    ov, oi, _ = oracle.replay(x, 32)
    two = np.full((512, 32), 0x4000, dtype=np.uint16)  # bf16 2.0
    np.testing.assert_array_equal(vals_np(g), oracle.maxk_backward(two, oi.astype(np.int16), 256))


def test_pinned_host_buffers_zero_copy():
    """The kernels read and write pinned host memory in place (no staging copy)."""
    x = synth.normal_f32(5000, 256, seed=12)
    xh = torch.from_numpy(x).pin_memory()
    v, i = api.rtopk_select(xh, 32)
    torch.cuda.synchronize()
    assert not v.is_cuda and v.is_pinned() and i.is_pinned()
    ov, oi, _ = oracle.replay(x, 32)
    assert_same_selection(v.numpy().view(np.uint32), i.numpy(), ov, oi, what="pinned host")
    xb = synth.normal_bf16(3000, 256, seed=13)
    xbh = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).pin_memory()
    fv, fi = api.maxk_forward(xbh, 32)
    torch.cuda.synchronize()
    bv, bi, _ = oracle.replay(xb, 32)
    assert_same_selection(fv.view(torch.int16).numpy().view(np.uint16), fi.numpy(), bv, bi, what="pinned bf16")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("M,k,B", [(256, 32, 2), (256, 32, 4), (256, 32, 8), (256, 32, 32), (1024, 128, 8),
                                   (4096, 64, 4), (120, 12, 3)])
def test_bucketed_topk(M, k, B, dtype):
    x = synth.make("normal", 3000, M, seed=B, dtype=dtype)
    for m in (-1, 2):
        v, i = api.rtopk_select_bucketed(to_dev(x), k, B, m)
        torch.cuda.synchronize()
        ov, oi = oracle.bucketed_topk(x, k, B, m)
        assert_same_selection(v, i, ov, oi, what=f"bucketed M={M} k={k} B={B} {dtype} max_iter={m}")


@pytest.mark.parametrize("value_set", ["normal", "int_ties", "subnormal", "uniform"])
@pytest.mark.parametrize("M", [256, 512, 1000])
def test_bf16_search_stops_once_kept_set_is_final(value_set, M):
    """bf16 rows without pass counts requested stop as soon as [lo, hi) holds a
    single bf16 value; the kept set must equal the full replay's in every mode."""
    x = synth.make(value_set, 3000, M, seed=M, dtype="bf16")
    xt = to_dev(x)
    for k in (1, 32, M // 4):
        for m, eps in ((-1, 0.0), (3, 0.0), (12, 0.0), (-1, 1e-3)):
            v, i = api.rtopk_select(xt, k, m, eps)
            torch.cuda.synchronize()
            ov, oi, _ = oracle.replay(x, k, m, eps)
            assert_same_selection(v, i, ov, oi, what=f"bf16 stop {value_set} M={M} k={k} max_iter={m} eps={eps}")
        fv, fi = api.maxk_forward(xt, k)
        torch.cuda.synchronize()
        ov, oi, _ = oracle.replay(x, k)
        assert_same_selection(fv, fi, ov, oi, what=f"maxk_forward stop {value_set} M={M} k={k}")


# ---- exact mode without pass counts: the search may start from a tighter lower end --------
@pytest.mark.parametrize("value_set", ["normal", "uniform", "int_ties", "all_equal", "outliers", "subnormal"])
@pytest.mark.parametrize("M", [64, 100, 256, 1024, 3000, 8192, 20000])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_exact_without_pass_counts_is_the_definition(value_set, M, dtype):
    """rtopk_select in exact mode (no pass counts requested) against the
    definition of exact top-k, ties to the lowest index, over every kernel
    family (rows per warp, warp, block, cluster) and the tie-heavy sets."""
    N = 300 if M <= 8192 else 64
    x = synth.make(value_set, N, M, seed=M + 7, dtype=dtype)
    xt = to_dev(x)
    for k in sorted({1, 5, 16, 32, 33, 64, min(M, 200)}):
        v, i = api.rtopk_select(xt, k)
        torch.cuda.synchronize()
        ov, oi = oracle.sort_topk(x, k)
        assert_same_selection(v, i, ov, oi, what=f"{value_set} M={M} {dtype} k={k}")


# ---- rows beyond the pages' 8192-element limit: one CTA cluster per row -------------------
@pytest.mark.parametrize("M", [8193, 12000, 16384, 16385, 32768, 40000, 65536])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_cluster_rows(M, dtype):
    N = 150
    x = synth.make("int_ties" if M % 2 else "normal", N, M, seed=M, dtype=dtype)
    for k in (1, 64, 1000, M // 2):
        for m in (-1, 4):
            _check_full(x, k, m, what=f"cluster M={M} {dtype} k={k} max_iter={m}")


@pytest.mark.parametrize("value_set", ["all_equal", "outliers", "uniform"])
def test_cluster_rows_adversarial(value_set):
    N, M = 100, 20000
    x = synth.make(value_set, N, M, seed=5)
    for k in (3, 256, 5000):
        _check_full(x, k, what=f"cluster {value_set} k={k}")
        _check_full(x, k, 0, 1e-3, what=f"cluster {value_set} k={k} eps")


def test_cluster_rows_status_and_neighbours():
    """Non-finite and out-of-range rows in the cluster path set their status
    bits and leave the other rows of the same launch exact."""
    N, M, k = 24, 20000, 100
    x = synth.normal_f32(N, M, seed=9)
    x[2, 17] = np.nan
    x[7, 19999] = -np.inf
    x[11, 4000] = np.float32(2e38)
    v, i, it, st = _run(x, k)
    assert st & 0x1 and st & 0x2 and not st & 0x4
    good = np.setdiff1d(np.arange(N), [2, 7, 11])
    ov, oi, oit = oracle.replay(x[good], k)
    assert_same_selection(v, i, ov, oi, rows=good, what="cluster good rows beside bad ones")
    np.testing.assert_array_equal(it[good], oit)


def test_binding_rejects_bad_outputs():
    """Caller-supplied outputs of the wrong shape, dtype or layout are refused
    before any launch; a correct one is written in place."""
    x = to_dev(synth.normal_f32(64, 256, seed=3))
    with pytest.raises(ValueError):
        api.rtopk_select(x, 32, vals=torch.empty((64, 31), device="cuda"))
    with pytest.raises(ValueError):
        api.rtopk_select(x, 32, idx=torch.empty((64, 32), dtype=torch.int64, device="cuda"))
    with pytest.raises(ValueError):
        api.rtopk_select(x, 32, vals=torch.empty((32, 64), device="cuda").t())
    with pytest.raises(ValueError):
        api.maxk_backward_scatter(torch.zeros((4, 2), dtype=torch.bfloat16, device="cuda"),
                                  torch.zeros((4, 2), dtype=torch.int16, device="cuda"), 8,
                                  grad=torch.empty((4, 7), dtype=torch.bfloat16, device="cuda"))
    v = torch.empty((64, 32), device="cuda")
    i = torch.empty((64, 32), dtype=torch.int32, device="cuda")
    v2, i2 = api.rtopk_select(x, 32, vals=v, idx=i)
    torch.cuda.synchronize()
    assert v2.data_ptr() == v.data_ptr() and i2.data_ptr() == i.data_ptr()
    ov, oi, _ = oracle.replay(x.cpu().numpy(), 32)
    assert_same_selection(v, i, ov, oi, what="caller-supplied outputs")


@pytest.mark.parametrize("M,k", [(256, 32), (256, 16), (512, 64), (128, 8), (2048, 256), (64, 12), (1024, 40)])
def test_backward_group_shapes(M, k):
    """The backward scatter's row groups: partial last group, 16-byte and
    2-byte pair loads, a bad index in the last group (flagged, skipped, the
    rest of the output exact)."""
    N = 8 * 3 + 5
    rng = np.random.default_rng(M + k)
    idx = np.sort(np.stack([rng.choice(M, size=k, replace=False) for _ in range(N)]), axis=1).astype(np.int16)
    dy = synth.normal_bf16(N, k, seed=7)
    g = api.maxk_backward_scatter(to_dev(dy), torch.from_numpy(idx).cuda(), M)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(vals_np(g), oracle.maxk_backward(dy, idx, M))
    bad = idx.copy()
    bad[N - 2, k // 2] = M + 3  # out of range
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = api.maxk_backward_scatter(to_dev(dy), torch.from_numpy(bad).cuda(), M, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 0x8
    ok = np.setdiff1d(np.arange(N), [N - 2])
    np.testing.assert_array_equal(vals_np(g)[ok], oracle.maxk_backward(dy[ok], idx[ok], M))


@pytest.mark.parametrize("value_set", ["normal", "int_ties", "dense_bucket", "subnormal", "all_equal",
                                       "wide_range", "signed_zeros"])
@pytest.mark.parametrize("dtype,M", [("f32", 128), ("f32", 256), ("f32", 384), ("f32", 512),
                                     ("bf16", 128), ("bf16", 256), ("bf16", 512)])
def test_bucketed_exact_side_by_side_buckets(value_set, dtype, M):
    """Exact bucketed top-k where one warp searches all buckets of a row side
    by side (B in {2, 4, 8}): every row against the oracle, on value sets that
    make buckets collapse (ties, rows inside one 16-bit bucket) so the
    bucket-by-bucket binary32 finish runs too."""
    N = 500
    x = synth.make(value_set, N, M, seed=M + 3, dtype=dtype)
    xt = to_dev(x)
    for B in (2, 4, 8):
        for k in sorted({B, 4 * B, 8 * B, 16 * B, 32 * B}):
            if k > M or k > 256:
                continue
            v, i = api.rtopk_select_bucketed(xt, k, B)
            torch.cuda.synchronize()
            ov, oi = oracle.bucketed_topk(x, k, B)
            assert_same_selection(v, i, ov, oi, what=f"bucketed {value_set} {dtype} M={M} B={B} k={k}")


@pytest.mark.parametrize("M", [128, 256, 384, 512])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("value_set", ["normal", "int_ties", "all_equal", "signed_zeros", "wide_range"])
def test_bucketed_one_or_two_per_bucket(value_set, dtype, M):
    """Exact bucketed top-k where each bucket keeps one or two elements
    (k / B <= 2, B in {2, ..., 32}: per-lane best elements merged by shuffles,
    no search): every row against the oracle, on value sets full of ties so
    the lowest-index rule decides most buckets; 501 rows leave a ragged tail."""
    if dtype == "bf16" and M == 384:
        pytest.skip("bf16 rows of 384 are not a full-row shape of the lean kernel")
    N = 501
    x = synth.make(value_set, N, M, seed=M + 5, dtype=dtype)
    xt = to_dev(x)
    for B in (2, 4, 8, 16, 32):
        for k in (B, 2 * B):
            if M % B:
                continue
            v, i = api.rtopk_select_bucketed(xt, k, B)
            torch.cuda.synchronize()
            ov, oi = oracle.bucketed_topk(x, k, B)
            assert_same_selection(v, i, ov, oi, what=f"bucketed small {value_set} {dtype} M={M} B={B} k={k}")


@pytest.mark.parametrize("M", [2048, 4096, 8192])
@pytest.mark.parametrize("value_set", ["normal", "int_ties", "dense_bucket", "signed_zeros", "wide_range"])
def test_long_rows_default_path_bf16_and_maxk_forward(M, value_set):
    """Exact rows of 2048 / 4096 / 8192 without pass counts (a team of 2 / 4 /
    8 warps per row, 16-bit images): bf16 through rtopk_select (int32
    indices) and maxk_forward (int16 indices), every row against the oracle,
    k up to 1024; 301 rows leave a ragged last block of teams."""
    N = 301
    xb = synth.make(value_set, N, M, seed=M + 11, dtype="bf16")
    xt = to_dev(xb)
    for k in (1, 33, 64, 256, 1024):
        ov, oi, _ = oracle_rows(oracle.replay, xb, k)
        v, i = api.rtopk_select(xt, k)
        fv, fi = api.maxk_forward(xt, k)
        torch.cuda.synchronize()
        assert_same_selection(v, i, ov, oi, what=f"bf16 M={M} {value_set} k={k}")
        assert_same_selection(fv, fi, ov, oi, what=f"maxk_forward M={M} {value_set} k={k}")
    xf = synth.make(value_set, N, M, seed=M + 12)
    xft = to_dev(xf)
    for k in (1, 33, 64, 256, 1024):
        ov, oi, _ = oracle_rows(oracle.replay, xf, k)
        v, i = api.rtopk_select(xft, k)
        torch.cuda.synchronize()
        assert_same_selection(v, i, ov, oi, what=f"f32 M={M} {value_set} k={k}")


def _saturating_rows(case, N, M, seed):
    """fp32 rows whose binary16 images saturate at +-65504 in bulk: half of the
    entries +-1e30; 90% at -1e30 with 2% at +1e30; or values around the
    binary16 rounding boundary (65488 rounds to 65472, above it to 65504)."""
    g = np.random.default_rng(seed)
    x = g.standard_normal((N, M)).astype(np.float32)
    u = g.random((N, M))
    if case == "half_outliers":
        x = np.where(u < 0.25, np.float32(1e30), np.where(u < 0.5, np.float32(-1e30), x))
    elif case == "mostly_negative":
        x = np.where(u < 0.9, np.float32(-1e30), np.where(u < 0.92, np.float32(1e30), x))
    else:
        pool = np.array([65472.0, 65487.99, 65488.0, 65488.01, 65504.0, 65520.0, 1e30], dtype=np.float32)
        pick = pool[g.integers(0, pool.size, size=(N, M))]
        sign = np.where(g.random((N, M)) < 0.5, np.float32(-1), np.float32(1))
        x = np.where(u < 0.6, pick * sign, x * np.float32(1000))
    return np.ascontiguousarray(x.astype(np.float32))


@pytest.mark.parametrize("case", ["half_outliers", "mostly_negative", "boundary"])
@pytest.mark.parametrize("M", [2048, 4096, 8192])
def test_long_rows_saturated_images(M, case):
    """Exact rows of 2048 / 4096 / 8192 whose 16-bit images saturate in bulk:
    the bracket starts from the counts at +-65504 and the extremes of the other
    images (all three branches: C(65504) >= k, a lower end above -65504, and
    -65504 itself), every row against the definition, k on both sides of the
    team's thread count."""
    N = 97
    x = _saturating_rows(case, N, M, seed=M + len(case))
    xt = to_dev(x)
    for k in (1, 64, 200, 1024):
        v, i = api.rtopk_select(xt, k)
        torch.cuda.synchronize()
        ov, oi = oracle.sort_topk(x, k)
        assert_same_selection(v, i, ov, oi, what=f"saturated {case} M={M} k={k}")


@pytest.mark.parametrize("M,dtype", [(1024, "f32"), (512, "bf16"), (1024, "bf16"), (2048, "f32"), (4096, "bf16"),
                                     (8192, "f32"), (16384, "f32")])
def test_guessed_probes_under_shifting_row_scales(M, dtype):
    """Exact mode without pass counts probes guessed thresholds (the previous
    row's, then Newton or interpolation steps with a density carried over
    rows). Consecutive rows here differ in scale by up to 10^6 and in sign, so
    the carried guesses and densities are wrong by orders of magnitude: every
    row must still be the definition (a guess only ever replaces a midpoint
    strictly inside the bracket)."""
    N = 203
    g = np.random.default_rng(M + 17)
    base = g.standard_normal((N, M)).astype(np.float32)
    scale = np.array([1e-3, 1.0, 1e3, -1.0, 3e-3, -1e3, 0.5], dtype=np.float32)[np.arange(N) % 7]
    x = base * scale[:, None]
    if dtype == "bf16":
        x = synth.f32_to_bf16_bits(x)
    xt = to_dev(x)
    for k in (33, 64, 256, 1000):
        if k > M:
            continue
        v, i = api.rtopk_select(xt, k)
        torch.cuda.synchronize()
        ov, oi = oracle.sort_topk(x, k)
        assert_same_selection(v, i, ov, oi, what=f"shifting scales M={M} {dtype} k={k}")


@pytest.mark.parametrize("M", [128, 256, 512, 1024, 2048, 3000])
@pytest.mark.parametrize("value_set", ["normal", "int_ties", "signed_zeros"])
def test_maxk_forward_early_stop_and_eps(M, value_set):
    """maxk_forward (bf16 in, int16 indices) with early stop and eps follows the
    pages' trajectory like rtopk_select: every row against the oracle's replay
    (the replay kernel on full rows of 128..1024, the binary32 kernels
    elsewhere), values and indices."""
    N = 777
    x = synth.make(value_set, N, M, seed=M + 29, dtype="bf16")
    xt = to_dev(x)
    for k in (1, 32, min(M, 200)):
        for m, eps in ((0, 0.0), (2, 0.0), (5, 0.0), (-1, 1e-2), (3, 1e-3)):
            fv, fi = api.maxk_forward(xt, k, m, eps)
            torch.cuda.synchronize()
            ov, oi, _ = oracle.replay(x, k, m, eps)
            assert_same_selection(fv, fi, ov, oi, what=f"maxk_forward {value_set} M={M} k={k} max_iter={m} eps={eps}")
