"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Sources: "RTop-K: Ultra-Fast Row-Wise Top-K Selection for Neural Network
Acceleration on GPUs" (summary page: "Problem", "Approach", "Key results",
"Surprising findings") and "MaxK-GNN: Extremely Fast GPU Kernel Design for
Accelerating Graph Neural Networks Training" ("One layer, one epoch, on Reddit",
"Asymmetric passes, one mask").

What pins what:
* brute force over all k-subsets (tiny rows)      -> the sort definition;
* exact-mode replay == sort definition            -> the search + fill pass;
* hand-worked rows in tests/golden/                -> early stop, eps, ties, collapse;
* max_iter = 0 closed form, eps >= range           -> fill pass without search;
* capped runs are prefixes of the uncapped search  -> what max_iter counts;
* torch.topk value multiset                        -> an independent library routine;
* the pages' printed statistics (hit rate > 80% for k >= 64 at 4 iterations,
  the exact search ends after few passes on most rows, the pivot search takes
  fewer than ten on normal features).
"""
import json
import os

import numpy as np
import pytest

from maxk_sparse_activations_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def _bits_to_f32(hexes):
    return np.array([int(h, 16) for h in hexes], dtype=np.uint32).view(np.float32)


def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["pins"])
def test_hand_worked_examples(oracle_mod, case):
    if "x_bits_f32" in case:
        x = _bits_to_f32(case["x_bits_f32"])[None, :]
    else:
        x = np.array([case["x"]], dtype=np.float32)
    vals, idx, iters = oracle_mod.replay(x, case["k"], case["max_iter"], case["eps"])
    assert idx[0].tolist() == case["idx"]
    assert int(iters[0]) == case["iters"]
    if "vals_bits_f32" in case:
        assert vals[0].view(np.uint32).tolist() == [int(h, 16) for h in case["vals_bits_f32"]]
    else:
        assert vals[0].tolist() == case["vals"]
    if case["max_iter"] < 0 and case["eps"] == 0.0:
        _, sidx = oracle_mod.sort_topk(x, case["k"])
        assert sidx[0].tolist() == case["idx"]


def test_hand_worked_accuracy():
    from maxk_sparse_activations_gb300 import accuracy
    case = [c for c in _golden_cases() if "accuracy" in c][0]
    exact = [c for c in _golden_cases() if c.get("x") == case["x"] and c["max_iter"] < 0 and c["eps"] == 0][0]
    acc = accuracy.compare(np.array([case["vals"]], np.float32), np.array([case["idx"]]),
                           np.array([exact["vals"]], np.float32), np.array([exact["idx"]]))
    for key in ("hit_rate", "r_max", "r_min"):
        assert acc[key + "_mean"] == pytest.approx(case["accuracy"][key], abs=0)


def _tiny_rows(rng, n, M, kind):
    if kind == "ints":
        return rng.integers(0, 4, size=(n, M)).astype(np.float32)
    if kind == "signed_zero":
        return rng.choice(np.array([-0.0, 0.0, -1.0, 1.0], np.float32), size=(n, M))
    return rng.standard_normal((n, M), dtype=np.float32)


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 10])
@pytest.mark.parametrize("kind", ["ints", "normal", "signed_zero"])
def test_sort_definition_matches_brute_force(oracle_mod, M, kind):
    rng = np.random.default_rng(1000 + M)
    x = _tiny_rows(rng, 60, M, kind)
    for k in range(1, M + 1):
        _, a = oracle_mod.sort_topk(x, k)
        _, b = oracle_mod.brute_topk(x, k)
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("kind", ["ints", "normal", "signed_zero"])
def test_exact_replay_equals_definition_small(oracle_mod, kind):
    rng = np.random.default_rng(7)
    for M in (1, 2, 3, 7, 16, 33):
        x = _tiny_rows(rng, 300, M, kind)
        for k in sorted({kk for kk in (1, 2, max(1, M // 2), M) if kk <= M}):
            v1, i1, _ = oracle_mod.replay(x, k, -1, 0.0)
            v2, i2 = oracle_mod.sort_topk(x, k)
            np.testing.assert_array_equal(i1, i2)
            np.testing.assert_array_equal(v1.view(np.uint32), v2.view(np.uint32))


@pytest.mark.parametrize("value_set", list(synth.VALUE_SETS))
@pytest.mark.parametrize("M,k", [(256, 32), (300, 17), (1024, 256), (2048, 64)])
def test_exact_replay_equals_definition_value_sets(oracle_mod, value_set, M, k):
    x = synth.make(value_set, 64, M, seed=3)
    v1, i1, it = oracle_mod.replay(x, k, -1, 0.0)
    v2, i2 = oracle_mod.sort_topk(x, k)
    np.testing.assert_array_equal(i1, i2)
    np.testing.assert_array_equal(v1.view(np.uint32), v2.view(np.uint32))
    # a binary32 bisection over [min, max] halves a range of at most 2e38 down to
    # the smallest spacing 2^-149: fewer than 300 passes
    assert it.max() < 300


def test_invariants_exact(oracle_mod):
    x = synth.make("int_ties", 200, 64, seed=5)
    k = 20
    vals, idx, _ = oracle_mod.replay(x, k)
    for r in range(x.shape[0]):
        row, kept = x[r], idx[r]
        assert np.all(np.diff(kept) > 0) and kept[0] >= 0 and kept[-1] < x.shape[1]
        np.testing.assert_array_equal(vals[r], row[kept])
        dropped = np.setdiff1d(np.arange(x.shape[1]), kept)
        if dropped.size:
            assert row[kept].min() >= row[dropped].max()
            kth = row[kept].min()
            tie_drop = dropped[row[dropped] == kth]
            tie_keep = kept[row[kept] == kth]
            if tie_drop.size:
                assert tie_keep.max() < tie_drop.min()


def test_torch_topk_value_multiset(oracle_mod):
    torch = pytest.importorskip("torch")
    for vs in ("normal", "int_ties", "subnormal", "outliers"):
        x = synth.make(vs, 128, 512, seed=11)
        for k in (1, 32, 200):
            vals, _ = oracle_mod.sort_topk(x, k)
            tv, _ = torch.topk(torch.from_numpy(x), k, dim=1, largest=True, sorted=True)
            a = np.sort(vals.astype(np.float64), axis=1)
            b = np.sort(tv.numpy().astype(np.float64), axis=1)
            np.testing.assert_array_equal(a, b)


def _closed_form_no_search(row, k):
    """max_iter = 0: keep the maximum's ties and fill the rest lowest index first."""
    mx = row.max()
    ties = np.flatnonzero(row >= mx)
    if ties.size >= k:
        return ties[:k]
    others = np.flatnonzero(row < mx)[: k - ties.size]
    return np.sort(np.concatenate([ties, others]))


@pytest.mark.parametrize("value_set", ["normal", "int_ties", "uniform"])
def test_max_iter_zero_and_large_eps_closed_form(oracle_mod, value_set):
    x = synth.make(value_set, 100, 96, seed=9)
    for k in (1, 5, 48, 96):
        _, i0, it0 = oracle_mod.replay(x, k, 0, 0.0)
        big_eps = float(np.float32((x.max() - x.min()) * 2))
        _, ie, ite = oracle_mod.replay(x, k, -1, big_eps)
        assert np.all(it0 == 0) and np.all(ite == 0)
        for r in range(x.shape[0]):
            want = _closed_form_no_search(x[r], k)
            assert i0[r].tolist() == want.tolist()
            assert ie[r].tolist() == want.tolist()


def test_capped_search_is_prefix(oracle_mod):
    x = synth.make("normal", 400, 256, seed=2)
    k = 32
    _, iex, itex = oracle_mod.replay(x, k, -1, 0.0)
    for m in (1, 2, 3, 5, 8, 12):
        _, im, itm = oracle_mod.replay(x, k, m, 0.0)
        np.testing.assert_array_equal(itm, np.minimum(itex, m))
        done = itex <= m
        np.testing.assert_array_equal(im[done], iex[done])
    # eps only ever stops earlier
    for eps in (1e-4, 1e-2, 0.5):
        _, _, ite = oracle_mod.replay(x, k, -1, eps)
        assert np.all(ite <= itex)


def test_pages_iteration_statistics(oracle_mod):
    """The exact search ends after a small, bounded number of passes on most rows
    (at most 16 on nearly all N(0,1) rows); the pivot search of normal features
    takes fewer than ten passes at the median."""
    x = synth.normal_f32(4000, 256, seed=0)
    _, _, it = oracle_mod.replay(x, 32, -1, 0.0)
    assert np.mean(it <= 16) > 0.9
    assert np.median(it) < 10


@pytest.mark.parametrize("k", [64, 128])
def test_pages_hit_rate_claim(oracle_mod, k):
    """For k >= 64, four iterations give hit rates above 80% (normal synthetic rows)."""
    from maxk_sparse_activations_gb300 import accuracy
    x = synth.normal_f32(4000, 256, seed=0)
    ve, ie, _ = oracle_mod.replay(x, k, -1, 0.0)
    va, ia, _ = oracle_mod.replay(x, k, 4, 0.0)
    acc = accuracy.compare(va, ia, ve, ie)
    assert acc["hit_rate_mean"] > 0.8
    assert acc["r_max_worst"] == 0.0  # the row maximum is always kept


def test_bf16_widening_matches_torch(oracle_mod):
    torch = pytest.importorskip("torch")
    bits = synth.normal_bf16(64, 256, seed=4)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(oracle_mod.widen_bf16(bits).view(np.uint32), t.view(np.uint32))


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = np.concatenate([synth.normal_f32(16, 256, seed=6).ravel(),
                        synth.subnormals_f32(4, 256, seed=6).ravel(),
                        synth.outliers_f32(4, 256, seed=6).ravel()])
    mine = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(mine, ref)


def test_bf16_replay_uses_widened_values(oracle_mod):
    bits = synth.normal_bf16(50, 256, seed=8)
    vals, idx, _ = oracle_mod.replay(bits, 32)
    _, idx_f = oracle_mod.sort_topk(oracle_mod.widen_bf16(bits), 32)
    np.testing.assert_array_equal(idx, idx_f)
    np.testing.assert_array_equal(vals, np.take_along_axis(bits, idx.astype(np.int64), 1))


def test_backward_scatter_properties(oracle_mod):
    fwd = synth.normal_bf16(64, 256, seed=0)
    _, idx, _ = oracle_mod.replay(fwd, 32)
    dy = synth.normal_bf16(64, 32, seed=1)
    g = oracle_mod.maxk_backward(dy, idx.astype(np.int16), 256)
    np.testing.assert_array_equal(np.take_along_axis(g, idx.astype(np.int64), 1), dy)
    mask = np.zeros_like(g, dtype=bool)
    np.put_along_axis(mask, idx.astype(np.int64), True, 1)
    assert np.all(g[~mask] == 0)


def test_rejects_invalid_rows(oracle_mod):
    for bad in (np.nan, np.inf, -np.inf, 2e38):
        x = np.zeros((1, 8), np.float32)
        x[0, 3] = bad
        with pytest.raises(ValueError):
            oracle_mod.replay(x, 2)


def test_bucketed_reduces_to_exact_and_argmax(oracle_mod):
    """Bucketed top-k ("Approximate Top-k for Increased Parallelism"): one bucket
    is the plain selection; k buckets keep each bucket's maximum, first
    occurrence (numpy argmax)."""
    x = synth.make("int_ties", 300, 256, seed=17)
    v1, i1 = oracle_mod.bucketed_topk(x, 32, 1)
    v0, i0, _ = oracle_mod.replay(x, 32)
    np.testing.assert_array_equal(i1, i0)
    _, ik = oracle_mod.bucketed_topk(x, 32, 32)
    want = np.argmax(x.reshape(300, 32, 8), axis=2) + np.arange(32) * 8
    np.testing.assert_array_equal(ik, want)
    v4, i4 = oracle_mod.bucketed_topk(synth.normal_f32(200, 256, seed=3), 32, 4)
    assert np.all(np.diff(i4, axis=1) > 0)
    assert np.all((i4 // 64) == np.repeat(np.arange(4), 8)[None, :])
