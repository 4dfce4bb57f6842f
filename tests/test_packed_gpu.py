"""GPU parity of exact mode without pass counts on rows of 128..1024 elements.

There the kernel runs its threshold search on packed 16-bit images of the row
(binary16 for fp32 rows, the data themselves for bf16 rows) and finishes in
binary32 only inside the last 16-bit bucket. The result must still be the
definition: the k largest values, ties at the k-th value to the lowest index
("RTop-K ..." summary, "Problem", "Approach") -- bit-exact values and indices
against the oracle, on value sets chosen to break a 16-bit image (magnitudes
beyond binary16's range and below its subnormals, rows inside one binary16
bucket, signed zeros, heavy ties, all-equal rows).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from maxk_sparse_activations_gb300 import _lib, api, synth

from gpu_util import assert_same_selection, oracle_rows, to_dev

pytestmark = pytest.mark.gpu

VALUE_SETS = ["normal", "uniform", "int_ties", "all_equal", "outliers", "subnormal", "wide_range",
              "dense_bucket", "negative", "signed_zeros"]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    oracle.build()


@pytest.mark.parametrize("value_set", VALUE_SETS)
@pytest.mark.parametrize("M", [128, 256, 384, 512, 768, 1024])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_packed_exact_is_the_definition(value_set, M, dtype):
    N = 400
    x = synth.make(value_set, N, M, seed=M + 31, dtype=dtype)
    xt = to_dev(x)
    for k in sorted({1, 5, 16, 31, 32, 33, 64, 100, M // 2, M - 1, M}):
        if k > 256:
            continue
        v, i = api.rtopk_select(xt, k)
        torch.cuda.synchronize()
        ov, oi = oracle.sort_topk(x, k)
        assert_same_selection(v, i, ov, oi, what=f"packed {value_set} M={M} {dtype} k={k}")
        if dtype == "bf16":
            fv, fi = api.maxk_forward(xt, k)
            torch.cuda.synchronize()
            assert_same_selection(fv, fi, ov, oi, what=f"maxk_forward {value_set} M={M} k={k}")


def test_packed_equals_binary32_path_on_the_same_rows():
    """The packed search (no pass counts) and the binary32 replay (pass counts
    requested) return the same CBSR rows on the same input."""
    for dtype in ("f32", "bf16"):
        x = synth.make("normal", 50000, 256, seed=77, dtype=dtype)
        xt = to_dev(x)
        v1, i1 = api.rtopk_select(xt, 32)
        v2, i2, _, st = api.rtopk_select_stats(xt, 32)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.equal(i1, i2)
        assert torch.equal(v1.view(torch.int16 if dtype == "bf16" else torch.int32),
                           v2.view(torch.int16 if dtype == "bf16" else torch.int32))


def test_packed_headline_size_every_row():
    """2^20 rows x 256 fp32, k = 32, in the launch the benchmark times: every
    row bit-exact against the oracle (values and indices, so the lowest-index
    tie rule at the k-th value is checked wherever it applies); the bf16 rows
    of the MaxK forward at the same size likewise."""
    N, M, k = 1 << 20, 256, 32
    x = synth.normal_f32(N, M, seed=0)
    xt = to_dev(x)
    v, i = api.rtopk_select(xt, k)
    torch.cuda.synchronize()
    ov, oi, _ = oracle_rows(oracle.replay, x, k)
    assert_same_selection(v, i, ov, oi, what="packed headline")
    del xt, v, i
    xb = synth.normal_bf16(N, M, seed=0)
    fv, fi = api.maxk_forward(to_dev(xb), k)
    torch.cuda.synchronize()
    ov, oi, _ = oracle_rows(oracle.replay, xb, k)
    assert_same_selection(fv, fi, ov, oi, what="packed maxk_forward")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_packed_status_word_flags_bad_rows(dtype):
    """Through the C ABI with pass counts not requested (iters = NULL) and a
    status word: rows with NaN, infinity or |x| > 1e38 set their bits, the
    other rows of the launch stay exact."""
    N, M, k = 64, 256, 32
    x = synth.normal_f32(N, M, seed=0)
    x[3, 10] = np.nan
    x[9, 0] = np.inf
    x[20, 5] = np.float32(3e38)
    xin = x if dtype == "f32" else synth.f32_to_bf16_bits(x)
    xt = to_dev(xin)
    vals = torch.empty((N, k), dtype=xt.dtype, device="cuda")
    idx = torch.empty((N, k), dtype=torch.int32, device="cuda")
    word = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib = _lib.load()
    rc = lib.rtopk_select_stats(xt.data_ptr(), N, M, k, -1, ctypes.c_float(0.0),
                                _lib.RTOPK_F32 if dtype == "f32" else _lib.RTOPK_BF16,
                                vals.data_ptr(), idx.data_ptr(), None, word.data_ptr(),
                                torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    st = int(word.item())
    assert st & 0x1 and st & 0x2 and not st & 0x4
    good = np.setdiff1d(np.arange(N), [3, 9, 20])
    ov, oi = oracle.sort_topk(xin[good], k)
    assert_same_selection(vals, idx, ov, oi, rows=good, what="packed good rows beside bad ones")
