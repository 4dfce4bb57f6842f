"""The C ABI without a GPU: the library builds, exports every symbol that
include/rtopk.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    with open(os.path.join(ROOT, "include", "rtopk.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from maxk_sparse_activations_gb300 import _lib
    return _lib.load()


def test_header_declares_the_entry_points():
    names = _declared_functions()
    from maxk_sparse_activations_gb300 import _lib
    assert set(_lib.EXPORTED) <= set(names)
    assert {"rtopk_select", "rtopk_select_stats", "maxk_forward", "maxk_backward_scatter"} <= set(names)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_strerror_and_version(lib):
    from maxk_sparse_activations_gb300 import _lib
    assert _lib.strerror(0) == "ok"
    default = _lib.strerror(-99)
    assert "unknown rtopk status" in default
    texts = {_lib.strerror(code) for code in (-1, -2, -3, -4, -5, -6)}
    assert len(texts) == 6 and default not in texts
    assert lib.rtopk_version() >= 100


def test_argument_errors_launch_nothing(lib):
    # every call below must return before any CUDA call (no GPU here)
    S = lambda *a: lib.rtopk_select(*a)
    assert S(None, 10, 0, 1, -1, 0.0, 0, None, None, None) == -1          # M < 1
    assert S(None, 10, 65537, 1, -1, 0.0, 0, None, None, None) == -1      # M > 65536
    assert S(None, 10, 8193, 1, -1, 0.0, 0, None, None, None) == -3       # long rows accepted: NULL pointers
    assert lib.maxk_forward(None, 10, 8193, 1, -1, 0.0, None, None, None) == -1  # maxk_forward: M <= 8192
    Bk = lib.rtopk_select_bucketed
    assert Bk(None, 10, 16384, 32, 2, -1, 0.0, 0, None, None, None) == -1  # bucketed: M <= 8192
    assert S(None, -1, 8, 1, -1, 0.0, 0, None, None, None) == -1          # N < 0
    assert S(None, 10, 8, 0, -1, 0.0, 0, None, None, None) == -2          # k < 1
    assert S(None, 10, 8, 9, -1, 0.0, 0, None, None, None) == -2          # k > M
    assert S(None, 10, 8, 2, -1, 0.0, 0, None, None, None) == -3          # NULL pointers
    assert S(None, 10, 8, 2, -1, 0.0, 7, None, None, None) == -4          # dtype
    assert S(None, 10, 8, 2, -1, -1.0, 0, None, None, None) == -6         # eps < 0
    assert S(None, 10, 8, 2, -1, float("nan"), 0, None, None, None) == -6 # eps NaN
    assert S(None, 0, 8, 2, -1, 0.0, 0, None, None, None) == 0            # N == 0: no-op
    assert lib.maxk_forward(None, 5, 8, 9, -1, 0.0, None, None, None) == -2
    assert lib.maxk_forward(None, 0, 8, 2, -1, 0.0, None, None, None) == 0
    assert lib.maxk_backward_scatter(None, None, 5, 8, 2, None, None, None) == -3
    assert lib.maxk_backward_scatter(None, None, 5, 9000, 2, None, None, None) == -1
    assert lib.maxk_backward_scatter(None, None, 0, 8, 2, None, None, None) == 0
    Bk = lib.rtopk_select_bucketed
    assert Bk(None, 10, 256, 32, 3, -1, 0.0, 0, None, None, None) == -6   # 3 does not divide 256
    assert Bk(None, 10, 256, 30, 4, -1, 0.0, 0, None, None, None) == -6   # 4 does not divide 30
    assert Bk(None, 10, 256, 32, 4, -1, 0.0, 0, None, None, None) == -3   # NULL pointers
    assert Bk(None, 0, 256, 32, 4, -1, 0.0, 0, None, None, None) == 0
    F = lib.maxk_spgemm_forward
    assert F(None, None, None, -1, 4, None, None, 8, 2, None, None, None) == -1   # n_dst < 0
    assert F(None, None, None, 4, 4, None, None, 8, 9, None, None, None) == -2    # k > M
    assert F(None, None, None, 4, 4, None, None, 512, 300, None, None, None) == -2  # k > 256
    assert F(None, None, None, 4, 4, None, None, 8, 2, None, None, None) == -3    # NULL pointers
    assert F(None, None, None, 0, 4, None, None, 8, 2, None, None, None) == 0     # no rows
    B = lib.maxk_sspmm_backward
    assert B(None, None, None, 4, 4, None, None, 9000, 2, None, None, None) == -1  # M > 8192
    assert B(None, None, None, 4, 4, None, None, 8, 2, None, None, None) == -3
    assert B(None, None, None, 0, 4, None, None, 8, 2, None, None, None) == 0
    BS = lib.maxk_sspmm_backward_scatter
    assert BS(None, None, None, 4, 4, None, None, 9000, 2, None, None, None) == -1  # M > 8192
    assert BS(None, None, None, 4, 4, None, None, 8, 9, None, None, None) == -2     # k > M
    assert BS(None, None, None, 4, 4, None, None, 8, 2, None, None, None) == -3     # NULL pointers
    assert BS(None, None, None, 0, 4, None, None, 8, 2, None, None, None) == 0      # no rows


def test_status_read_arguments(lib):
    # a NULL word is an argument error, returned before any CUDA call
    assert lib.rtopk_status_read(None, None, None) == -3
    from maxk_sparse_activations_gb300 import _lib
    assert "status word" in _lib.strerror(-7)
