"""The torch binding's checks of caller-supplied outputs, without a GPU: a
wrong shape, dtype or layout is rejected before the C ABI is called (the
kernels write every element of the expected shape, so a smaller or strided
tensor would take writes past its storage)."""
import pytest
import torch

from maxk_sparse_activations_gb300 import api


def test_output_shape_dtype_and_layout_are_checked():
    x = torch.empty((8, 16))
    with pytest.raises(ValueError, match="shape"):
        api._check_out(torch.empty((8, 3)), (8, 4), torch.float32, x, "vals")
    with pytest.raises(ValueError, match="dtype"):
        api._check_out(torch.empty((8, 4), dtype=torch.float64), (8, 4), torch.float32, x, "vals")
    with pytest.raises(ValueError, match="contiguous"):
        api._check_out(torch.empty((4, 8)).t(), (8, 4), torch.float32, x, "vals")
    # a plain (unpinned) host tensor is not memory the kernels may address
    with pytest.raises(ValueError, match="device"):
        api._check_out(torch.empty((8, 4)), (8, 4), torch.float32, x, "vals")
    with pytest.raises(ValueError, match="status"):
        api._check_status(torch.empty((2,), dtype=torch.int32), x)
    with pytest.raises(ValueError, match="status"):
        api._check_status(torch.empty((1,), dtype=torch.float32), x)


def test_inputs_must_be_addressable_by_the_gpu():
    with pytest.raises(ValueError, match="CUDA tensor or a pinned host tensor"):
        api.rtopk_select(torch.empty((8, 16)), 4)
