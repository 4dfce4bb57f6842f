"""Row-wise top-k (RTop-K) and the MaxK sparse-activation layer on GB300 (sm_103a).

The compute path is librtopk.so (hand-written CUDA kernels behind a C ABI, see
include/rtopk.h); ``api`` is its thin torch binding. Submodules load lazily so
that the input generators and host-side reporting import without a GPU.
"""

__all__ = ["rtopk_select", "rtopk_select_stats", "rtopk_select_bucketed", "maxk_forward", "maxk_backward_scatter", "MaxK",
           "read_status",
           "maxk_spgemm_forward", "maxk_sspmm_backward", "maxk_sspmm_backward_scatter"]


def __getattr__(name):
    if name in __all__:
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
