"""Single-GPU MoE expert-parallel dispatch / combine for GB300 (sm_103a).

The hot path -- routing layout, dispatch copy epilogue (BF16 or fused FP8
quantisation) and combine -- is hand-written CUDA in ``libep.so`` behind the
C ABI declared in ``include/ep.h``; this package is its thin Python binding
(argument marshalling; torch supplies device memory and streams).
"""
from ._binding import (  # noqa: F401
    EP_ABI_VERSION, EP_ERR_BAD_TOPK_IDX, EP_ERR_CUDA, EP_ERR_INVALID_ARG, EP_ERR_OOM,
    EP_ERR_OVERFLOW, EP_ERR_TIMEOUT, EP_ERR_UNSUPPORTED, EP_ERRBIT_BAD_TOPK_IDX,
    EP_ERRBIT_OVERFLOW, EP_OK, LIB_PATH, EpConfigC, EpError, EpLayoutInfoC, Handle,
    alloc_recv, ep_combine, ep_dispatch, ep_handle_free, ep_layout, host_wait_flag,
    load_library, make_config, status_string, upper_bound_rows, validate_config,
    EP_NOALLOC_SCRATCH_WORDS, EpLayoutBuffersC, alloc_layout_buffers, ep_layout_noalloc,
    EP_ERRBIT_TIMEOUT, selftest_bounded_wait, ep_combine_backward, ep_dispatch_backward,
    ep_dispatch_fp8, alloc_recv_planned, ep_layout_dispatch, plan_layout,
)
