"""GB300 (sm_103a) MoE expert-parallel hot path: routing layout, dispatch
(BF16 or fused FP8 e4m3 with per-128-channel scales) and weighted top-k
combine, as hand-written CUDA kernels behind a C ABI (``include/ep.h``).

``binding`` marshals torch tensors into that ABI; ``workloads`` draws the
seeded synthetic inputs.
"""
from .binding import (  # noqa: F401
    EpError, LayoutOut, Pipeline, combine, combine_fp8, dispatch, dispatch_fp8, layout, layout_dispatch,
    layout_workspace_bytes, load,
    layout_static_ws, status_read, rank_layout, rank_rows_bound, expand, expand_fp8, combine_partial,
    combine_reduce, RankLayoutOut, EP_FLAG_BAD_EXPERT, EP_FLAG_OVERFLOW, EP_FLAG_BAD_ROW, EP_FLAG_TIMEOUT,
)
