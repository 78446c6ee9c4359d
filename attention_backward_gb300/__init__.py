"""GB300-native fused softmax-attention backward.

The compute lives in the CUDA library ``_build/libattn_bwd.so`` (C ABI,
``include/attn_bwd.h``); this package only marshals torch tensors into that
ABI.  There is no CPU path: every call fails loudly when the library or a
CUDA device is missing.
"""
from ._binding import (  # noqa: F401
    AttnBwdError,
    LIB_PATH,
    attn_bwd,
    attn_bwd_gqa,
    attn_bwd_sparse,
    attn_fwd_gqa,
    backward,
    backward_host,
    check_error,
    dq_land,
    forward,
    gqa_main,
    gqa_workspace_size,
    host_scratch_size,
    library,
    preprocess,
    query_block_range,
    query_block_range_qk,
    selftest_timeout,
    sink_grad,
    sparse_backward,
    sparse_land,
    sparse_main,
    tail_plan,
    tile_schedule,
    tile_schedule_split,
    workspace_size,
)
