"""GB300 (sm_103a) routed-attention DiT forward: Python binding of libh3dit.so.

The computation lives in the CUDA library; this package only marshals
arguments (see ``_binding``).  Importing it does not load the library; the
first call does, and fails loudly if the library has not been built.
"""
from ._binding import (  # noqa: F401
    EXPORTED, STAGES, H3DIT_PASS_CORE_REUSE, H3DIT_PASS_EXTRAPOLATE, H3DIT_PASS_FRESH,
    H3DIT_KEEP_INTERMEDIATES, H3DIT_POOLED, H3DIT_QK_NORM, H3DIT_ROPE, H3DIT_SWIGLU,
    H3DIT_TOKEN_REDUCTION, BlockWeights,
    H3DitError, Ends, Reduction, Schedule, Shape, attn_shape, block_forward, block_weights, check_shape,
    denoise_step, gemm_cta_pairs, launch_count, lib, linear, make_ends, make_shape, profile_begin, profile_end,
    routed_attention, routed_attention_static, routed_attention_static_status, sample_step, select_blocks, selftest_timeout, sync_status,
    tile_spans, version, video_order, workspace_bytes, workspace_layout,
)
