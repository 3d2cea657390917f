"""GB300 (sm_103a) routed-attention DiT forward: Python binding of libh3dit.so.

The computation lives in the CUDA library; this package only marshals
arguments (see ``_binding``).  Importing it does not load the library; the
first call does, and fails loudly if the library has not been built.
"""
from ._binding import (  # noqa: F401
    EXPORTED, Schedule, H3DIT_POOLED, H3DIT_QK_NORM, H3DIT_ROPE, H3DIT_SWIGLU, BlockWeights, H3DitError, Shape,
    attn_shape, block_forward, block_weights, check_shape, denoise_step, lib, linear, make_shape,
    routed_attention, routed_attention_static, select_blocks, sync_status, version, workspace_bytes, STAGES, profile_begin,
    profile_end, launch_count, selftest_timeout,
)
