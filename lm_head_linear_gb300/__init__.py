"""Fused linear cross-entropy for GB300 (sm_103a).

``flce_forward`` / ``flce_backward`` call the C ABI of the in-tree CUDA
library (``include/flce.h``); ``linear_cross_entropy`` wraps them in autograd.
The library is loaded on first use; a missing library raises, there is no
fallback.
"""

from .binding import (  # noqa: F401
    FlceError,
    LinearCrossEntropy,
    REDUCTIONS,
    SIGNATURES,
    flce_backward,
    flce_backward_chunk_tokens,
    flce_backward_workspace_size_for_chunk,
    flce_backward_shard,
    flce_combine_shards,
    flce_backward_workspace_size,
    flce_forward,
    flce_forward_valid,
    flce_forward_valid_workspace_size,
    flce_forward_shard,
    flce_forward_workspace_size,
    flce_profile_collect,
    flce_profile_enable,
    flce_read_device_status,
    flce_score,
    flce_score_valid,
    flce_selftest_wait_timeout,
    flce_set_wait_timeout_ns,
    library_path,
    linear_cross_entropy,
    linear_log_probs,
    load_library,
)
