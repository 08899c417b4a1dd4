"""Fused linear cross-entropy for GB300 (sm_103a): loss and gradients of the LM head without the
(BT, V) logits in device memory, plus a standalone in-place row-wise CE kernel.

The compute path is libflce.so (hand-written CUDA, C ABI in include/flce.h); this package only
marshals arguments to it.  Build it with ``python -m linear_cross_entropy_tma_gb300.build``.
"""
from ._lib import (  # noqa: F401
    STATUS_BAD_TARGET,
    STATUS_TIMEOUT,
    ce_with_grad,
    ce_workspace_size,
    cross_entropy,
    flce_fwd_bwd,
    load,
    read_device_status,
    read_filter_skips,
    read_side_clusters,
    read_side_launches,
    read_single_clusters,
    read_single_launches,
    read_single_units,
    read_token_split_units,
    read_vocab_split_units,
    workspace_size,
)
