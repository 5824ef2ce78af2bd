"""GB300-native (sm_103a) BF16 multi-head attention leaf.

O = softmax(Q K^T * D^-0.5) V over [B, N, H, D] bf16 tensors, D in {64, 128},
in three forms: dense non-causal attention (``attn_dense_fwd``), prefix-cached
full-visibility attention over cat(K_prefix, K_current) without a copy
(``attn_prefix_fwd``), and block-causal attention over text and image segments
(``attn_block_causal_fwd``).  The compute runs in hand-written tcgen05/TMA kernels
behind the C ABI of ``include/ncp_attn.h``; this package only builds, loads
and calls that library.
"""
from ._binding import (  # noqa: F401
    ATTN_ERR_ALIAS, ATTN_ERR_ALIGN, ATTN_ERR_CUDA, ATTN_ERR_HEADDIM, ATTN_ERR_NULL,
    ATTN_ERR_SHAPE, ATTN_ERR_TIMEOUT, ATTN_OK, SIGNATURES, AttnError, attn_dense_fwd,
    attn_block_causal_fwd, attn_dense_cross_fwd, attn_dense_fwd_noalloc, attn_masked_prefix_fwd,
    block_causal_attention,
    attn_prefix_fwd, debug_exp2, debug_schedule, debug_set_fault, dense_attention, device_status,
    library_path,
    load_library, prefix_attention, status_string,
)
from ._build import build  # noqa: F401

attn_status_string = status_string
