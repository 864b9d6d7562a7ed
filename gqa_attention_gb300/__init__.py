"""Grouped-query fused attention forward for one GB300 (sm_103a).

The compute runs in ``libgqa_attn.so`` (CUDA kernels behind a C ABI declared in
``include/gqa_attn.h``); this package is its thin Python binding.  The library
is loaded on first use and a missing or unbuildable library raises: there is no
CPU fallback.
"""

from ._binding import (  # noqa: E402,F401
    GQA_ERR_CUDA,
    GQA_ERR_INVALID_ARG,
    GQA_ERR_TIMEOUT,
    GQA_ERR_UNSUPPORTED,
    GQA_OK,
    GQAError,
    decode,
    decode_fp8,
    decode_fused,
    decode_multi,
    decode_paged,
    decode_workspace,
    gqa_attn_decode,
    gqa_attn_decode_combine,
    gqa_attn_decode_default_splits,
    gqa_attn_decode_fp8,
    gqa_attn_decode_fused,
    gqa_attn_decode_fused_splits,
    gqa_attn_decode_multi,
    gqa_attn_decode_multi_default_splits,
    gqa_attn_decode_noalloc,
    gqa_attn_decode_paged,
    gqa_attn_decode_paged_fp8,
    gqa_attn_decode_paged_multi,
    gqa_attn_decode_split_chunk,
    gqa_attn_decode_workspace_bytes,
    gqa_attn_prefill_causal,
    gqa_attn_prefill_chunk,
    gqa_attn_prefill_chunk_default_parts,
    gqa_attn_prefill_chunk_split,
    gqa_attn_prefill_chunk_workspace_bytes,
    gqa_last_device_error,
    gqa_trace_clear,
    gqa_trace_mma_rate,
    gqa_trace_prefill_read,
    gqa_trace_read,
    gqa_selftest_wait_timeout,
    gqa_set_wait_limit_ns,
    load,
    paged_default_splits,
    prefill_causal,
    prefill_chunk,
    split_workspace,
    status_str,
)
