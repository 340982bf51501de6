"""GQA attention with a learned per-head softmax sink, native to GB300 (sm_103a).

Public API (thin wrappers over the C ABI in ``include/sinkattn.h``):
``sinkattn_prefill``, ``sinkattn_decode_split``, ``sinkattn_merge``,
``sinkattn_decode``, ``sinkattn_decode_fused``, ``sinkattn_decode_noalloc``, ``sinkattn_decode_workspace_bytes``,
``sinkattn_decode_default_splits``, ``sinkattn_prefill_paged``,
``sinkattn_decode_split_paged``, ``sinkattn_decode_paged`` (paged KV cache),
``sinkattn_decode_split_fp8``, ``sinkattn_decode_fp8`` (FP8 e4m3 KV cache),
``sinkattn_status_string``,
``sinkattn_last_error``, ``sinkattn_debug_status``, ``sinkattn_debug_set_hooks`` (tests),
``sinkattn_set_decode_kernel``,
``sinkattn_set_prefill_kernel``.

The compiled library is loaded on first use; if it has not been built, every
call raises (there is no CPU fallback).
"""
from ._binding import (  # noqa: F401
    SinkAttnError,
    lib,
    sinkattn_debug_set_hooks,
    sinkattn_debug_status,
    sinkattn_decode,
    sinkattn_decode_default_splits,
    sinkattn_decode_fp8,
    sinkattn_decode_fused,
    sinkattn_decode_noalloc,
    sinkattn_decode_paged,
    sinkattn_decode_split,
    sinkattn_decode_split_fp8,
    sinkattn_decode_split_paged,
    sinkattn_decode_workspace_bytes,
    sinkattn_last_error,
    sinkattn_merge,
    sinkattn_prefill,
    sinkattn_prefill_paged,
    sinkattn_set_decode_kernel,
    sinkattn_set_prefill_kernel,
    sinkattn_status_string,
)
from . import workloads  # noqa: F401
