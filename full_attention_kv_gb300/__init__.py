"""Hybrid-SWA dual-KV-pool attention for GB300 (sm_103a).

The library is ``_build/libhsa.so`` with the C ABI of ``include/hsa.h``; this
package is its thin Python binding.  Build it with ``__graft_entry__.build()``
(or ``python -m full_attention_kv_gb300.build``).
"""
from .binding import (  # noqa: F401
    EXPORTS, HSA_CUDA_ERROR, HSA_DECODE_APPEND, HSA_DECODE_EARLY_POOL_READ, HSA_DEVERR_BAD_BLOCK,
    HSA_DEVERR_BAD_LEN, HSA_DEVERR_BAD_PAGE, HSA_DEVERR_BAD_RING, HSA_DEVERR_BAD_SEQ,
    HSA_DEVERR_TIMEOUT, HSA_INVALID_ARG, HSA_KV_E4M3, HSA_KV_E5M2, HSA_OK, HSA_OUT_OF_RANGE,
    HSA_UNSUPPORTED_SHAPE, TREE_EXPORTS, DualPool, HsaError, HsaPools, PrefixTree, decode_workspace, hsa_decode_attn,
    fp8_code, hsa_decode_attn_append, hsa_decode_attn_noalloc, hsa_decode_workspace_bytes,
    hsa_kv_append,
    hsa_prefill_attn, hsa_swa_prefetch, hsa_window_safe_len, hsa_window_safe_len_bitmap, lib,
    status_string)
