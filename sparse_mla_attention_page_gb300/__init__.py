"""GB300 (sm_103a) DSA top-k sparse MLA attention over a paged FP8 KV cache.

The compute lives in the C-ABI CUDA library ``libdsa_gb300.so`` (declared in
include/dsa.h); ``binding`` exposes its entry points under the same names.
"""
from .binding import (  # noqa: F401
    DSA_KV_RAW512, DSA_KV_SCALED528, DsaError, dsa_kv_row_bytes, dsa_kv_write_raw,
    dsa_kv_write_scaled, dsa_quantize_q8, dsa_sparse_attn_decode, dsa_sparse_attn_prefill_q8,
    dsa_sparse_attn_workspace_bytes, workspace_for,
)
