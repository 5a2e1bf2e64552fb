"""GB300 (sm_103a) three-tier compressed attention of the DeepSeek V4 Flash
engine (DwarfStar, ds4): indexer score -> top-k select -> sparse attention,
hand-written CUDA behind the C ABI of include/ds4a.h.

The Python surface is the ctypes binding (same names as the C entry points)
and DecodeStep / PrefillStep, which chain the three ops on one stream, plus
DenseStep for the ratio-128 layers (attention over all rows, no indexer).
"""
from ._binding import (Ds4aError, load, ds4a_version, ds4a_workspace_bytes, ds4a_get_device_status,
                       ds4a_debug_inject_error, ds4a_debug_wait_timeout, ds4a_indexer_score, ds4a_topk_select,
                       ds4a_sparse_attn_decode, ds4a_sparse_attn_prefill, ds4a_dense_attn_decode,
                       ds4a_kv_push_raw, ds4a_compressor_pool, ds4a_sparse_attn_decode_heads,
                       ds4a_sparse_attn_prefill_heads, ds4a_dense_attn_decode_heads, ds4a_rows_to_fp8,
                       ds4a_sparse_attn_decode_fp8, ds4a_sparse_attn_prefill_fp8, ds4a_indexer_topk)
from .step import DecodeStep, PrefillStep, DenseStep, ProducerStep, DEFAULT_SCALE

__all__ = ["Ds4aError", "load", "ds4a_version", "ds4a_workspace_bytes", "ds4a_get_device_status",
           "ds4a_debug_inject_error", "ds4a_debug_wait_timeout", "ds4a_indexer_score", "ds4a_topk_select", "ds4a_sparse_attn_decode",
           "ds4a_sparse_attn_prefill", "ds4a_dense_attn_decode", "ds4a_kv_push_raw", "ds4a_compressor_pool",
           "ds4a_sparse_attn_decode_heads", "ds4a_sparse_attn_prefill_heads", "ds4a_dense_attn_decode_heads",
           "ds4a_rows_to_fp8", "ds4a_sparse_attn_decode_fp8", "ds4a_sparse_attn_prefill_fp8", "ds4a_indexer_topk",
           "DecodeStep", "PrefillStep", "DenseStep", "ProducerStep",
           "DEFAULT_SCALE"]
