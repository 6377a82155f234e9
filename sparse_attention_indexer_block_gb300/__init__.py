"""GB300-native (sm_103a) decode/prefill sparse-attention indexer.

The compute lives in ``libsaib.so`` (hand-written CUDA, see ``include/indexer.h``
for the C ABI); this package builds it (``build.build()``) and binds it with
ctypes (``binding``). Importing the package does not load the library; the
first call does, and raises if it has not been built.
"""
from .binding import (  # noqa: F401
    IndexerError,
    decode_workspace,
    indexer_block_topk,
    indexer_dcp_merge,
    indexer_index_key_counts,
    indexer_decode_logits,
    indexer_decode_logits_mxfp4,
    indexer_decode_topk,
    indexer_decode_topk_from_lens,
    indexer_decode_topk_mxfp4,
    indexer_decode_topk_noalloc,
    indexer_decode_topk_values,
    indexer_decode_workspace_bytes,
    indexer_expand_decode_rows,
    indexer_expand_pools,
    indexer_insert_keys,
    indexer_plan_prefill_chunks,
    indexer_prefill_topk,
    indexer_prefill_topk_values,
    indexer_prefill_workspace_bytes,
    indexer_profile_events,
    indexer_trace_buffer,
    indexer_debug_divide,
    indexer_debug_wait_limit,
    indexer_debug_decode_plan,
    indexer_quantize_q,
    indexer_status_string,
    load,
)
