"""GB300 (sm_103a) implementation of Slow-Fast Inference decode attention over a
sparse, recallable KV memory.

The compute path is libsfi.so (CUDA kernels behind the C ABI in include/sfi.h);
this package is its Python binding (same function names) plus the host runtime
that orders the kernels on a main and an aux stream. Nothing here falls back to
another implementation: every call fails loudly if libsfi.so is missing.
"""
from .api import (SFI_ATTN_EARLY_KV_PREFETCH, SFI_ATTN_RAGGED, SFI_ATTN_TEST_WITHHOLD, SFI_MAX_QUERY_TOKENS,
                  AttnShape, CompactKV, PagedKV, SFIError, alloc_mixed_workspace, alloc_multi_workspace,
                  alloc_ragged_workspace, alloc_workspace, sfi_compact_gather, sfi_dense_verify_attn,
                  sfi_fast_decode_attn, sfi_fast_decode_attn_noalloc, sfi_mixed_decode_attn,
                  sfi_mixed_workspace_size, sfi_multi_workspace_size, sfi_paged_kv_append,
                  sfi_paged_kv_append_tokens, sfi_plan_splits, sfi_attn_cluster_capacity, sfi_select_compact,
                  sfi_select_topk, sfi_slow_dense_attn_with_scores, sfi_sparse_draft_attn, sfi_version,
                  sfi_workspace_size)
from .runtime import (DecodeBatch, LayerBuffers, SFIDecoder, SlowFastSchedule, StepIO, allocate_layers,
                      compact_layout)

__all__ = [
    "SFI_ATTN_EARLY_KV_PREFETCH", "SFI_ATTN_RAGGED", "SFI_ATTN_TEST_WITHHOLD", "SFI_MAX_QUERY_TOKENS", "AttnShape", "CompactKV",
    "PagedKV", "SFIError", "alloc_mixed_workspace", "alloc_multi_workspace", "alloc_ragged_workspace",
    "alloc_workspace", "sfi_compact_gather", "sfi_dense_verify_attn", "sfi_fast_decode_attn",
    "sfi_fast_decode_attn_noalloc", "sfi_mixed_decode_attn", "sfi_mixed_workspace_size",
    "sfi_multi_workspace_size", "sfi_paged_kv_append", "sfi_paged_kv_append_tokens", "sfi_plan_splits",
    "sfi_attn_cluster_capacity",
    "sfi_select_compact", "sfi_select_topk", "sfi_slow_dense_attn_with_scores", "sfi_sparse_draft_attn",
    "sfi_version", "sfi_workspace_size", "DecodeBatch", "LayerBuffers", "SFIDecoder", "SlowFastSchedule",
    "StepIO", "allocate_layers", "compact_layout",
]
