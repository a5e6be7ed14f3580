"""Python binding of libsfi with the C ABI's names (argument marshalling only).

Each function takes torch CUDA tensors, checks their dtype, device and layout,
passes their device pointers to the C entry point of the same name on the given
(or current) stream, and raises SFIError on a non-zero status. No arithmetic of
the method happens here.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional

import torch

from . import _abi


SFI_ATTN_EARLY_KV_PREFETCH = _abi.SFI_ATTN_EARLY_KV_PREFETCH
SFI_MAX_QUERY_TOKENS = _abi.SFI_MAX_QUERY_TOKENS
SFI_ATTN_RAGGED = _abi.SFI_ATTN_RAGGED
SFI_ATTN_TEST_WITHHOLD = _abi.SFI_ATTN_TEST_WITHHOLD


class SFIError(RuntimeError):
    def __init__(self, status: int, where: str):
        name = _abi.lib().sfi_status_string(status).decode()
        super().__init__(f"{where}: {name}")
        self.status = status


@dataclass(frozen=True)
class AttnShape:
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int = 16
    softmax_scale: float = 0.0  # <= 0: 1/sqrt(head_dim)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def c(self) -> _abi.sfi_attn_shape:
        return _abi.sfi_attn_shape(self.num_q_heads, self.num_kv_heads, self.head_dim, self.page_size,
                                   float(self.softmax_scale))


@dataclass
class PagedKV:
    """Paged bf16 KV cache: pools [num_pages][Hkv][P][D], page_table int32 [B][max_pages], seq_lens int32 [B]."""
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    page_table: torch.Tensor
    seq_lens: torch.Tensor

    def c(self) -> _abi.sfi_paged_kv:
        for name, t, dt in (("k_pool", self.k_pool, torch.bfloat16), ("v_pool", self.v_pool, torch.bfloat16),
                            ("page_table", self.page_table, torch.int32), ("seq_lens", self.seq_lens, torch.int32)):
            _need(t, dt, name)
        return _abi.sfi_paged_kv(self.k_pool.data_ptr(), self.v_pool.data_ptr(), self.k_pool.shape[0],
                                 self.page_table.shape[1], self.page_table.data_ptr(), self.seq_lens.data_ptr())


@dataclass
class CompactKV:
    """Compact buffer: k, v bf16 [total_rows][D]; row_offset int64 [B]; capacity, count int32 [B]."""
    k: torch.Tensor
    v: torch.Tensor
    row_offset: torch.Tensor
    capacity: torch.Tensor
    count: torch.Tensor

    def c(self) -> _abi.sfi_compact_kv:
        _need(self.k, torch.bfloat16, "compact.k")
        _need(self.v, torch.bfloat16, "compact.v")
        _need(self.row_offset, torch.int64, "compact.row_offset")
        _need(self.capacity, torch.int32, "compact.capacity")
        _need(self.count, torch.int32, "compact.count")
        return _abi.sfi_compact_kv(self.k.data_ptr(), self.v.data_ptr(), self.k.shape[0],
                                   self.row_offset.data_ptr(), self.capacity.data_ptr(), self.count.data_ptr())


def _need(t: Optional[torch.Tensor], dtype, name: str):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _ptr(t: Optional[torch.Tensor], dtype=None, name: str = "") -> Optional[int]:
    if t is None:
        return None
    if dtype is not None:
        _need(t, dtype, name)
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _batch(batch, req_ids, seq_lens) -> int:
    if batch is not None:
        return int(batch)
    if req_ids is not None:
        return int(req_ids.numel())
    return int(seq_lens.numel())


def _check(status: int, where: str):
    if status != _abi.SFI_OK:
        raise SFIError(status, where)


def sfi_paged_kv_append(shape: AttnShape, kv: PagedKV, k_new: torch.Tensor, v_new: torch.Tensor,
                        req_ids: Optional[torch.Tensor] = None, batch: Optional[int] = None,
                        dev_status: Optional[torch.Tensor] = None, stream=None):
    st = _abi.lib().sfi_paged_kv_append(
        ctypes.byref(shape.c()), ctypes.byref(kv.c()), _ptr(k_new, torch.bfloat16, "k_new"),
        _ptr(v_new, torch.bfloat16, "v_new"), _ptr(req_ids, torch.int32, "req_ids"),
        _batch(batch, req_ids, kv.seq_lens), _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(st, "sfi_paged_kv_append")


def sfi_fast_decode_attn(shape: AttnShape, kv: PagedKV, compact: CompactKV, sink: int, recent: int,
                         q: torch.Tensor, out: torch.Tensor, lse: Optional[torch.Tensor] = None,
                         req_ids: Optional[torch.Tensor] = None, batch: Optional[int] = None, max_tokens: int = 0,
                         num_splits: int = 0, workspace: Optional[torch.Tensor] = None,
                         dev_status: Optional[torch.Tensor] = None, stream=None,
                         k_new: Optional[torch.Tensor] = None, v_new: Optional[torch.Tensor] = None,
                         flags: int = 0):
    ws = _ptr(workspace, torch.uint8, "workspace")
    st = _abi.lib().sfi_fast_decode_attn(
        ctypes.byref(shape.c()), ctypes.byref(kv.c()), ctypes.byref(compact.c()), int(sink), int(recent),
        _ptr(q, torch.bfloat16, "q"), _ptr(k_new, torch.bfloat16, "k_new"), _ptr(v_new, torch.bfloat16, "v_new"),
        _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"),
        _ptr(req_ids, torch.int32, "req_ids"), _batch(batch, req_ids, kv.seq_lens), int(max_tokens),
        int(num_splits), int(flags), ws, 0 if workspace is None else workspace.numel(),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(st, "sfi_fast_decode_attn")


def sfi_slow_dense_attn_with_scores(shape: AttnShape, kv: PagedKV, sink: int, recent: int, q: torch.Tensor,
                                    out: torch.Tensor, lse: Optional[torch.Tensor] = None,
                                    scores: Optional[torch.Tensor] = None, req_ids: Optional[torch.Tensor] = None,
                                    batch: Optional[int] = None, max_tokens: int = 0, num_splits: int = 0,
                                    workspace: Optional[torch.Tensor] = None,
                                    dev_status: Optional[torch.Tensor] = None, stream=None,
                                    k_new: Optional[torch.Tensor] = None, v_new: Optional[torch.Tensor] = None,
                                    flags: int = 0):
    ws = _ptr(workspace, torch.uint8, "workspace")
    stride = 0 if scores is None else int(scores.shape[-1])
    st = _abi.lib().sfi_slow_dense_attn_with_scores(
        ctypes.byref(shape.c()), ctypes.byref(kv.c()), int(sink), int(recent), _ptr(q, torch.bfloat16, "q"),
        _ptr(k_new, torch.bfloat16, "k_new"), _ptr(v_new, torch.bfloat16, "v_new"), _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"), _ptr(scores, torch.float32, "scores"),
        stride, _ptr(req_ids, torch.int32, "req_ids"), _batch(batch, req_ids, kv.seq_lens), int(max_tokens),
        int(num_splits), int(flags), ws, 0 if workspace is None else workspace.numel(),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(st, "sfi_slow_dense_attn_with_scores")


def sfi_mixed_decode_attn(shape: AttnShape, kv: PagedKV, compact: Optional[CompactKV], sink: int, recent: int,
                          q: torch.Tensor, out: torch.Tensor, fast_ids: torch.Tensor, slow_ids: torch.Tensor,
                          lse: Optional[torch.Tensor] = None, scores: Optional[torch.Tensor] = None,
                          k_new: Optional[torch.Tensor] = None, v_new: Optional[torch.Tensor] = None,
                          max_fast_tokens: int = 0, max_dense_tokens: int = 0, flags: int = 0,
                          workspace: Optional[torch.Tensor] = None, dev_status: Optional[torch.Tensor] = None,
                          stream=None):
    ws = _ptr(workspace, torch.uint8, "workspace")
    n_fast, n_slow = int(fast_ids.numel()), int(slow_ids.numel())
    st = _abi.lib().sfi_mixed_decode_attn(
        ctypes.byref(shape.c()), ctypes.byref(kv.c()), None if compact is None else ctypes.byref(compact.c()),
        int(sink), int(recent), _ptr(q, torch.bfloat16, "q"), _ptr(k_new, torch.bfloat16, "k_new"),
        _ptr(v_new, torch.bfloat16, "v_new"), _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"),
        _ptr(scores, torch.float32, "scores"), 0 if scores is None else int(scores.shape[-1]),
        _ptr(fast_ids, torch.int32, "fast_ids") if n_fast else None, n_fast,
        _ptr(slow_ids, torch.int32, "slow_ids") if n_slow else None, n_slow, int(max_fast_tokens),
        int(max_dense_tokens), int(flags), ws, 0 if workspace is None else workspace.numel(),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(st, "sfi_mixed_decode_attn")


def sfi_mixed_workspace_size(shape: AttnShape, n_fast: int, n_slow: int, max_fast_tokens: int,
                             max_dense_tokens: int) -> int:
    return int(_abi.lib().sfi_mixed_workspace_size(ctypes.byref(shape.c()), int(n_fast), int(n_slow),
                                                   int(max_fast_tokens), int(max_dense_tokens)))


def alloc_mixed_workspace(shape: AttnShape, batch: int, max_fast_tokens: int, max_dense_tokens: int,
                          device="cuda") -> torch.Tensor:
    """A zero-filled workspace large enough for every split of `batch` requests into
    fast and slow subsets."""
    n = max([256] + [sfi_mixed_workspace_size(shape, batch - ns, ns, max_fast_tokens, max_dense_tokens)
                     for ns in range(batch + 1)])
    return torch.zeros(n, dtype=torch.uint8, device=device)


def alloc_ragged_workspace(shape: AttnShape, batch: int, max_tokens: int, dense: bool = False,
                           device="cuda") -> torch.Tensor:
    """A zero-filled workspace for sfi_fast_decode_attn (dense=False) or
    sfi_slow_dense_attn_with_scores (dense=True) with SFI_ATTN_RAGGED, valid for every
    batch size 1..batch."""
    n = max([256] + [sfi_mixed_workspace_size(shape, 0, b, 0, max_tokens) if dense
                     else sfi_mixed_workspace_size(shape, b, 0, max_tokens, 0) for b in range(1, batch + 1)])
    return torch.zeros(n, dtype=torch.uint8, device=device)


def sfi_paged_kv_append_tokens(shape: AttnShape, kv: PagedKV, k_new: torch.Tensor, v_new: torch.Tensor,
                               num_tokens: int, req_ids: Optional[torch.Tensor] = None, batch: Optional[int] = None,
                               dev_status: Optional[torch.Tensor] = None, stream=None):
    st = _abi.lib().sfi_paged_kv_append_tokens(
        ctypes.byref(shape.c()), ctypes.byref(kv.c()), _ptr(k_new, torch.bfloat16, "k_new"),
        _ptr(v_new, torch.bfloat16, "v_new"), int(num_tokens), _ptr(req_ids, torch.int32, "req_ids"),
        _batch(batch, req_ids, kv.seq_lens), _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(st, "sfi_paged_kv_append_tokens")


def sfi_dense_verify_attn(shape: AttnShape, kv: PagedKV, sink: int, recent: int, q: torch.Tensor, num_tokens: int,
                          out: torch.Tensor, lse: Optional[torch.Tensor] = None,
                          scores: Optional[torch.Tensor] = None, req_ids: Optional[torch.Tensor] = None,
                          batch: Optional[int] = None, max_tokens: int = 0, num_splits: int = 0,
                          workspace: Optional[torch.Tensor] = None, dev_status: Optional[torch.Tensor] = None,
                          stream=None, flags: int = 0, k_new: Optional[torch.Tensor] = None,
                          v_new: Optional[torch.Tensor] = None):
    ws = _ptr(workspace, torch.uint8, "workspace")
    stride = 0 if scores is None else int(scores.shape[-1])
    st = _abi.lib().sfi_dense_verify_attn(
        ctypes.byref(shape.c()), ctypes.byref(kv.c()), int(sink), int(recent), _ptr(q, torch.bfloat16, "q"),
        int(num_tokens), _ptr(k_new, torch.bfloat16, "k_new"), _ptr(v_new, torch.bfloat16, "v_new"),
        _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"),
        _ptr(scores, torch.float32, "scores"), stride, _ptr(req_ids, torch.int32, "req_ids"),
        _batch(batch, req_ids, kv.seq_lens), int(max_tokens), int(num_splits), int(flags), ws,
        0 if workspace is None else workspace.numel(), _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(st, "sfi_dense_verify_attn")


def sfi_sparse_draft_attn(shape: AttnShape, kv: PagedKV, compact: CompactKV, sink: int, recent: int,
                          q: torch.Tensor, num_tokens: int, out: torch.Tensor, lse: Optional[torch.Tensor] = None,
                          req_ids: Optional[torch.Tensor] = None, batch: Optional[int] = None, max_tokens: int = 0,
                          num_splits: int = 0, workspace: Optional[torch.Tensor] = None,
                          dev_status: Optional[torch.Tensor] = None, stream=None, flags: int = 0,
                          k_new: Optional[torch.Tensor] = None, v_new: Optional[torch.Tensor] = None):
    ws = _ptr(workspace, torch.uint8, "workspace")
    st = _abi.lib().sfi_sparse_draft_attn(
        ctypes.byref(shape.c()), ctypes.byref(kv.c()), ctypes.byref(compact.c()), int(sink), int(recent),
        _ptr(q, torch.bfloat16, "q"), int(num_tokens), _ptr(k_new, torch.bfloat16, "k_new"),
        _ptr(v_new, torch.bfloat16, "v_new"), _ptr(out, torch.float32, "out"),
        _ptr(lse, torch.float32, "lse"), _ptr(req_ids, torch.int32, "req_ids"), _batch(batch, req_ids, kv.seq_lens),
        int(max_tokens), int(num_splits), int(flags), ws, 0 if workspace is None else workspace.numel(),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(st, "sfi_sparse_draft_attn")


def sfi_multi_workspace_size(shape: AttnShape, batch: int, num_tokens: int, max_tokens: int,
                             num_splits: int = 0) -> int:
    return int(_abi.lib().sfi_multi_workspace_size(ctypes.byref(shape.c()), int(batch), int(num_tokens),
                                                   int(max_tokens), int(num_splits)))


def alloc_multi_workspace(shape: AttnShape, batch: int, num_tokens: int, max_tokens: int, num_splits: int = 0,
                          device="cuda") -> torch.Tensor:
    """A zero-filled workspace for the multi-token calls, valid for every batch size 1..batch."""
    n = max([256] + [sfi_multi_workspace_size(shape, b, num_tokens, max_tokens, num_splits)
                     for b in range(1, batch + 1)])
    return torch.zeros(n, dtype=torch.uint8, device=device)


def sfi_select_topk(scores: torch.Tensor, num_kv_heads: int, seq_lens: torch.Tensor, sink: int, recent: int,
                    k_per_req: torch.Tensor, idx_out: torch.Tensor, count_out: torch.Tensor,
                    req_ids: Optional[torch.Tensor] = None, batch: Optional[int] = None,
                    dev_status: Optional[torch.Tensor] = None, stream=None):
    st = _abi.lib().sfi_select_topk(
        _ptr(scores, torch.float32, "scores"), int(scores.shape[-1]), int(num_kv_heads),
        _ptr(seq_lens, torch.int32, "seq_lens"), int(sink), int(recent), _ptr(k_per_req, torch.int32, "k_per_req"),
        int(idx_out.shape[-1]), _ptr(idx_out, torch.int32, "idx_out"), _ptr(count_out, torch.int32, "count_out"),
        _ptr(req_ids, torch.int32, "req_ids"), _batch(batch, req_ids, seq_lens),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(st, "sfi_select_topk")


def sfi_select_compact(shape: AttnShape, kv: PagedKV, scores: torch.Tensor, sink: int, recent: int,
                       k_per_req: torch.Tensor, idx_out: torch.Tensor, compact: CompactKV,
                       count_out: Optional[torch.Tensor] = None, req_ids: Optional[torch.Tensor] = None,
                       batch: Optional[int] = None, dev_status: Optional[torch.Tensor] = None, stream=None):
    """Selector + compaction in one launch; count_out defaults to compact.count."""
    count_out = compact.count if count_out is None else count_out
    st = _abi.lib().sfi_select_compact(
        ctypes.byref(shape.c()), ctypes.byref(kv.c()), _ptr(scores, torch.float32, "scores"), int(scores.shape[-1]),
        int(sink), int(recent), _ptr(k_per_req, torch.int32, "k_per_req"), int(idx_out.shape[-1]),
        _ptr(idx_out, torch.int32, "idx_out"), _ptr(count_out, torch.int32, "count_out"), ctypes.byref(compact.c()),
        _ptr(req_ids, torch.int32, "req_ids"), _batch(batch, req_ids, kv.seq_lens),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(st, "sfi_select_compact")


def sfi_compact_gather(shape: AttnShape, kv: PagedKV, idx: torch.Tensor, count: torch.Tensor, sink: int,
                       compact: CompactKV, req_ids: Optional[torch.Tensor] = None, batch: Optional[int] = None,
                       dev_status: Optional[torch.Tensor] = None, stream=None):
    st = _abi.lib().sfi_compact_gather(
        ctypes.byref(shape.c()), ctypes.byref(kv.c()), _ptr(idx, torch.int32, "idx"),
        _ptr(count, torch.int32, "count"), int(idx.shape[-1]), int(sink), ctypes.byref(compact.c()),
        _ptr(req_ids, torch.int32, "req_ids"), _batch(batch, req_ids, kv.seq_lens),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(st, "sfi_compact_gather")


def sfi_fast_decode_attn_noalloc(shape: AttnShape, kv: PagedKV, compact: CompactKV, sink: int, recent: int,
                                 q: torch.Tensor, out: torch.Tensor, lse: Optional[torch.Tensor] = None,
                                 req_ids: Optional[torch.Tensor] = None, batch: Optional[int] = None,
                                 max_tokens: int = 0, num_splits: int = 0,
                                 dev_status: Optional[torch.Tensor] = None, stream=None,
                                 k_new: Optional[torch.Tensor] = None, v_new: Optional[torch.Tensor] = None,
                                 flags: int = 0):
    """sfi_fast_decode_attn without a workspace argument, for callers that cannot
    allocate device memory: the split-KV scratch is a fixed array inside the library
    (SFI_NOALLOC_SCRATCH_BYTES per GPU). Calls that may overlap on the GPU share that
    array and race; order them on one stream."""
    st = _abi.lib().sfi_fast_decode_attn_noalloc(
        ctypes.byref(shape.c()), ctypes.byref(kv.c()), ctypes.byref(compact.c()), int(sink), int(recent),
        _ptr(q, torch.bfloat16, "q"), _ptr(k_new, torch.bfloat16, "k_new"), _ptr(v_new, torch.bfloat16, "v_new"),
        _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"),
        _ptr(req_ids, torch.int32, "req_ids"), _batch(batch, req_ids, kv.seq_lens), int(max_tokens),
        int(num_splits), int(flags), _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(st, "sfi_fast_decode_attn_noalloc")


def sfi_workspace_size(shape: AttnShape, batch: int, max_tokens: int, num_splits: int = 0) -> int:
    return int(_abi.lib().sfi_workspace_size(ctypes.byref(shape.c()), int(batch), int(max_tokens), int(num_splits)))


def sfi_plan_splits(shape: AttnShape, batch: int, max_tokens: int, num_splits: int = 0) -> int:
    return int(_abi.lib().sfi_plan_splits(ctypes.byref(shape.c()), int(batch), int(max_tokens), int(num_splits)))


def sfi_attn_cluster_capacity(cluster_size: int) -> int:
    return int(_abi.lib().sfi_attn_cluster_capacity(int(cluster_size)))


def sfi_version() -> int:
    return int(_abi.lib().sfi_version())


def alloc_workspace(shape: AttnShape, batch: int, max_tokens: int, num_splits: int = 0, device="cuda",
                    any_subset: bool = True) -> torch.Tensor:
    """A zero-filled workspace (at least 256 bytes; torch allocations are 256-byte aligned).

    With any_subset, it is large enough for every batch size 1..batch (calls on a
    subset of the requests plan their splits for the subset's size).
    """
    sizes = range(1, batch + 1) if any_subset else [batch]
    n = max([256] + [sfi_workspace_size(shape, b, max_tokens, num_splits) for b in sizes])
    return torch.zeros(n, dtype=torch.uint8, device=device)
