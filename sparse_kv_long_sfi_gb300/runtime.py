"""Host runtime of the SFI decode path: per-layer buffers, the slow/fast schedule and
the two-stream pipeline.

Slow-Fast Inference (Xie et al., 2026):
  * Figure 2 caption: a slow step is triggered by a boundary token or when a fixed
    refresh interval is reached; otherwise the step is fast.
  * Figure 3 caption (A): while the main stream computes attention for layer i+1,
    an aux stream runs the Selector and the cache reorganisation of layer i.
"A Sparse Glimpse of the Whole: Train-Free Self-Speculative Decoding" (abstract):
drafts over the sparse state, a full-context verification whose per-head statistics
refresh the selection (verify_step, refresh_selection, draft_step).
Every device operation of a step is one of libsfi's kernels; this module only
orders them on streams with events and keeps the per-request counters.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np
import torch

from .api import (SFI_ATTN_EARLY_KV_PREFETCH, SFI_ATTN_RAGGED, SFI_MAX_QUERY_TOKENS, AttnShape, CompactKV,
                  PagedKV, alloc_mixed_workspace, alloc_multi_workspace, alloc_ragged_workspace, alloc_workspace,
                  sfi_dense_verify_attn, sfi_fast_decode_attn, sfi_mixed_decode_attn, sfi_paged_kv_append,
                  sfi_paged_kv_append_tokens, sfi_select_compact, sfi_slow_dense_attn_with_scores,
                  sfi_sparse_draft_attn)


class SlowFastSchedule:
    """Per-request slow/fast decisions (host counters).

    Step t of request b is slow if it is the request's first step, if a boundary event
    fired, or if `interval` steps have passed since its last slow step.
    """

    def __init__(self, batch: int, interval: int):
        self.interval = int(interval)
        self.last_slow = np.full(batch, -1, np.int64)
        self.t = 0

    def next(self, boundary: Optional[np.ndarray] = None) -> np.ndarray:
        b = np.zeros_like(self.last_slow, dtype=bool) if boundary is None else np.asarray(boundary, bool)
        slow = (self.last_slow < 0) | b | (self.t - self.last_slow >= self.interval)
        self.last_slow[slow] = self.t
        self.t += 1
        return slow.astype(np.uint8)


@dataclass
class LayerBuffers:
    """Device state of one attention layer."""
    k_pool: torch.Tensor      # bf16 [num_pages][Hkv][P][D]
    v_pool: torch.Tensor
    compact: CompactKV        # sink + selected rows
    scores: torch.Tensor      # fp32 [B][Hkv][score_stride]
    idx: torch.Tensor         # int32 [B][Hkv][k_cap]


@dataclass
class DecodeBatch:
    """Requests shared by all layers: page table, capacities, per-request k."""
    page_table: torch.Tensor  # int32 [B][max_pages]
    row_offset: torch.Tensor  # int64 [B]
    capacity: torch.Tensor    # int32 [B]
    k_per_req: torch.Tensor   # int32 [B]
    k_cap: int
    score_stride: int


def allocate_layers(shape: AttnShape, num_layers: int, num_pages: int, batch: DecodeBatch, sink: int,
                    device="cuda", pool_init=None) -> List[LayerBuffers]:
    """Allocate per-layer pools, compact buffers, score and index arrays.

    pool_init(layer, k_pool, v_pool) fills the pools (e.g. seeded synthetic KV).
    """
    B = batch.page_table.shape[0]
    total_rows = int((batch.row_offset[-1] + shape.num_kv_heads * batch.capacity[-1]).item()) if B else 1
    layers = []
    for i in range(num_layers):
        kp = torch.empty((num_pages, shape.num_kv_heads, shape.page_size, shape.head_dim), dtype=torch.bfloat16,
                         device=device)
        vp = torch.empty_like(kp)
        if pool_init is not None:
            pool_init(i, kp, vp)
        ck = torch.zeros((max(total_rows, 1), shape.head_dim), dtype=torch.bfloat16, device=device)
        cv = torch.zeros_like(ck)
        comp = CompactKV(ck, cv, batch.row_offset, batch.capacity,
                         torch.zeros(B, dtype=torch.int32, device=device))
        scores = torch.empty((B, shape.num_kv_heads, batch.score_stride), dtype=torch.float32, device=device)
        idx = torch.zeros((B, shape.num_kv_heads, max(batch.k_cap, 1)), dtype=torch.int32, device=device)
        layers.append(LayerBuffers(kp, vp, comp, scores, idx))
    return layers


def compact_layout(shape: AttnShape, sink: int, k_per_req, device="cuda"):
    """Row offsets and capacities of a packed compact buffer (capacity = sink + k_r per KV head)."""
    k = np.asarray(k_per_req, np.int64)
    cap = sink + k
    off = np.concatenate([[0], np.cumsum(cap * shape.num_kv_heads)[:-1]]).astype(np.int64)
    return (torch.tensor(off, dtype=torch.int64, device=device), torch.tensor(cap, dtype=torch.int32, device=device))


@dataclass
class StepIO:
    """Per-step inputs/outputs of all layers (leading dim = layer). Multi-token steps
    (verify_step, draft_step) carry a token dim after the request dim:
    q [NL][B][T][Hq][D], k_new/v_new [NL][B][T][Hkv][D], out [NL][B][T][Hq][D]."""
    q: torch.Tensor           # bf16 [NL][B][Hq][D]
    k_new: torch.Tensor       # bf16 [NL][B][Hkv][D]
    v_new: torch.Tensor
    out: torch.Tensor         # fp32 [NL][B][Hq][D]
    lse: Optional[torch.Tensor] = None  # fp32 [NL][B][Hq]


class SFIDecoder:
    """Runs decode steps over all layers with a main and an aux stream.

    Slow step, per layer i (main stream): append, dense attention + masked scores,
    record e_i. Aux stream: wait e_i, Selector, compaction, record a_i. The main
    stream moves on to layer i + 1 at once (Figure 3A); the next use of layer i's
    compact buffer (a later step) waits a_i.
    """

    def __init__(self, shape: AttnShape, layers: List[LayerBuffers], batch: DecodeBatch, sink: int, recent: int,
                 max_len: int, dev_status: Optional[torch.Tensor] = None, device="cuda",
                 main_stream: Optional[torch.cuda.Stream] = None, aux_stream: Optional[torch.cuda.Stream] = None,
                 fuse_append: bool = True, single_launch_mixed: bool = True, ragged: bool = False,
                 k_max: Optional[int] = None):
        self.shape, self.layers, self.batch = shape, layers, batch
        # fuse_append: the attention kernels write the current token into the pages
        # themselves (no separate append launch per layer)
        self.fuse_append = bool(fuse_append)
        # single_launch_mixed: a mixed step runs one attention launch per layer for its
        # fast and slow requests together (sfi_mixed_decode_attn) instead of two
        self.single_launch_mixed = bool(single_launch_mixed)
        # ragged: the requests' lengths differ widely; the single-token fast and slow
        # launches are planned in fixed-size chunks sized by each request's own length
        # (SFI_ATTN_RAGGED) rather than with one split count for the whole batch
        self.ragged = bool(ragged)
        self.sink, self.recent = int(sink), int(recent)
        self.max_len = int(max_len)
        B = batch.page_table.shape[0]
        # k_max: the largest k_per_req the caller will set (default: the compact capacity).
        # It only sizes the split-KV plan of the fast launches: a bound above the real k
        # over-splits small batches, one below it costs speed, never correctness.
        k_plan = int(batch.k_cap) if k_max is None else max(0, min(int(k_max), int(batch.k_cap)))
        self.max_fast_tokens = self.sink + k_plan + self.recent + 2 * shape.page_size
        self.max_dense_tokens = self.max_len + shape.page_size
        if self.ragged:
            self.ws_fast = alloc_ragged_workspace(shape, B, self.max_fast_tokens, device=device)
            self.ws_dense = alloc_ragged_workspace(shape, B, self.max_dense_tokens, dense=True, device=device)
        else:
            self.ws_fast = alloc_workspace(shape, B, self.max_fast_tokens, device=device)
            self.ws_dense = alloc_workspace(shape, B, self.max_dense_tokens, device=device)
        self.ws_mixed = (alloc_mixed_workspace(shape, B, self.max_fast_tokens, self.max_dense_tokens, device=device)
                         if single_launch_mixed else None)
        self.ws_multi = None  # multi-token workspaces, allocated on first use
        self._device = device
        self.dev_status = dev_status if dev_status is not None else torch.zeros(1, dtype=torch.int32, device=device)
        lo, hi = torch.cuda.Stream.priority_range()
        self.main = main_stream or torch.cuda.Stream(device=device, priority=hi)
        self.aux = aux_stream or torch.cuda.Stream(device=device, priority=lo)
        self.e_attn = [torch.cuda.Event() for _ in layers]
        self.e_aux = [torch.cuda.Event() for _ in layers]
        self.pending = [False] * len(layers)
        # Consecutive attention launches on the main stream touch different layers (or,
        # within a mixed step, different requests' pages): each may stream its KV while
        # the previous one finishes. The separate-append path writes the pages right
        # before the attention, so it keeps the conservative launch.
        self.attn_flags = SFI_ATTN_EARLY_KV_PREFETCH if self.fuse_append else 0
        # flags of the single-token fast and slow launches
        self.step_flags = self.attn_flags | (SFI_ATTN_RAGGED if self.ragged else 0)
        # Optional instrumentation: called as timer(kind, "start"|"end", stream) around
        # each attention launch (kind "slow", "fast" or "dense"), e.g. to record events.
        self.timer = None

    def _mark(self, kind: str, phase: str):
        if self.timer is not None:
            self.timer(kind, phase, self.main)

    def kv(self, i: int, seq_lens: torch.Tensor) -> PagedKV:
        L = self.layers[i]
        return PagedKV(L.k_pool, L.v_pool, self.batch.page_table, seq_lens)

    def _append(self, i, kv, io, append, req_ids, n):
        """The current token of layer i: returned for the attention kernel to write
        (fused), or written now by the paged-append kernel."""
        if not append:
            return None, None
        if self.fuse_append:
            return io.k_new[i], io.v_new[i]
        sfi_paged_kv_append(self.shape, kv, io.k_new[i], io.v_new[i], req_ids=req_ids, batch=n,
                            dev_status=self.dev_status, stream=self.main)
        return None, None

    def _append_tokens(self, i, kv, io, T, append, req_ids, n):
        """The T newest tokens of layer i: returned for the multi-token kernel to write
        (fused), or written now by the T-token append kernel."""
        if not append:
            return None, None
        if self.fuse_append:
            return io.k_new[i], io.v_new[i]
        sfi_paged_kv_append_tokens(self.shape, kv, io.k_new[i], io.v_new[i], T, req_ids=req_ids, batch=n,
                                   dev_status=self.dev_status, stream=self.main)
        return None, None

    def _enter(self, name: str):
        """Order the main stream after the caller's stream (inputs such as seq_lens, q or
        k_new may have just been written there; torch streams do not synchronise with
        each other implicitly), and open the step's NVTX range ("sfi.<name>") so that a
        profiler's timeline groups its launches."""
        torch.cuda.nvtx.range_push("sfi." + name)
        cur = torch.cuda.current_stream(self.main.device)
        if cur != self.main:
            self.main.wait_stream(cur)

    def _leave(self, close_range: bool = True):
        """Order the caller's stream after the main stream (outputs, and reuse of the
        input tensors' memory by the caching allocator); close the step's NVTX range."""
        cur = torch.cuda.current_stream(self.main.device)
        if cur != self.main:
            cur.wait_stream(self.main)
        if close_range:
            torch.cuda.nvtx.range_pop()

    def _refresh(self, i: int, L: LayerBuffers, kv: PagedKV, seq_lens: torch.Tensor,
                 req_ids: Optional[torch.Tensor], n: Optional[int]):
        """Selector + compaction of layer i on the aux stream (already ordered after the
        scores), then record a_i."""
        sfi_select_compact(self.shape, PagedKV(kv.k_pool, kv.v_pool, kv.page_table, seq_lens), L.scores, self.sink,
                           self.recent, self.batch.k_per_req, L.idx, L.compact, req_ids=req_ids, batch=n,
                           dev_status=self.dev_status, stream=self.aux)
        self.e_aux[i].record(self.aux)
        self.pending[i] = True

    def _wait_aux(self, i: int):
        if self.pending[i]:
            self.main.wait_event(self.e_aux[i])
            self.pending[i] = False

    def _slow_layer(self, i: int, L: LayerBuffers, kv: PagedKV, io: StepIO, seq_lens: torch.Tensor,
                    req_ids: Optional[torch.Tensor], n: Optional[int], kn, vn):
        """Layer i of a slow step: dense attention + masked scores on the main stream,
        then the Selector and the compaction on the aux stream (Figure 3A)."""
        self._mark("slow", "start")
        sfi_slow_dense_attn_with_scores(self.shape, kv, self.sink, self.recent, io.q[i], io.out[i],
                                        None if io.lse is None else io.lse[i], L.scores, k_new=kn, v_new=vn,
                                        req_ids=req_ids, batch=n, max_tokens=self.max_dense_tokens,
                                        workspace=self.ws_dense, dev_status=self.dev_status, stream=self.main,
                                        flags=self.step_flags)
        self._mark("slow", "end")
        self.e_attn[i].record(self.main)
        self.aux.wait_event(self.e_attn[i])
        self._refresh(i, L, kv, seq_lens, req_ids, n)

    def slow_step(self, io: StepIO, seq_lens: torch.Tensor, req_ids: Optional[torch.Tensor] = None,
                  append: bool = True):
        n = None if req_ids is None else req_ids.numel()
        self._enter("slow_step")
        for i, L in enumerate(self.layers):
            kv = self.kv(i, seq_lens)
            self._wait_aux(i)
            kn, vn = self._append(i, kv, io, append, req_ids, n)
            self._slow_layer(i, L, kv, io, seq_lens, req_ids, n, kn, vn)
        self._leave()

    def fast_step(self, io: StepIO, seq_lens: torch.Tensor, req_ids: Optional[torch.Tensor] = None,
                  append: bool = True, refresh_layers: Sequence[int] = ()):
        """A fast step over all layers. Layers in refresh_layers take the slow path
        instead (dense attention, scores, Selector, compaction): ASPIRE's intra-draft
        refresh layer, which keeps one layer's sparse state current at every step."""
        n = None if req_ids is None else req_ids.numel()
        refresh = set(int(x) for x in refresh_layers)
        self._enter("fast_step")
        for i, L in enumerate(self.layers):
            kv = self.kv(i, seq_lens)
            self._wait_aux(i)
            kn, vn = self._append(i, kv, io, append, req_ids, n)
            if i in refresh:
                self._slow_layer(i, L, kv, io, seq_lens, req_ids, n, kn, vn)
                continue
            self._mark("fast", "start")
            sfi_fast_decode_attn(self.shape, kv, L.compact, self.sink, self.recent, io.q[i], io.out[i],
                                 None if io.lse is None else io.lse[i], k_new=kn, v_new=vn, req_ids=req_ids,
                                 batch=n, max_tokens=self.max_fast_tokens, workspace=self.ws_fast,
                                 dev_status=self.dev_status, stream=self.main, flags=self.step_flags)
            self._mark("fast", "end")
        self._leave()

    def mixed_step(self, io: StepIO, seq_lens: torch.Tensor, slow_ids: torch.Tensor, fast_ids: torch.Tensor):
        """One step where each request is slow or fast (ASPIRE-style mixed batch): one
        attention launch per layer for both kinds (or two with single_launch_mixed off)."""
        ns, nf = slow_ids.numel(), fast_ids.numel()
        self._enter("mixed_step")
        for i, L in enumerate(self.layers):
            kv = self.kv(i, seq_lens)
            self._wait_aux(i)
            kn, vn = self._append(i, kv, io, True, None, None)
            lse = None if io.lse is None else io.lse[i]
            if self.single_launch_mixed:
                self._mark("mixed", "start")
                sfi_mixed_decode_attn(self.shape, kv, L.compact, self.sink, self.recent, io.q[i], io.out[i],
                                      fast_ids, slow_ids, lse=lse, scores=L.scores if ns else None, k_new=kn,
                                      v_new=vn, max_fast_tokens=self.max_fast_tokens,
                                      max_dense_tokens=self.max_dense_tokens, flags=self.attn_flags,
                                      workspace=self.ws_mixed, dev_status=self.dev_status, stream=self.main)
                self._mark("mixed", "end")
            else:
                if nf:
                    sfi_fast_decode_attn(self.shape, kv, L.compact, self.sink, self.recent, io.q[i], io.out[i],
                                         lse, k_new=kn, v_new=vn, req_ids=fast_ids, batch=nf,
                                         max_tokens=self.max_fast_tokens, workspace=self.ws_fast,
                                         dev_status=self.dev_status, stream=self.main, flags=self.step_flags)
                if ns:
                    sfi_slow_dense_attn_with_scores(self.shape, kv, self.sink, self.recent, io.q[i], io.out[i],
                                                    lse, L.scores, k_new=kn, v_new=vn, req_ids=slow_ids, batch=ns,
                                                    max_tokens=self.max_dense_tokens, workspace=self.ws_dense,
                                                    dev_status=self.dev_status, stream=self.main,
                                                    flags=self.step_flags)
            if ns:
                self.e_attn[i].record(self.main)
                self.aux.wait_event(self.e_attn[i])
                self._refresh(i, L, kv, seq_lens, slow_ids, ns)
        self._leave()

    def _multi_workspaces(self):
        if self.ws_multi is None:
            B = self.batch.page_table.shape[0]
            T = SFI_MAX_QUERY_TOKENS
            self.ws_multi = (alloc_multi_workspace(self.shape, B, 1, self.max_dense_tokens, device=self._device),
                             alloc_multi_workspace(self.shape, B, 1, self.max_fast_tokens + T, device=self._device))
        return self.ws_multi

    def verify_step(self, io: StepIO, seq_lens: torch.Tensor, num_tokens: int,
                    req_ids: Optional[torch.Tensor] = None, append: bool = True):
        """Verification of num_tokens drafted tokens over all layers: their K/V go into
        the pages (overwriting the draft's), causal dense attention runs, and each
        layer's score rows receive the recycled statistic. seq_lens count the T tokens.
        The selection is refreshed afterwards, on the accepted lengths, by
        refresh_selection."""
        T, n = int(num_tokens), None if req_ids is None else req_ids.numel()
        ws_v, _ = self._multi_workspaces()
        self._enter("verify_step")
        for i, L in enumerate(self.layers):
            kv = self.kv(i, seq_lens)
            self._wait_aux(i)
            kn, vn = self._append_tokens(i, kv, io, T, append, req_ids, n)
            self._mark("verify", "start")
            sfi_dense_verify_attn(self.shape, kv, self.sink, self.recent, io.q[i], T, io.out[i],
                                  None if io.lse is None else io.lse[i], L.scores, req_ids=req_ids, batch=n,
                                  max_tokens=self.max_dense_tokens, workspace=ws_v, dev_status=self.dev_status,
                                  stream=self.main, flags=self.attn_flags, k_new=kn, v_new=vn)
            self._mark("verify", "end")
        self._leave()

    def refresh_selection(self, seq_lens: torch.Tensor, req_ids: Optional[torch.Tensor] = None):
        """Selector and compaction of every layer from the statistics of the last
        verify_step, at the accepted lengths seq_lens (at most the verified ones), on
        the aux stream; the next use of each layer's compact buffer waits for it."""
        n = None if req_ids is None else req_ids.numel()
        self._enter("refresh_selection")
        self.aux.wait_stream(self.main)
        for i, L in enumerate(self.layers):
            self._refresh(i, L, self.kv(i, seq_lens), seq_lens, req_ids, n)
        self._leave()

    def draft_step(self, io: StepIO, seq_lens: torch.Tensor, num_tokens: int,
                   req_ids: Optional[torch.Tensor] = None, append: bool = True):
        """num_tokens query tokens per request over the sparse state in one pass per
        layer (token t sees what a fast step at length L - T + t + 1 sees); their K/V
        go into the pages first. seq_lens count the T tokens."""
        T, n = int(num_tokens), None if req_ids is None else req_ids.numel()
        _, ws_d = self._multi_workspaces()
        self._enter("draft_step")
        for i, L in enumerate(self.layers):
            kv = self.kv(i, seq_lens)
            self._wait_aux(i)
            kn, vn = self._append_tokens(i, kv, io, T, append, req_ids, n)
            self._mark("draft", "start")
            sfi_sparse_draft_attn(self.shape, kv, L.compact, self.sink, self.recent, io.q[i], T, io.out[i],
                                  None if io.lse is None else io.lse[i], req_ids=req_ids, batch=n,
                                  max_tokens=self.max_fast_tokens + T, workspace=ws_d, dev_status=self.dev_status,
                                  stream=self.main, flags=self.attn_flags, k_new=kn, v_new=vn)
            self._mark("draft", "end")
        self._leave()

    def dense_step(self, io: StepIO, seq_lens: torch.Tensor, append: bool = True):
        """Full-KV decode step (the baseline of the paper's Table 1)."""
        self._enter("dense_step")
        for i, L in enumerate(self.layers):
            kv = self.kv(i, seq_lens)
            kn, vn = self._append(i, kv, io, append, None, None)
            self._mark("dense", "start")
            sfi_slow_dense_attn_with_scores(self.shape, kv, self.sink, self.recent, io.q[i], io.out[i],
                                            None if io.lse is None else io.lse[i], None, k_new=kn, v_new=vn,
                                            max_tokens=self.max_dense_tokens, workspace=self.ws_dense,
                                            dev_status=self.dev_status, stream=self.main, flags=self.step_flags)
            self._mark("dense", "end")
        self._leave()

    def join(self):
        """Make the main stream (and the caller's stream) wait for all outstanding aux work."""
        for i in range(len(self.layers)):
            self._wait_aux(i)
        self._leave(close_range=False)
