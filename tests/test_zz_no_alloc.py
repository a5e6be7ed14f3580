"""The allocation-free fast step (sfi_fast_decode_attn_noalloc) against the regular one.

Some callers cannot allocate device memory (a plugin inside a host application that
owns every device allocation, or a latency-critical path that must not call
cudaMalloc), so they cannot hand sfi_fast_decode_attn a workspace. The no-alloc
entry point keeps the split-KV scratch in a fixed array inside the library instead.
These tests call it through the C ABI twice in a row, with different queries, and
check each result against the regular entry point (with a workspace) within the
parity tolerance, and against the CPU oracle. The split count is forced high enough
that the scratch is used. A call whose bounded wait runs out must leave the shared
scratch usable for the next call, with and without SFI_ATTN_RAGGED (whose chunked
plan lays the scratch out differently). This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import oracle
import sfi_synth as syn
from tests.gpu_harness import (Problem, assert_close, dev_bf16, dev_i32, oracle_compact_request,
                               run_oracle_selection)

pytestmark = pytest.mark.gpu


def _setup():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from sparse_kv_long_sfi_gb300 import build
    build.build()
    import sparse_kv_long_sfi_gb300 as sfi
    return sfi


def _filled_compact(sfi, prob, k):
    """Slow step, Selector and compaction with the regular entry points."""
    S, W = prob.S, prob.W
    B = prob.B
    stride = int(prob.lens.max())
    scores = torch.empty((B, prob.Hkv, stride), device="cuda")
    out = torch.empty((B, prob.Hq, prob.D), device="cuda")
    ws = sfi.alloc_workspace(prob.shape, B, stride + 16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sfi.sfi_slow_dense_attn_with_scores(prob.shape, prob.d_kv, S, W, prob.d_q, out, None, scores,
                                        max_tokens=stride + 16, workspace=ws, dev_status=st)
    off, cap = sfi.compact_layout(prob.shape, S, [k] * B)
    rows = int((off[-1] + prob.Hkv * cap[-1]).item())
    comp = sfi.CompactKV(torch.zeros((rows, prob.D), dtype=torch.bfloat16, device="cuda"),
                         torch.zeros((rows, prob.D), dtype=torch.bfloat16, device="cuda"), off, cap,
                         torch.zeros(B, dtype=torch.int32, device="cuda"))
    idx = torch.zeros((B, prob.Hkv, k), dtype=torch.int32, device="cuda")
    sfi.sfi_select_topk(scores, prob.Hkv, prob.d_kv.seq_lens, S, W, dev_i32([k] * B), idx, comp.count,
                        dev_status=st)
    sfi.sfi_compact_gather(prob.shape, prob.d_kv, idx, comp.count, S, comp, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return comp, scores.cpu().numpy()


def _oracle_fast(prob, q_host, scores_host, k):
    """The oracle's fast step for every request, from the oracle's own selection over the
    GPU-written scores (the bytes the GPU Selector ranked)."""
    oracle.build()
    S, W = prob.S, prob.W
    ref_idx, ref_count = run_oracle_selection(prob, scores_host, [k] * prob.B, k)
    outs, lses = [], []
    for r in range(prob.B):
        rk, rv = oracle_compact_request(prob, r, ref_idx[r], ref_count[r], S + k)
        o, l = oracle.fast_attn(q_host[r], rk, rv, ref_count[r], prob.kv.k_pool, prob.kv.v_pool,
                                prob.kv.page_table[r], prob.lens[r], S, W, prob.Hq, prob.Hkv, prob.D, 16)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def _regular_and_noalloc(sfi, prob, comp, q, max_tokens, splits, flags):
    """The fast step through the regular entry point (own zeroed workspace) and the
    no-alloc one, on the same inputs; returns both (out, lse) pairs on the host."""
    ref_out = torch.full((prob.B, prob.Hq, prob.D), float("nan"), device="cuda")
    ref_lse = torch.full((prob.B, prob.Hq), float("nan"), device="cuda")
    ragged = bool(flags & sfi.SFI_ATTN_RAGGED)
    ws = (sfi.alloc_ragged_workspace(prob.shape, prob.B, max_tokens) if ragged
          else sfi.alloc_workspace(prob.shape, prob.B, max_tokens, splits))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sfi.sfi_fast_decode_attn(prob.shape, prob.d_kv, comp, prob.S, prob.W, q, ref_out, ref_lse,
                             max_tokens=max_tokens, num_splits=splits, workspace=ws, dev_status=st, flags=flags)
    out = torch.full_like(ref_out, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    sfi.sfi_fast_decode_attn_noalloc(prob.shape, prob.d_kv, comp, prob.S, prob.W, q, out, lse,
                                     max_tokens=max_tokens, num_splits=splits, dev_status=st, flags=flags)
    torch.cuda.synchronize()
    assert st.item() == 0, f"device status {st.item()}"
    return (out.cpu().numpy(), lse.cpu().numpy()), (ref_out.cpu().numpy(), ref_lse.cpu().numpy())


def _problem(sfi, seed):
    # k = 1536 over four requests: 12 splits are more than fit in one thread-block
    # cluster, so the partial results go through the scratch (plans of up to 8 splits
    # merge in shared memory and need none)
    S, W, k, splits = 4, 32, 1536, 12
    prob = Problem(seed=seed, lens=[4096, 3000, 2000, 1600], Hq=16, Hkv=8, D=128, S=S, W=W,
                   heavy_frac=0.02).to_device()
    comp, scores = _filled_compact(sfi, prob, k)
    max_tokens = S + k + W + 32
    assert sfi.sfi_plan_splits(prob.shape, prob.B, max_tokens, splits) == splits
    assert 0 < sfi.sfi_workspace_size(prob.shape, prob.B, max_tokens, splits) <= (4 << 20)
    assert 0 < sfi.sfi_mixed_workspace_size(prob.shape, prob.B, 0, max_tokens, 0) <= (4 << 20)
    return prob, comp, scores, k, splits, max_tokens


@pytest.mark.parametrize("ragged", [False, True], ids=["split-plan", "ragged-plan"])
def test_noalloc_fast_step_matches_regular_entry_point_on_two_calls(ragged):
    sfi = _setup()
    prob, comp, scores, k, splits, max_tokens = _problem(sfi, 901)
    flags = sfi.SFI_ATTN_RAGGED if ragged else 0
    g = syn.rng(902, 1)
    for call in range(2):
        q_host = prob.q if call == 0 else syn.normal_bf16(g, (prob.B, prob.Hq, prob.D))
        q = prob.d_q if call == 0 else dev_bf16(q_host)
        (out, lse), (ref_out, ref_lse) = _regular_and_noalloc(sfi, prob, comp, q, max_tokens, splits, flags)
        assert_close(out, ref_out, f"call {call} out vs the regular entry point")
        assert_close(lse, ref_lse, f"call {call} lse vs the regular entry point")
        o_ref, l_ref = _oracle_fast(prob, q_host, scores, k)
        assert_close(out, o_ref, f"call {call} out vs the oracle")
        assert_close(lse, l_ref, f"call {call} lse vs the oracle")


@pytest.mark.parametrize("ragged", [False, True], ids=["split-plan", "ragged-plan"])
def test_noalloc_recovers_after_a_timed_out_call(ragged):
    """A no-alloc call whose bounded wait runs out (SFI_ATTN_TEST_WITHHOLD: every CTA's
    producer withholds its second stage, so the consumers give up after about 2 s)
    reports SFI_DEV_TIMEOUT and writes no output; the next no-alloc call on the same
    scratch is correct."""
    sfi = _setup()
    prob, comp, scores, k, splits, max_tokens = _problem(sfi, 905)
    flags = sfi.SFI_ATTN_RAGGED if ragged else 0
    out = torch.full((prob.B, prob.Hq, prob.D), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sfi.sfi_fast_decode_attn_noalloc(prob.shape, prob.d_kv, comp, prob.S, prob.W, prob.d_q, out, None,
                                     max_tokens=max_tokens, num_splits=splits, dev_status=st,
                                     flags=flags | sfi.SFI_ATTN_TEST_WITHHOLD)
    torch.cuda.synchronize()
    assert st.item() & 16, f"status {st.item()}"  # SFI_DEV_TIMEOUT
    assert np.isnan(out.cpu().numpy()).all(), "a timed-out call writes no output"
    (out, lse), (ref_out, ref_lse) = _regular_and_noalloc(sfi, prob, comp, prob.d_q, max_tokens, splits, flags)
    assert_close(out, ref_out, "after the timeout: out vs the regular entry point")
    assert_close(lse, ref_lse, "after the timeout: lse vs the regular entry point")


def test_noalloc_rejects_plans_larger_than_its_scratch():
    sfi = _setup()
    prob = Problem(seed=903, lens=[64] * 16, Hq=16, Hkv=8, D=128, S=4, W=32).to_device()
    comp, _ = _filled_compact(sfi, prob, 8)
    out = torch.empty((16, 16, 128), device="cuda")
    assert sfi.sfi_workspace_size(prob.shape, 16, 65536, 256) > (4 << 20)
    with pytest.raises(sfi.SFIError) as exc:
        sfi.sfi_fast_decode_attn_noalloc(prob.shape, prob.d_kv, comp, 4, 32, prob.d_q, out, None,
                                         max_tokens=65536, num_splits=256)
    assert exc.value.status == 3  # SFI_ERR_WORKSPACE
