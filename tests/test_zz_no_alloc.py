"""The allocation-free fast step (sfi_fast_decode_attn_noalloc) against the regular one.

Some callers cannot allocate device memory (a plugin inside a host application that
owns every device allocation, or a latency-critical path that must not call
cudaMalloc), so they cannot hand sfi_fast_decode_attn a workspace. The no-alloc
entry point keeps the split-KV scratch in a fixed array inside the library instead.
This test calls it through the C ABI twice in a row, with different queries, and
checks each result against the regular entry point (with a workspace) within the
parity tolerance. The split count is forced high enough that the scratch is used.
This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import sfi_synth as syn
from tests.gpu_harness import Problem, assert_close, dev_bf16, dev_i32

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
    return comp


def test_noalloc_fast_step_matches_regular_entry_point_on_two_calls():
    sfi = _setup()
    # 12 splits: more than fit in one thread-block cluster, so the partial results go
    # through the scratch (plans of up to 8 splits merge in shared memory and need none)
    S, W, k, splits = 4, 32, 1536, 12
    prob = Problem(seed=901, lens=[4096, 3000, 2000, 1600], Hq=16, Hkv=8, D=128, S=S, W=W,
                   heavy_frac=0.02).to_device()
    comp = _filled_compact(sfi, prob, k)
    max_tokens = S + k + W + 32
    assert sfi.sfi_plan_splits(prob.shape, prob.B, max_tokens, splits) == splits
    assert 0 < sfi.sfi_workspace_size(prob.shape, prob.B, max_tokens, splits) <= (4 << 20)
    g = syn.rng(902, 1)
    for call in range(2):
        q = prob.d_q if call == 0 else dev_bf16(syn.normal_bf16(g, (prob.B, prob.Hq, prob.D)))
        ref_out = torch.full((prob.B, prob.Hq, prob.D), float("nan"), device="cuda")
        ref_lse = torch.full((prob.B, prob.Hq), float("nan"), device="cuda")
        ws = sfi.alloc_workspace(prob.shape, prob.B, max_tokens, splits)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        sfi.sfi_fast_decode_attn(prob.shape, prob.d_kv, comp, S, W, q, ref_out, ref_lse, max_tokens=max_tokens,
                                 num_splits=splits, workspace=ws, dev_status=st)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        sfi.sfi_fast_decode_attn_noalloc(prob.shape, prob.d_kv, comp, S, W, q, out, lse, max_tokens=max_tokens,
                                         num_splits=splits, dev_status=st)
        torch.cuda.synchronize()
        assert st.item() == 0, f"call {call}: device status {st.item()}"
        assert_close(out.cpu().numpy(), ref_out.cpu().numpy(), f"call {call} out")
        assert_close(lse.cpu().numpy(), ref_lse.cpu().numpy(), f"call {call} lse")
        assert np.isfinite(out.cpu().numpy()).all()


def test_noalloc_rejects_plans_larger_than_its_scratch():
    sfi = _setup()
    prob = Problem(seed=903, lens=[64] * 16, Hq=16, Hkv=8, D=128, S=4, W=32).to_device()
    comp = _filled_compact(sfi, prob, 8)
    out = torch.empty((16, 16, 128), device="cuda")
    assert sfi.sfi_workspace_size(prob.shape, 16, 65536, 256) > (4 << 20)
    with pytest.raises(sfi.SFIError) as exc:
        sfi.sfi_fast_decode_attn_noalloc(prob.shape, prob.d_kv, comp, 4, 32, prob.d_q, out, None,
                                         max_tokens=65536, num_splits=256)
    assert exc.value.status == 3  # SFI_ERR_WORKSPACE
