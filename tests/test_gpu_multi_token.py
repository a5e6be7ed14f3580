"""GPU parity of the multi-token calls ("A Sparse Glimpse of the Whole: Train-Free
Self-Speculative Decoding", abstract: drafts over the sparse, recallable state and a
full-context verification whose statistics are recycled) through the C ABI, against
the CPU oracle on the same seeded inputs: the T-token append bit-exact, verification
and multi-token drafting within |gpu - oracle| <= 2e-3 + 1e-2 |oracle|, the recycled
statistic within the fp32 dot-product bound."""
import math

import numpy as np
import pytest
import torch

import oracle
import sfi_synth as syn
from tests.gpu_harness import (Problem, assert_close, dev_bf16, dev_i32, host_bf16, oracle_compact_request,
                               run_oracle_selection)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from sparse_kv_long_sfi_gb300 import build
    build.build()
    oracle.build()


def _sfi():
    import sparse_kv_long_sfi_gb300 as sfi
    return sfi


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _queries(seed, B, T, Hq, D):
    return syn.normal_bf16(syn.rng(400, seed), (B, T, Hq, D))


def _verify(prob, q, T, num_splits=0, scores=None, req_ids=None):
    sfi = _sfi()
    B = prob.B
    out = torch.full((B, T, prob.Hq, prob.D), float("nan"), device="cuda")
    lse = torch.full((B, T, prob.Hq), float("nan"), device="cuda")
    maxL = int(prob.lens.max()) + 16
    ws = sfi.alloc_multi_workspace(prob.shape, B, T, maxL, num_splits)
    st = _status()
    sfi.sfi_dense_verify_attn(prob.shape, prob.d_kv, prob.S, prob.W, dev_bf16(q), T, out, lse, scores,
                              req_ids=None if req_ids is None else dev_i32(req_ids), max_tokens=maxL,
                              num_splits=num_splits, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert not ws[:4 * B * prob.Hkv].any(), "split counters must be left zeroed"
    return out.cpu().numpy(), lse.cpu().numpy()


def test_append_tokens_bit_exact():
    sfi = _sfi()
    T = 5
    prob = Problem(seed=501, lens=[40, 16, 11, 100], Hq=8, Hkv=2, D=128, S=4, W=32, extra_tokens=T).to_device()
    g = syn.rng(401, 1)
    kn, vn = syn.normal_bf16(g, (4, T, 2, 128)), syn.normal_bf16(g, (4, T, 2, 128))
    new_lens = prob.lens + T
    prob.set_lens(new_lens)
    st = _status()
    sfi.sfi_paged_kv_append_tokens(prob.shape, prob.d_kv, dev_bf16(kn), dev_bf16(vn), T, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    kp, vp = prob.kv.k_pool.copy(), prob.kv.v_pool.copy()
    for r in range(4):
        oracle.paged_append_tokens(kp, vp, prob.kv.page_table[r], new_lens[r], T, kn[r], vn[r], 2, 128, 16)
    np.testing.assert_array_equal(host_bf16(prob.d_kv.k_pool), kp)
    np.testing.assert_array_equal(host_bf16(prob.d_kv.v_pool), vp)


@pytest.mark.parametrize("D,Hq,Hkv,T", [(128, 16, 8, 8), (128, 32, 8, 4), (128, 64, 8, 2), (64, 8, 2, 3),
                                        (128, 8, 8, 16), (128, 16, 8, 1), (128, 16, 8, 5)])
@pytest.mark.parametrize("splits", [1, 3, 0, 12])
def test_verify_matches_oracle(D, Hq, Hkv, T, splits):
    lens = sorted({T, T + 1, 15 + T, 16, 17 + T, 100, 777, 1500})
    lens = [L for L in lens if L >= T]
    prob = Problem(seed=D * 1000 + Hq * 10 + T + splits, lens=lens, Hq=Hq, Hkv=Hkv, D=D, S=4, W=32).to_device()
    q = _queries(D + Hq + T, prob.B, T, Hq, D)
    out, lse = _verify(prob, q, T, num_splits=splits)
    for r in range(prob.B):
        o_ref, l_ref = oracle.verify_attn(q[r], prob.kv.k_pool, prob.kv.v_pool, prob.kv.page_table[r], prob.lens[r],
                                          T, Hq, Hkv, D, 16)
        assert_close(out[r], o_ref, f"verify out r={r}")
        assert_close(lse[r], l_ref, f"verify lse r={r}")


def _verify_score_bound(prob, q, r, T, stride):
    """fp32 bound per statistic: 2 * (T*G) * D * 2^-24 * sum over the rows of |scale q k|."""
    L = int(prob.lens[r])
    scale = 1.0 / math.sqrt(prob.D)
    out = np.zeros((prob.Hkv, stride))
    qa = np.abs(syn.bf16_values(q[r]))  # [T][Hq][D]
    for kvh in range(prob.Hkv):
        rows = np.stack([np.abs(syn.bf16_values(
            prob.kv.k_pool[prob.kv.page_table[r, j // 16], kvh, j % 16])) for j in range(L)])
        qg = qa[:, kvh * prob.G:(kvh + 1) * prob.G].reshape(-1, prob.D)
        mag = (rows @ qg.T).sum(1) * scale
        out[kvh, :L] = 2 * T * prob.G * prob.D * 2.0 ** -24 * mag + 1e-30
    return out


@pytest.mark.parametrize("T,W", [(5, 2), (4, 32), (8, 0)])
def test_verify_statistic_matches_oracle_within_fp32_bound(T, W):
    prob = Problem(seed=510 + T, lens=[37, 300, 1024, 1031, T + 5], Hq=16, Hkv=8, D=128, S=4, W=W,
                   heavy_frac=0.04).to_device()
    q = _queries(510 + T, prob.B, T, 16, 128)
    stride = 1040
    scores = torch.full((prob.B, prob.Hkv, stride), float("nan"), device="cuda")
    out, lse = _verify(prob, q, T, scores=scores)
    sc = scores.cpu().numpy()
    for r in range(prob.B):
        L = int(prob.lens[r])
        ref = oracle.verify_scores(q[r], prob.kv.k_pool, prob.kv.page_table[r], L, T, prob.S, W, 16, 8, 128, 16,
                                   stride=stride)
        bound = _verify_score_bound(prob, q, r, T, stride)
        assert np.isnan(sc[r, :, L:]).all(), "entries at j >= L must not be written"
        masked = np.isneginf(ref[:, :L])
        assert np.array_equal(np.isneginf(sc[r, :, :L]), masked)
        err = np.abs(sc[r, :, :L][~masked].astype(np.float64) - ref[:, :L][~masked])
        assert (err <= bound[:, :L][~masked]).all(), err.max()
        o_ref, l_ref = oracle.verify_attn(q[r], prob.kv.k_pool, prob.kv.v_pool, prob.kv.page_table[r], L, T, 16, 8,
                                          128, 16)
        assert_close(out[r], o_ref, f"out r={r}")


def test_verify_subset_of_requests():
    T = 4
    prob = Problem(seed=520, lens=[300, 1024, 64, 900], Hq=16, Hkv=8, D=128, S=4, W=32).to_device()
    q = _queries(520, prob.B, T, 16, 128)
    out, _ = _verify(prob, q, T, req_ids=[3, 1])
    for r in (3, 1):
        o_ref, _ = oracle.verify_attn(q[r], prob.kv.k_pool, prob.kv.v_pool, prob.kv.page_table[r], prob.lens[r], T,
                                      16, 8, 128, 16)
        assert_close(out[r], o_ref, f"out r={r}")
    assert np.isnan(out[[0, 2]]).all()


def _compact_buffers(prob, k_per_req):
    sfi = _sfi()
    off, cap = sfi.compact_layout(prob.shape, prob.S, k_per_req)
    rows = int((off[-1] + prob.Hkv * cap[-1]).item())
    ck = torch.zeros((rows, prob.D), dtype=torch.bfloat16, device="cuda")
    cv = torch.zeros_like(ck)
    count = torch.zeros(prob.B, dtype=torch.int32, device="cuda")
    return sfi.CompactKV(ck, cv, off, cap, count)


def _draft_case(seed, lens_slow, Hq, Hkv, D, S, W, T, k_per_req, k_cap, splits=0, req_ids=None):
    """Slow step + Selector + compaction at lens_slow, T tokens appended, then one multi-token draft pass."""
    sfi = _sfi()
    prob = Problem(seed=seed, lens=lens_slow, Hq=Hq, Hkv=Hkv, D=D, S=S, W=W, extra_tokens=T,
                   heavy_frac=0.02).to_device()
    stride = int(max(lens_slow))
    scores = torch.full((prob.B, Hkv, stride), float("nan"), device="cuda")
    st = _status()
    ws1 = sfi.alloc_workspace(prob.shape, prob.B, stride + 16)
    o1 = torch.empty((prob.B, Hq, D), device="cuda")
    sfi.sfi_slow_dense_attn_with_scores(prob.shape, prob.d_kv, S, W, prob.d_q, o1, None, scores,
                                        max_tokens=stride + 16, workspace=ws1, dev_status=st)
    comp = _compact_buffers(prob, k_per_req)
    idx = torch.zeros((prob.B, Hkv, k_cap), dtype=torch.int32, device="cuda")
    sfi.sfi_select_topk(scores, Hkv, prob.d_kv.seq_lens, S, W, dev_i32(k_per_req), idx, comp.count, dev_status=st)
    sfi.sfi_compact_gather(prob.shape, prob.d_kv, idx, comp.count, S, comp, dev_status=st)
    torch.cuda.synchronize()
    sc = scores.cpu().numpy()
    ref_idx, ref_count = run_oracle_selection(prob, sc, k_per_req, k_cap)
    cap = comp.capacity.cpu().numpy()
    ref_compact = [oracle_compact_request(prob, r, ref_idx[r], ref_count[r], cap[r]) for r in range(prob.B)]
    # T drafted tokens enter the cache, then one pass over the sparse state
    g = syn.rng(402, seed)
    kn, vn = syn.normal_bf16(g, (prob.B, T, Hkv, D)), syn.normal_bf16(g, (prob.B, T, Hkv, D))
    lens = prob.lens + T
    prob.set_lens(lens)
    sfi.sfi_paged_kv_append_tokens(prob.shape, prob.d_kv, dev_bf16(kn), dev_bf16(vn), T, dev_status=st)
    for r in range(prob.B):
        oracle.paged_append_tokens(prob.kv.k_pool, prob.kv.v_pool, prob.kv.page_table[r], lens[r], T, kn[r], vn[r],
                                   Hkv, D, 16)
    q = _queries(seed, prob.B, T, Hq, D)
    out = torch.full((prob.B, T, Hq, D), float("nan"), device="cuda")
    lse = torch.full((prob.B, T, Hq), float("nan"), device="cuda")
    max_tokens = S + k_cap + W + T + 32
    ws = sfi.alloc_multi_workspace(prob.shape, prob.B, T, max_tokens, splits)
    sfi.sfi_sparse_draft_attn(prob.shape, prob.d_kv, comp, S, W, dev_bf16(q), T, out, lse,
                              req_ids=None if req_ids is None else dev_i32(req_ids), max_tokens=max_tokens,
                              num_splits=splits, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert not ws[:4 * prob.B * Hkv].any()
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    for r in (range(prob.B) if req_ids is None else req_ids):
        rk, rv = ref_compact[r]
        o_ref, l_ref = oracle.fast_multi_attn(q[r], rk, rv, ref_count[r], prob.kv.k_pool, prob.kv.v_pool,
                                              prob.kv.page_table[r], lens[r], T, S, W, Hq, Hkv, D, 16)
        assert_close(o[r], o_ref, f"draft out r={r}")
        assert_close(l[r], l_ref, f"draft lse r={r}")
    if req_ids is not None:
        assert np.isnan(o[sorted(set(range(prob.B)) - set(req_ids))]).all()


@pytest.mark.parametrize("splits", [1, 2, 5, 0, 12])
def test_draft_matches_oracle(splits):
    lens = [1024, 1031, 530, 36, 30, 4, 17]
    _draft_case(530 + splits, lens, 16, 8, 128, 4, 32, 4, [64, 64, 100, 5, 5, 5, 5], 128, splits=splits)


@pytest.mark.parametrize("T,W", [(6, 3), (8, 0), (1, 32)])
def test_draft_windows_shorter_than_the_draft(T, W):
    """Token windows that do not overlap the first token's (W < T) and W = 0 (sink + selection only)."""
    lens = [700, 333, 64, 20]
    _draft_case(540 + T, lens, 16, 8, 128, 4, W, T, [40, 40, 20, 3], 64)


def test_draft_d64_g4_and_subset():
    _draft_case(550, [1024, 600, 1100, 900], 8, 2, 64, 4, 32, 4, [64, 64, 64, 64], 64, req_ids=[2, 0])


def test_draft_g8_two_tokens():
    _draft_case(560, [1500, 800, 47], 64, 8, 128, 4, 32, 2, [100, 50, 5], 128, splits=3)


@pytest.mark.parametrize("T,splits,flags", [(4, 0, 0), (8, 3, 1), (3, 12, 1), (16, 1, 0)])
def test_verify_with_fused_append_matches_oracle(T, splits, flags):
    """k_new/v_new given to the verification: it equals the T-token append followed by the
    verification, pages included, with and without early KV prefetch."""
    _verify_fused_case(T, splits, flags, [300, 1023, 17, 40])


@pytest.mark.parametrize("T,splits,D", [(8, 2, 128), (8, 3, 128), (16, 2, 128), (8, 2, 64), (4, 12, 64)])
def test_verify_fused_append_across_splits(T, splits, D):
    """Query tokens that straddle a page boundary and a split boundary of a short request:
    the first split of a cluster appends its part straight from global memory (its receive
    region takes the other splits' partials), the later ones from shared-memory staging;
    at D = 64 too, and with the workspace merge (12 splits)."""
    _verify_fused_case(T, splits, 1, [10, 13, 5, 2] if splits <= 3 else [300, 1023, 17, 40], D=D)


def _verify_fused_case(T, splits, flags, lens0, D=128):
    sfi = _sfi()
    Hq, Hkv = (8, 8) if T == 16 else (16, 8)
    prob = Problem(seed=800 + T, lens=lens0, Hq=Hq, Hkv=Hkv, D=D, S=4, W=32,
                   extra_tokens=T).to_device()
    g = syn.rng(403, T)
    kn, vn = syn.normal_bf16(g, (prob.B, T, Hkv, D)), syn.normal_bf16(g, (prob.B, T, Hkv, D))
    lens = prob.lens + T
    prob.set_lens(lens)
    q = _queries(810 + T, prob.B, T, Hq, D)
    stride = int(lens.max())
    scores = torch.full((prob.B, Hkv, stride), float("nan"), device="cuda")
    out = torch.full((prob.B, T, Hq, D), float("nan"), device="cuda")
    maxL = stride + 16
    ws = sfi.alloc_multi_workspace(prob.shape, prob.B, T, maxL, splits)
    st = _status()
    sfi.sfi_dense_verify_attn(prob.shape, prob.d_kv, prob.S, prob.W, dev_bf16(q), T, out, None, scores,
                              max_tokens=maxL, num_splits=splits, workspace=ws, dev_status=st, flags=flags,
                              k_new=dev_bf16(kn), v_new=dev_bf16(vn))
    torch.cuda.synchronize()
    assert st.item() == 0
    for r in range(prob.B):
        oracle.paged_append_tokens(prob.kv.k_pool, prob.kv.v_pool, prob.kv.page_table[r], lens[r], T, kn[r], vn[r],
                                   Hkv, D, 16)
    np.testing.assert_array_equal(host_bf16(prob.d_kv.k_pool), prob.kv.k_pool)
    np.testing.assert_array_equal(host_bf16(prob.d_kv.v_pool), prob.kv.v_pool)
    o, sc = out.cpu().numpy(), scores.cpu().numpy()
    for r in range(prob.B):
        o_ref, _ = oracle.verify_attn(q[r], prob.kv.k_pool, prob.kv.v_pool, prob.kv.page_table[r], lens[r], T, Hq, Hkv,
                                      D, 16)
        assert_close(o[r], o_ref, f"out r={r}")
        ref = oracle.verify_scores(q[r], prob.kv.k_pool, prob.kv.page_table[r], lens[r], T, prob.S, prob.W, Hq, Hkv,
                                   D, 16, stride=stride)
        L = lens[r]
        assert np.array_equal(np.isneginf(sc[r, :, :L]), np.isneginf(ref[:, :L]))


@pytest.mark.parametrize("T,flags", [(4, 1), (8, 0), (1, 1)])
def test_draft_with_fused_append_matches_oracle(T, flags):
    """k_new/v_new given to the draft pass: equals the T-token append followed by the draft
    (T = 1 runs the single-token fast-step kernel)."""
    sfi = _sfi()
    S, W, Hq, Hkv, D = 4, 32, 16, 8, 128
    lens_slow = [1024, 530, 36]
    k_per_req, k_cap = [64, 100, 5], 128
    prob = Problem(seed=820 + T, lens=lens_slow, Hq=Hq, Hkv=Hkv, D=D, S=S, W=W, extra_tokens=T,
                   heavy_frac=0.02).to_device()
    stride = int(max(lens_slow))
    scores = torch.full((prob.B, Hkv, stride), float("nan"), device="cuda")
    st = _status()
    ws1 = sfi.alloc_workspace(prob.shape, prob.B, stride + 16)
    o1 = torch.empty((prob.B, Hq, D), device="cuda")
    sfi.sfi_slow_dense_attn_with_scores(prob.shape, prob.d_kv, S, W, prob.d_q, o1, None, scores,
                                        max_tokens=stride + 16, workspace=ws1, dev_status=st)
    comp = _compact_buffers(prob, k_per_req)
    idx = torch.zeros((prob.B, Hkv, k_cap), dtype=torch.int32, device="cuda")
    sfi.sfi_select_compact(prob.shape, prob.d_kv, scores, S, W, dev_i32(k_per_req), idx, comp, dev_status=st)
    torch.cuda.synchronize()
    ref_idx, ref_count = run_oracle_selection(prob, scores.cpu().numpy(), k_per_req, k_cap)
    cap = comp.capacity.cpu().numpy()
    ref_compact = [oracle_compact_request(prob, r, ref_idx[r], ref_count[r], cap[r]) for r in range(prob.B)]
    g = syn.rng(404, T)
    kn, vn = syn.normal_bf16(g, (prob.B, T, Hkv, D)), syn.normal_bf16(g, (prob.B, T, Hkv, D))
    lens = prob.lens + T
    prob.set_lens(lens)
    q = _queries(830 + T, prob.B, T, Hq, D)
    out = torch.full((prob.B, T, Hq, D), float("nan"), device="cuda")
    max_tokens = S + k_cap + W + T + 32
    ws = sfi.alloc_multi_workspace(prob.shape, prob.B, T, max_tokens)
    sfi.sfi_sparse_draft_attn(prob.shape, prob.d_kv, comp, S, W, dev_bf16(q), T, out, None, max_tokens=max_tokens,
                              workspace=ws, dev_status=st, flags=flags, k_new=dev_bf16(kn), v_new=dev_bf16(vn))
    torch.cuda.synchronize()
    assert st.item() == 0
    for r in range(prob.B):
        oracle.paged_append_tokens(prob.kv.k_pool, prob.kv.v_pool, prob.kv.page_table[r], lens[r], T, kn[r], vn[r],
                                   Hkv, D, 16)
    np.testing.assert_array_equal(host_bf16(prob.d_kv.k_pool), prob.kv.k_pool)
    o = out.cpu().numpy()
    for r in range(prob.B):
        rk, rv = ref_compact[r]
        o_ref, _ = oracle.fast_multi_attn(q[r], rk, rv, ref_count[r], prob.kv.k_pool, prob.kv.v_pool,
                                          prob.kv.page_table[r], lens[r], T, S, W, Hq, Hkv, D, 16)
        assert_close(o[r], o_ref, f"draft out r={r}")


@pytest.mark.parametrize("splits", [16, 32])
def test_verify_and_draft_many_splits(splits):
    """Multi-token passes split 16 and 32 ways (merged from the workspace)."""
    D, Hq, Hkv, T = 128, 16, 8, 4
    lens = [8200, 6600, 5000]
    prob = Problem(seed=90 + splits, lens=lens, Hq=Hq, Hkv=Hkv, D=D, S=4, W=32).to_device()
    q = _queries(91 + splits, prob.B, T, Hq, D)
    out, lse = _verify(prob, q, T, num_splits=splits)
    for r in range(prob.B):
        o_ref, l_ref = oracle.verify_attn(q[r], prob.kv.k_pool, prob.kv.v_pool, prob.kv.page_table[r], prob.lens[r],
                                          T, Hq, Hkv, D, 16)
        assert_close(out[r], o_ref, f"verify out r={r}")
        assert_close(lse[r], l_ref, f"verify lse r={r}")
    _draft_case(95 + splits, lens, Hq, Hkv, D, 4, 32, T, [4300, 4100, 4200], 4300, splits=splits)
