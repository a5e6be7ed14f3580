"""GPU parity: every CUDA entry point, called through the C ABI, against the CPU oracle
on the same seeded inputs. Attention within |gpu - oracle| <= 2e-3 + 1e-2 |oracle|;
scores within the fp32 dot-product bound; selection, compaction and append bit-exact
(selection is checked by running the oracle's Selector on the GPU-written fp32
scores, the same bytes the kernel ranked)."""
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


def counters_zero(ws, units):
    """The split-merge counters (one int32 per (request, KV head) at the start of the
    workspace) are back to zero after a launch."""
    return not ws[:4 * units].any()


def _dense(prob, num_splits=0, scores=None, req_ids=None, ragged=False, max_tokens=None):
    sfi = _sfi()
    B = prob.B
    out = torch.full((B, prob.Hq, prob.D), float("nan"), device="cuda")
    lse = torch.full((B, prob.Hq), float("nan"), device="cuda")
    maxL = int(prob.lens.max()) + 16 if max_tokens is None else max_tokens
    if ragged:
        ws = sfi.alloc_ragged_workspace(prob.shape, B, maxL, dense=True)
    else:
        ws = sfi.alloc_workspace(prob.shape, B, maxL, num_splits)
    st = _status()
    sfi.sfi_slow_dense_attn_with_scores(prob.shape, prob.d_kv, prob.S, prob.W, prob.d_q, out, lse, scores,
                                        req_ids=req_ids, max_tokens=maxL, num_splits=num_splits, workspace=ws,
                                        dev_status=st, flags=sfi.SFI_ATTN_RAGGED if ragged else 0)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert counters_zero(ws, B * prob.Hkv), "split counters must be left zeroed"
    return out.cpu().numpy(), lse.cpu().numpy()


# ---------------------------------------------------------------------------
# Dense / slow-step attention
# ---------------------------------------------------------------------------
def test_automatic_split_plans():
    """The automatic plans on this GPU: about 85% of one wave of two CTAs per SM (8 when
    that lands between 8 and 16), never fewer than three stages (12 sub-blocks) per split
    while the splits merge inside a cluster and four (16 sub-blocks) beyond it, and a
    cluster plan leaves a ninth of the SM slots free in whole clusters; the workspace
    follows the plans of every batch size up to the given one (none when all of them
    merge inside a cluster)."""
    sfi = _sfi()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    shape = sfi.AttnShape(16, 8, 128)
    cap = {c: sfi.sfi_attn_cluster_capacity(c) for c in range(1, 9)}
    assert cap[1] == 2 * sms  # two CTAs per SM
    for c in range(2, 9):  # whole clusters never hold more CTAs than the SM slots
        assert 0 < cap[c] * c <= 2 * sms, (c, cap[c])

    def plan(batch, L):
        units, nb = batch * 8, (L + 15) // 16 + 1
        s = max(1, sms * 2 * 17 // 20 // units)
        if 8 < s < 16:
            s = 8
        s = max(1, min(s, max(nb // 16, min(8, -(-nb // 12))), 256))
        while 1 < s <= 8 and (cap[s] - units) * s < sms * 2 // 9:
            s -= 1
        return s

    assert plan(1, 1056) == 6 and plan(16, 16400) == 2  # the two workloads of the decode step
    for batch in (1, 2, 3, 4, 5, 8, 16, 64):
        for L in (150, 1040, 1500, 2100, 16400, 65600):
            assert sfi.sfi_plan_splits(shape, batch, L, 0) == plan(batch, L), (batch, L)
            needs = any(plan(b, L) > 8 for b in range(1, batch + 1))
            assert (sfi.sfi_workspace_size(shape, batch, L, 0) > 0) == needs, (batch, L)


@pytest.mark.parametrize("ragged", [False, True])
def test_workspace_shared_by_calls_of_different_batch_sizes(ragged):
    """One workspace, sized for 12 requests, serves calls on subsets of 3, 12, 5 and 12
    requests in turn: each call's partial states stay clear of the split counters of
    every other call (counters at the start, partial states at the end of the buffer),
    so every output matches the oracle and the counters end zeroed."""
    sfi = _sfi()
    lens = [9000, 300, 5000, 40, 7000, 2500, 1200, 8100, 60, 3300, 6400, 900]
    prob = Problem(seed=71, lens=lens, Hq=16, Hkv=8, D=128, S=4, W=32).to_device()
    maxL = int(prob.lens.max()) + 16
    splits = 0 if ragged else 12
    ws = (sfi.alloc_ragged_workspace(prob.shape, prob.B, maxL, dense=True) if ragged
          else sfi.alloc_workspace(prob.shape, prob.B, maxL, splits))
    st = _status()
    refs = [prob.oracle_dense(r) for r in range(prob.B)]
    for subset in ([0, 4, 7], list(range(12)), [11, 2, 9, 0, 5], list(range(11, -1, -1))):
        out = torch.full((prob.B, prob.Hq, prob.D), float("nan"), device="cuda")
        lse = torch.full((prob.B, prob.Hq), float("nan"), device="cuda")
        sfi.sfi_slow_dense_attn_with_scores(prob.shape, prob.d_kv, prob.S, prob.W, prob.d_q, out, lse, None,
                                            req_ids=dev_i32(subset), max_tokens=maxL, num_splits=splits,
                                            workspace=ws, dev_status=st,
                                            flags=sfi.SFI_ATTN_RAGGED if ragged else 0)
        torch.cuda.synchronize()
        assert st.item() == 0
        assert counters_zero(ws, prob.B * prob.Hkv), subset
        o, l = out.cpu().numpy(), lse.cpu().numpy()
        for r in subset:
            assert_close(o[r], refs[r][0], f"out r={r} subset={subset}")
            assert_close(l[r], refs[r][1], f"lse r={r} subset={subset}")


@pytest.mark.parametrize("D,Hq,Hkv", [(128, 16, 8), (128, 32, 8), (128, 64, 8), (64, 8, 2), (128, 8, 8)])
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_dense_attention_matches_oracle(D, Hq, Hkv, splits):
    lens = [1, 2, 15, 16, 17, 100, 777, 1500]
    prob = Problem(seed=D * 1000 + Hq + splits, lens=lens, Hq=Hq, Hkv=Hkv, D=D, S=4, W=32).to_device()
    out, lse = _dense(prob, num_splits=splits)
    for r in range(prob.B):
        o_ref, l_ref = prob.oracle_dense(r)
        assert_close(out[r], o_ref, f"out r={r}")
        assert_close(lse[r], l_ref, f"lse r={r}")


@pytest.mark.parametrize("D,Hq,Hkv", [(64, 8, 2), (128, 8, 8), (128, 16, 8), (128, 32, 8), (128, 64, 8)],
                         ids=["d64-g4", "d128-g1", "d128-g2", "d128-g4", "d128-g8"])
@pytest.mark.parametrize("splits", [0, 12], ids=["auto", "workspace-merge"])
def test_slow_step_scores_match_oracle_within_fp32_bound(D, Hq, Hkv, splits):
    """Score values element-wise against the oracle's fp64 group sums (rounded once to
    fp32), within the fp32 dot-product bound, at every group size G = 1, 2, 4, 8."""
    prob = Problem(seed=7 + Hq + D, lens=[37, 300, 1024, 2000], Hq=Hq, Hkv=Hkv, D=D, S=4, W=32,
                   heavy_frac=0.04).to_device()
    stride = 2016
    if splits:
        assert _sfi().sfi_plan_splits(prob.shape, prob.B, 2016, splits) == splits
    scores = torch.full((prob.B, prob.Hkv, stride), float("nan"), device="cuda")
    out, lse = _dense(prob, scores=scores, num_splits=splits)
    sc = scores.cpu().numpy()
    for r in range(prob.B):
        L = prob.lens[r]
        ref = prob.oracle_scores(r, stride)
        bound = prob.score_bound(r, stride)
        assert np.isnan(sc[r, :, L:]).all(), "entries at j >= L must not be written"
        masked = np.isneginf(ref[:, :L])
        assert np.array_equal(np.isneginf(sc[r, :, :L]), masked)
        err = np.abs(sc[r, :, :L][~masked].astype(np.float64) - ref[:, :L][~masked])
        assert (err <= bound[:, :L][~masked]).all(), err.max()
        o_ref, l_ref = prob.oracle_dense(r)
        assert_close(out[r], o_ref, f"out r={r}")


# ---------------------------------------------------------------------------
# Selector
# ---------------------------------------------------------------------------
def _select(scores_np, lens, S, W, k_per_req, k_cap, Hkv, req_ids=None):
    sfi = _sfi()
    B = len(lens)
    scores = torch.as_tensor(scores_np).cuda()
    idx = torch.full((B, Hkv, max(k_cap, 1)), -7, dtype=torch.int32, device="cuda")
    count = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    st = _status()
    sfi.sfi_select_topk(scores, Hkv, dev_i32(lens), S, W, dev_i32(k_per_req), idx, count,
                        req_ids=None if req_ids is None else dev_i32(req_ids), dev_status=st)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), count.cpu().numpy(), st.item()


def _check_selection(scores_np, lens, S, W, k_per_req, k_cap, Hkv):
    idx, count, st = _select(scores_np, lens, S, W, k_per_req, k_cap, Hkv)
    assert st == 0
    for r in range(len(lens)):
        for kvh in range(Hkv):
            want = oracle.select_topk(scores_np[r, kvh], lens[r], S, W, k_per_req[r])
            assert count[r] == len(want)
            np.testing.assert_array_equal(idx[r, kvh, :len(want)], want, err_msg=f"r={r} kv={kvh}")
            assert (idx[r, kvh, len(want):] == -7).all(), "entries past k_eff must not be written"


def test_selector_planted_zipf_ties():
    S, W, Hkv = 64, 256, 2
    lens = [64 + 256 + 5000, 64 + 256 + 9000]
    ks = [400, 4096]
    stride = max(lens)
    sc = np.full((2, Hkv, stride), np.nan, np.float32)
    for r in range(2):
        for kvh in range(Hkv):
            n = lens[r] - S - W
            sc[r, kvh, :lens[r]] = -np.inf
            sc[r, kvh, S:S + n] = syn.zipf_scores_with_ties(syn.rng(200, r, kvh), n, ks[r])
    _check_selection(sc, lens, S, W, ks, 4096, Hkv)


SELECTOR_CASES = ["all_equal", "neg_inf_except_k", "nan_and_signed_zero", "k_zero", "k_all", "k_over_n", "short",
                  "gaussian"]


@pytest.mark.parametrize("case", SELECTOR_CASES)
def test_selector_edge_cases(case):
    S, W, Hkv = 4, 32, 2
    g = syn.rng(201, SELECTOR_CASES.index(case))
    lens = [1000, 1000, 30]
    k = [50, 50, 5]
    sc = np.zeros((3, Hkv, 1000), np.float32)
    if case == "neg_inf_except_k":
        sc[:] = -np.inf
        for r in range(3):
            n = lens[r] - S - W
            for kvh in range(Hkv):
                if n > 0:
                    sc[r, kvh, S + g.choice(n, size=min(3, n), replace=False)] = 1.0
    elif case == "nan_and_signed_zero":
        pal = np.array([0.0, -0.0, np.nan, -np.inf, 1.0], np.float32)
        sc[:] = pal[g.integers(0, 5, size=sc.shape)]
    elif case == "k_zero":
        k = [0, 0, 0]
        sc[:] = g.standard_normal(sc.shape)
    elif case == "k_all":
        k = [1000 - S - W, 1000 - S - W, 0]
        sc[:] = g.standard_normal(sc.shape)
    elif case == "k_over_n":
        k = [2000, 964, 100]
        sc[:] = g.standard_normal(sc.shape)
    elif case == "short":
        lens = [3, 36, 37]
        k = [10, 10, 10]
        sc[:] = g.standard_normal(sc.shape)
    elif case == "gaussian":
        sc[:] = g.standard_normal(sc.shape).astype(np.float32)
    _check_selection(sc, lens, S, W, k, 2000, Hkv)


def test_selector_rejects_k_over_cap():
    sc = np.zeros((2, 1, 500), np.float32)
    idx, count, st = _select(sc, [500, 500], 4, 32, [10, 99], 50, 1)
    assert st & 4  # SFI_DEV_K_OVERFLOW
    assert count[0] == 10 and count[1] == -7


# ---------------------------------------------------------------------------
# Compaction, append
# ---------------------------------------------------------------------------
def _compact_buffers(prob, k_per_req):
    sfi = _sfi()
    off, cap = sfi.compact_layout(prob.shape, prob.S, k_per_req)
    rows = int((off[-1] + prob.Hkv * cap[-1]).item())
    ck = torch.zeros((rows, prob.D), dtype=torch.bfloat16, device="cuda")
    cv = torch.zeros_like(ck)
    count = torch.zeros(prob.B, dtype=torch.int32, device="cuda")
    return sfi.CompactKV(ck, cv, off, cap, count)


def test_slow_step_selection_and_compaction_bit_exact():
    """Dense + scores -> Selector -> compaction on the GPU; the oracle ranks the GPU's score bytes."""
    sfi = _sfi()
    S, W = 4, 32
    lens = [1024, 777, 36, 3, 40]
    prob = Problem(seed=11, lens=lens, Hq=8, Hkv=2, D=64, S=S, W=W, heavy_frac=0.04).to_device()
    k_per_req = [64, 100, 64, 8, 64]
    k_cap = 128
    stride = 1024
    scores = torch.full((prob.B, prob.Hkv, stride), float("nan"), device="cuda")
    _dense(prob, scores=scores)
    sc = scores.cpu().numpy()
    comp = _compact_buffers(prob, k_per_req)
    idx = torch.full((prob.B, prob.Hkv, k_cap), -7, dtype=torch.int32, device="cuda")
    st = _status()
    sfi.sfi_select_topk(scores, prob.Hkv, prob.d_kv.seq_lens, S, W, dev_i32(k_per_req), idx, comp.count,
                        dev_status=st)
    sfi.sfi_compact_gather(prob.shape, prob.d_kv, idx, comp.count, S, comp, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    ref_idx, ref_count = run_oracle_selection(prob, sc, k_per_req, k_cap)
    got_idx, got_count = idx.cpu().numpy(), comp.count.cpu().numpy()
    np.testing.assert_array_equal(got_count, ref_count)
    ck, cv = host_bf16(comp.k), host_bf16(comp.v)
    off, cap = comp.row_offset.cpu().numpy(), comp.capacity.cpu().numpy()
    for r in range(prob.B):
        keff = ref_count[r]
        np.testing.assert_array_equal(got_idx[r, :, :keff], ref_idx[r, :, :keff])
        rk, rv = oracle_compact_request(prob, r, ref_idx[r], keff, cap[r])
        ns = min(S, lens[r])
        for kvh in range(prob.Hkv):
            base = off[r] + kvh * cap[r]
            for lo, hi in ((0, ns), (S, S + keff)):
                np.testing.assert_array_equal(ck[base + lo:base + hi], rk[kvh, lo:hi])
                np.testing.assert_array_equal(cv[base + lo:base + hi], rv[kvh, lo:hi])
    # planted heavy hitters dominate the selection of the long request
    assert got_count[0] == 64


def test_append_bit_exact_and_only_the_last_slot():
    sfi = _sfi()
    prob = Problem(seed=12, lens=[40, 16, 1], Hq=8, Hkv=2, D=128, S=4, W=32, extra_tokens=20).to_device()
    g = syn.rng(300, 1)
    kn, vn = syn.normal_bf16(g, (3, 2, 128)), syn.normal_bf16(g, (3, 2, 128))
    new_lens = prob.lens + 1
    prob.set_lens(new_lens)
    st = _status()
    sfi.sfi_paged_kv_append(prob.shape, prob.d_kv, dev_bf16(kn), dev_bf16(vn), dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    kp, vp = prob.kv.k_pool.copy(), prob.kv.v_pool.copy()
    for r in range(3):
        oracle.paged_append(kp, vp, prob.kv.page_table[r], new_lens[r], kn[r], vn[r], 2, 128, 16)
    np.testing.assert_array_equal(host_bf16(prob.d_kv.k_pool), kp)
    np.testing.assert_array_equal(host_bf16(prob.d_kv.v_pool), vp)


# ---------------------------------------------------------------------------
# Fast step
# ---------------------------------------------------------------------------
def _fast_case(seed, lens, Hq, Hkv, D, S, W, k_per_req, k_cap, splits=0, req_ids=None, heavy=0.02, ragged=False,
               max_tokens=None):
    """Slow step + Selector + compaction on the GPU, then the fast step at the same length."""
    sfi = _sfi()
    prob = Problem(seed=seed, lens=lens, Hq=Hq, Hkv=Hkv, D=D, S=S, W=W, heavy_frac=heavy).to_device()
    stride = int(max(lens))
    scores = torch.full((prob.B, prob.Hkv, stride), float("nan"), device="cuda")
    _dense(prob, scores=scores)
    comp = _compact_buffers(prob, k_per_req)
    idx = torch.zeros((prob.B, prob.Hkv, k_cap), dtype=torch.int32, device="cuda")
    st = _status()
    sfi.sfi_select_topk(scores, prob.Hkv, prob.d_kv.seq_lens, S, W, dev_i32(k_per_req), idx, comp.count,
                        dev_status=st)
    sfi.sfi_compact_gather(prob.shape, prob.d_kv, idx, comp.count, S, comp, dev_status=st)
    out = torch.full((prob.B, Hq, D), float("nan"), device="cuda")
    lse = torch.full((prob.B, Hq), float("nan"), device="cuda")
    max_tokens = S + k_cap + W + 32 if max_tokens is None else max_tokens
    if ragged:
        ws = sfi.alloc_ragged_workspace(prob.shape, prob.B, max_tokens)
    else:
        ws = sfi.alloc_workspace(prob.shape, prob.B, max_tokens, splits)
    rid = None if req_ids is None else dev_i32(req_ids)
    sfi.sfi_fast_decode_attn(prob.shape, prob.d_kv, comp, S, W, prob.d_q, out, lse, req_ids=rid,
                             max_tokens=max_tokens, num_splits=splits, workspace=ws, dev_status=st,
                             flags=sfi.SFI_ATTN_RAGGED if ragged else 0)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert counters_zero(ws, prob.B * Hkv)
    sc = scores.cpu().numpy()
    ref_idx, ref_count = run_oracle_selection(prob, sc, k_per_req, k_cap)
    cap = comp.capacity.cpu().numpy()
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    for r in (range(prob.B) if req_ids is None else req_ids):
        rk, rv = oracle_compact_request(prob, r, ref_idx[r], ref_count[r], cap[r])
        o_ref, l_ref = oracle.fast_attn(prob.q[r], rk, rv, ref_count[r], prob.kv.k_pool, prob.kv.v_pool,
                                        prob.kv.page_table[r], prob.lens[r], S, W, Hq, Hkv, D, 16)
        assert_close(o[r], o_ref, f"fast out r={r}")
        assert_close(l[r], l_ref, f"fast lse r={r}")
    if req_ids is not None:
        untouched = sorted(set(range(prob.B)) - set(req_ids))
        assert np.isnan(o[untouched]).all()
    return prob


@pytest.mark.parametrize("splits", [1, 2, 3, 4, 5, 0])
def test_fast_step_matches_oracle(splits):
    """Split plans of one CTA, clusters whose other CTAs send per-warp partials (2-4
    splits at G = 2), clusters that send one partial per CTA (5) and the automatic plan."""
    lens = [1024, 1031, 530, 36, 30, 3, 17]
    _fast_case(21 + splits, lens, 16, 8, 128, 4, 32, [64, 64, 100, 5, 5, 5, 5], 128, splits=splits)


@pytest.mark.parametrize("D,splits", [(128, 7), (64, 8)])
def test_fast_step_per_warp_partials_from_many_ctas(D, splits):
    """One query row per KV head (G = 1): the other CTAs of a 7- or 8-CTA cluster each
    send four per-warp partials (up to 28) into rank 0's receive region, merged in one pass."""
    lens = [2000, 1500, 1800, 1200]
    k_cap = 1024
    shape = _sfi().AttnShape(8, 8, D)
    assert _sfi().sfi_plan_splits(shape, len(lens), 4 + k_cap + 32 + 32, splits) == splits
    _fast_case(61 + splits, lens, 8, 8, D, 4, 32, [900, 700, 1000, 500], k_cap, splits=splits)


@pytest.mark.parametrize("bounds", ["tight", "underestimated"])
def test_ragged_fast_step_matches_oracle(bounds):
    """SFI_ATTN_RAGGED: the fast step planned in fixed-size chunks over requests whose
    selected counts differ by two orders of magnitude (one request past the host's
    bound when it is underestimated); a subset of the batch by request id."""
    lens = [9000, 700, 30, 5200, 3, 12000]
    k_per_req = [2000, 64, 5, 900, 5, 2500]
    mt = None if bounds == "tight" else 800
    _fast_case(41, lens, 16, 8, 128, 4, 32, k_per_req, 2560, req_ids=[0, 1, 2, 3, 5] if bounds == "tight" else None,
               ragged=True, max_tokens=mt)


@pytest.mark.parametrize("bounds", ["tight", "underestimated"])
def test_ragged_dense_with_scores_matches_oracle(bounds):
    """SFI_ATTN_RAGGED on the slow step: dense attention and the masked scores for a
    batch whose lengths span 1 to 20000 tokens, by request-id subset; with an
    underestimated bound the long requests take bigger chunks, same results."""
    lens = [20000, 1, 700, 4100, 17, 9000]
    prob = Problem(seed=43, lens=lens, Hq=8, Hkv=2, D=64, S=4, W=32, heavy_frac=0.03).to_device()
    stride = int(max(lens)) + 8
    scores = torch.full((prob.B, prob.Hkv, stride), float("nan"), device="cuda")
    rid = [5, 0, 1, 2, 3] if bounds == "tight" else None
    out, lse = _dense(prob, scores=scores, req_ids=None if rid is None else dev_i32(rid), ragged=True,
                      max_tokens=None if bounds == "tight" else 1000)
    sc = scores.cpu().numpy()
    for r in (range(prob.B) if rid is None else rid):
        o_ref, l_ref = prob.oracle_dense(r)
        assert_close(out[r], o_ref, f"ragged dense out r={r}")
        assert_close(lse[r], l_ref, f"ragged dense lse r={r}")
        L = prob.lens[r]
        ref = prob.oracle_scores(r, stride)
        masked = np.isneginf(ref[:, :L])
        assert np.array_equal(np.isneginf(sc[r, :, :L]), masked)
        err = np.abs(sc[r, :, :L][~masked].astype(np.float64) - ref[:, :L][~masked])
        assert (err <= prob.score_bound(r, stride)[:, :L][~masked]).all()
    if rid is not None:
        assert np.isnan(out[4]).all() and np.isnan(sc[4]).all()


def test_fast_step_d64_g4_and_subset():
    lens = [1024, 600, 1100, 900]
    _fast_case(31, lens, 8, 2, 64, 4, 32, [64, 64, 64, 64], 64, req_ids=[2, 0])


def test_fast_step_full_retention_equals_dense():
    """Table 1: at 100% retention the fast step is the dense computation."""
    S, W = 64, 256
    lens = [2000, 1500]
    k = [l - S - W for l in lens]
    prob = _fast_case(41, lens, 32, 8, 128, S, W, k, max(k), heavy=0.0)
    out_d, lse_d = _dense(prob)
    for r in range(prob.B):
        o_ref, l_ref = prob.oracle_dense(r)
        assert_close(out_d[r], o_ref, "dense")


def test_config1_slow_then_eight_fast_steps():
    """Single request, GQA 8/2, D 64, context 1024, sink 4 + top-64 + recent 32: one slow
    step at L = 1024, then 8 fast steps at L = 1025..1032, each appending its token."""
    sfi = _sfi()
    S, W, k = 4, 32, 64
    prob = Problem(seed=1, lens=[1024], Hq=8, Hkv=2, D=64, S=S, W=W, extra_tokens=8, heavy_frac=40 / 988,
                   heavy_beta=3.0).to_device()
    g = syn.rng(1, 99)
    st = _status()
    scores = torch.full((1, 2, 1040), float("nan"), device="cuda")
    _dense(prob, scores=scores)
    comp = _compact_buffers(prob, [k])
    idx = torch.zeros((1, 2, k), dtype=torch.int32, device="cuda")
    sfi.sfi_select_topk(scores, 2, prob.d_kv.seq_lens, S, W, dev_i32([k]), idx, comp.count, dev_status=st)
    sfi.sfi_compact_gather(prob.shape, prob.d_kv, idx, comp.count, S, comp, dev_status=st)
    torch.cuda.synchronize()
    sc = scores.cpu().numpy()
    ref_idx, ref_count = run_oracle_selection(prob, sc, [k], k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    rk, rv = oracle_compact_request(prob, 0, ref_idx[0], ref_count[0], S + k)
    ws = sfi.alloc_workspace(prob.shape, 1, S + k + W + 32)
    kp, vp = prob.kv.k_pool.copy(), prob.kv.v_pool.copy()
    for step in range(8):
        L = 1025 + step
        q = syn.normal_bf16(g, (1, 8, 64))
        kn, vn = syn.normal_bf16(g, (1, 2, 64)), syn.normal_bf16(g, (1, 2, 64))
        prob.set_lens([L])
        sfi.sfi_paged_kv_append(prob.shape, prob.d_kv, dev_bf16(kn), dev_bf16(vn), dev_status=st)
        out = torch.empty((1, 8, 64), device="cuda")
        lse = torch.empty((1, 8), device="cuda")
        sfi.sfi_fast_decode_attn(prob.shape, prob.d_kv, comp, S, W, dev_bf16(q), out, lse,
                                 max_tokens=S + k + W + 32, workspace=ws, dev_status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        oracle.paged_append(kp, vp, prob.kv.page_table[0], L, kn[0], vn[0], 2, 64, 16)
        o_ref, l_ref = oracle.fast_attn(q[0], rk, rv, ref_count[0], kp, vp, prob.kv.page_table[0], L, S, W,
                                        8, 2, 64, 16)
        assert_close(out.cpu().numpy()[0], o_ref, f"step {step}")
        assert_close(lse.cpu().numpy()[0], l_ref, f"lse step {step}")


# ---------------------------------------------------------------------------
# Device-side error reporting (host-made bad inputs the kernels check; nothing faults)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("splits", [1, 2, 12], ids=["one-split", "cluster-merge", "workspace-merge"])
def test_bad_page_and_length_are_reported_not_faulted(splits):
    """A page id outside the pool is reported (SFI_DEV_BAD_PAGE) and the offending
    request writes nothing: its outputs, log-sum-exps and score rows keep the caller's
    NaN sentinel, in every split plan (one CTA, cluster merge, workspace merge), while
    the healthy request matches the oracle. A bad length is reported the same way."""
    sfi = _sfi()
    prob = Problem(seed=51, lens=[1500, 1500], Hq=8, Hkv=2, D=64, S=4, W=32, extra_tokens=16).to_device()
    pt = prob.d_kv.page_table.clone()
    # a page id outside the pool, in the middle of request 1 (outside the first split of a
    # two-split plan, so the bad partial reaches the merge from a peer CTA)
    pt[1, 60] = 10_000_000
    bad = sfi.PagedKV(prob.d_kv.k_pool, prob.d_kv.v_pool, pt, prob.d_kv.seq_lens)
    stride = 1520
    maxL = 1520
    ws = sfi.alloc_workspace(prob.shape, 2, maxL, splits)
    for with_scores in (False, True):
        out = torch.full((2, 8, 64), float("nan"), device="cuda")
        lse = torch.full((2, 8), float("nan"), device="cuda")
        scores = torch.full((2, 2, stride), float("nan"), device="cuda") if with_scores else None
        st = _status()
        sfi.sfi_slow_dense_attn_with_scores(prob.shape, bad, 4, 32, prob.d_q, out, lse, scores, max_tokens=maxL,
                                            num_splits=splits, workspace=ws, dev_status=st)
        torch.cuda.synchronize()
        assert st.item() == 1, f"status {st.item()}"  # SFI_DEV_BAD_PAGE only
        o, l = out.cpu().numpy(), lse.cpu().numpy()
        assert np.isnan(o[1]).all() and np.isnan(l[1]).all(), "the bad request's outputs must not be written"
        o_ref, l_ref = prob.oracle_dense(0)
        assert_close(o[0], o_ref, "the healthy request is unaffected")
        assert_close(l[0], l_ref, "the healthy request's lse")
        if with_scores:
            sc = scores.cpu().numpy()
            assert np.isnan(sc[1]).all(), "the bad request's score rows must not be written"
            ref = prob.oracle_scores(0, stride)
            masked = np.isneginf(ref[:, :1500])
            assert np.array_equal(np.isneginf(sc[0, :, :1500]), masked)
        if splits > 8:
            assert counters_zero(ws, 2 * prob.Hkv), "split counters must be left zeroed"
    # the fast step over the same pages (the recent window holds the bad page)
    pt_fast = prob.d_kv.page_table.clone()
    pt_fast[1, 1490 // 16] = -3
    comp = _compact_buffers(prob, [64, 64])
    badf = sfi.PagedKV(prob.d_kv.k_pool, prob.d_kv.v_pool, pt_fast, prob.d_kv.seq_lens)
    out = torch.full((2, 8, 64), float("nan"), device="cuda")
    st = _status()
    sfi.sfi_fast_decode_attn(prob.shape, badf, comp, 4, 32, prob.d_q, out, None, max_tokens=4 + 64 + 32 + 32,
                             num_splits=min(splits, 2), workspace=sfi.alloc_workspace(prob.shape, 2, 132, 2),
                             dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 1, f"status {st.item()}"
    assert np.isnan(out.cpu().numpy()[1]).all(), "the bad request's fast-step outputs must not be written"
    assert np.isfinite(out.cpu().numpy()[0]).all()
    st.zero_()
    lens_bad = sfi.PagedKV(prob.d_kv.k_pool, prob.d_kv.v_pool, prob.d_kv.page_table, dev_i32([100, 0]))
    sfi.sfi_slow_dense_attn_with_scores(prob.shape, lens_bad, 4, 32, prob.d_q, out, None, None, dev_status=st)
    kn = torch.zeros((2, 2, 64), dtype=torch.bfloat16, device="cuda")
    sfi.sfi_paged_kv_append(prob.shape, bad, kn, kn, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & 2


@pytest.mark.parametrize("splits", [2, 12], ids=["cluster-merge", "workspace-merge"])
def test_bounded_wait_runs_out_and_reports_timeout(splits):
    """SFI_ATTN_TEST_WITHHOLD: every CTA's producer withholds its second stage, so the
    consumers' bounded wait runs out (about 2 s): the launch returns with SFI_DEV_TIMEOUT,
    writes no output and leaves the workspace counters zeroed, and a normal launch right
    after it (fresh status, same workspace) is correct, so the context stays usable."""
    sfi = _sfi()
    prob = Problem(seed=53, lens=[3000, 2500], Hq=16, Hkv=8, D=128, S=4, W=32).to_device()
    maxL = int(prob.lens.max()) + 16
    sentinel = float("nan")
    out = torch.full((prob.B, prob.Hq, prob.D), sentinel, device="cuda")
    ws = sfi.alloc_workspace(prob.shape, prob.B, maxL, splits)
    st = _status()
    sfi.sfi_slow_dense_attn_with_scores(prob.shape, prob.d_kv, prob.S, prob.W, prob.d_q, out, None, None,
                                        max_tokens=maxL, num_splits=splits, workspace=ws, dev_status=st,
                                        flags=sfi.SFI_ATTN_TEST_WITHHOLD)
    torch.cuda.synchronize()
    assert st.item() & 16, f"status {st.item()}"  # SFI_DEV_TIMEOUT
    assert np.isnan(out.cpu().numpy()).all(), "a timed-out launch writes no output"
    if splits > 8:
        # every split still reaches the merge counter, so it is left zeroed
        assert counters_zero(ws, prob.B * prob.Hkv), "split counters must be left zeroed after a timeout"
    st.zero_()
    sfi.sfi_slow_dense_attn_with_scores(prob.shape, prob.d_kv, prob.S, prob.W, prob.d_q, out, None, None,
                                        max_tokens=maxL, num_splits=splits, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    o = out.cpu().numpy()
    for r in range(prob.B):
        o_ref, _ = prob.oracle_dense(r)
        assert_close(o[r], o_ref, f"after the timeout r={r}")


def test_bad_selected_index_is_reported():
    sfi = _sfi()
    prob = Problem(seed=52, lens=[200], Hq=8, Hkv=2, D=64, S=4, W=32).to_device()
    comp = _compact_buffers(prob, [8])
    idx = torch.tensor([[[5, 6, 7, 8, 9, 10, 11, 5000], [5, 6, 7, 8, 9, 10, 11, 12]]], dtype=torch.int32,
                       device="cuda")
    comp.count.fill_(8)
    st = _status()
    sfi.sfi_compact_gather(prob.shape, prob.d_kv, idx, comp.count, 4, comp, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & 8


# ---------------------------------------------------------------------------
# Fused append (k_new / v_new passed to the attention entry points)
# ---------------------------------------------------------------------------
def _grow(prob, g):
    """Advance every request by one token: new lengths and seeded K/V for position L - 1."""
    kn = syn.normal_bf16(g, (prob.B, prob.Hkv, prob.D))
    vn = syn.normal_bf16(g, (prob.B, prob.Hkv, prob.D))
    prob.set_lens(prob.lens + 1)
    return kn, vn


@pytest.mark.parametrize("W", [32, 0])
def test_fused_append_dense_with_scores_matches_oracle(W):
    """Slow step with the append fused: equals append-then-attend, scores included
    (W = 0 puts the new token among the candidates), and the pages hold the token."""
    sfi = _sfi()
    lens = [1023, 40, 16, 1, 500]
    prob = Problem(seed=61 + W, lens=lens, Hq=16, Hkv=8, D=128, S=4, W=W, extra_tokens=16).to_device()
    kn, vn = _grow(prob, syn.rng(400, W))
    stride = int(prob.lens.max())
    scores = torch.full((prob.B, prob.Hkv, stride), float("nan"), device="cuda")
    out = torch.full((prob.B, 16, 128), float("nan"), device="cuda")
    lse = torch.full((prob.B, 16), float("nan"), device="cuda")
    ws = sfi.alloc_workspace(prob.shape, prob.B, stride + 16)
    st = _status()
    sfi.sfi_slow_dense_attn_with_scores(prob.shape, prob.d_kv, prob.S, W, prob.d_q, out, lse, scores,
                                        k_new=dev_bf16(kn), v_new=dev_bf16(vn), max_tokens=stride + 16,
                                        workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    for r in range(prob.B):
        oracle.paged_append(prob.kv.k_pool, prob.kv.v_pool, prob.kv.page_table[r], prob.lens[r], kn[r], vn[r],
                            prob.Hkv, prob.D, 16)
    np.testing.assert_array_equal(host_bf16(prob.d_kv.k_pool), prob.kv.k_pool)
    np.testing.assert_array_equal(host_bf16(prob.d_kv.v_pool), prob.kv.v_pool)
    o, l, sc = out.cpu().numpy(), lse.cpu().numpy(), scores.cpu().numpy()
    for r in range(prob.B):
        o_ref, l_ref = prob.oracle_dense(r)
        assert_close(o[r], o_ref, f"out r={r}")
        assert_close(l[r], l_ref, f"lse r={r}")
        L = prob.lens[r]
        ref = prob.oracle_scores(r, stride)
        masked = np.isneginf(ref[:, :L])
        assert np.array_equal(np.isneginf(sc[r, :, :L]), masked)
        err = np.abs(sc[r, :, :L][~masked].astype(np.float64) - ref[:, :L][~masked])
        assert (err <= prob.score_bound(r, stride)[:, :L][~masked]).all()


@pytest.mark.parametrize("splits", [1, 3, 0])
def test_fused_append_fast_step_matches_oracle(splits):
    """Fast step with the append fused, at L_slow + 1: the new token is the last row of
    the recent window (or a sink row when L <= S)."""
    sfi = _sfi()
    S, W, k = 4, 32, 64
    lens = [1024, 700, 36, 3, 2]
    prob = Problem(seed=71 + splits, lens=lens, Hq=16, Hkv=8, D=128, S=S, W=W, extra_tokens=16,
                   heavy_frac=0.02).to_device()
    # slow step + Selector + compaction at L_slow (regular calls)
    stride = int(prob.lens.max())
    scores = torch.full((prob.B, prob.Hkv, stride), float("nan"), device="cuda")
    _dense(prob, scores=scores)
    comp = _compact_buffers(prob, [k] * prob.B)
    idx = torch.zeros((prob.B, prob.Hkv, k), dtype=torch.int32, device="cuda")
    st = _status()
    sfi.sfi_select_topk(scores, prob.Hkv, prob.d_kv.seq_lens, S, W, dev_i32([k] * prob.B), idx, comp.count,
                        dev_status=st)
    sfi.sfi_compact_gather(prob.shape, prob.d_kv, idx, comp.count, S, comp, dev_status=st)
    torch.cuda.synchronize()
    ref_idx, ref_count = run_oracle_selection(prob, scores.cpu().numpy(), [k] * prob.B, k)
    cap = comp.capacity.cpu().numpy()
    compacts = [oracle_compact_request(prob, r, ref_idx[r], ref_count[r], cap[r]) for r in range(prob.B)]
    # one more token, fused into the fast step
    kn, vn = _grow(prob, syn.rng(401, splits))
    q = syn.normal_bf16(syn.rng(402, splits), (prob.B, 16, 128))
    out = torch.full((prob.B, 16, 128), float("nan"), device="cuda")
    lse = torch.full((prob.B, 16), float("nan"), device="cuda")
    max_tokens = S + k + W + 32
    ws = sfi.alloc_workspace(prob.shape, prob.B, max_tokens, splits)
    sfi.sfi_fast_decode_attn(prob.shape, prob.d_kv, comp, S, W, dev_bf16(q), out, lse, k_new=dev_bf16(kn),
                             v_new=dev_bf16(vn), max_tokens=max_tokens, num_splits=splits, workspace=ws,
                             dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    for r in range(prob.B):
        oracle.paged_append(prob.kv.k_pool, prob.kv.v_pool, prob.kv.page_table[r], prob.lens[r], kn[r], vn[r],
                            prob.Hkv, prob.D, 16)
    np.testing.assert_array_equal(host_bf16(prob.d_kv.k_pool), prob.kv.k_pool)
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    for r in range(prob.B):
        rk, rv = compacts[r]
        if prob.lens[r] <= S:  # the new token is a sink row: the oracle's compact copy must hold it too
            rk[:, prob.lens[r] - 1], rv[:, prob.lens[r] - 1] = kn[r], vn[r]
        o_ref, l_ref = oracle.fast_attn(q[r], rk, rv, ref_count[r], prob.kv.k_pool, prob.kv.v_pool,
                                        prob.kv.page_table[r], prob.lens[r], S, W, 16, 8, 128, 16)
        assert_close(o[r], o_ref, f"fast out r={r}")
        assert_close(l[r], l_ref, f"fast lse r={r}")


def test_early_prefetch_flag_gives_identical_results():
    """Back-to-back launches on one stream, each reading KV state the previous launch
    does not write, with SFI_ATTN_EARLY_KV_PREFETCH: bit-identical to the default."""
    sfi = _sfi()
    S, W, k = 4, 32, 64
    probs = [Problem(seed=81 + i, lens=[1024, 1500, 700, 40], Hq=16, Hkv=8, D=128, S=S, W=W,
                     heavy_frac=0.02).to_device() for i in range(3)]
    comps = []
    for prob in probs:
        scores = torch.empty((prob.B, prob.Hkv, 1500), device="cuda")
        _dense(prob, scores=scores)
        comp = _compact_buffers(prob, [k] * prob.B)
        idx = torch.zeros((prob.B, prob.Hkv, k), dtype=torch.int32, device="cuda")
        sfi.sfi_select_topk(scores, prob.Hkv, prob.d_kv.seq_lens, S, W, dev_i32([k] * prob.B), idx, comp.count)
        sfi.sfi_compact_gather(prob.shape, prob.d_kv, idx, comp.count, S, comp)
        comps.append(comp)
    torch.cuda.synchronize()

    def run(flags):
        outs = []
        st = _status()
        for rep in range(2):
            for prob, comp in zip(probs, comps):
                fo = torch.empty((prob.B, 16, 128), device="cuda")
                do = torch.empty((prob.B, 16, 128), device="cuda")
                sc = torch.full((prob.B, prob.Hkv, 1500), float("nan"), device="cuda")
                sfi.sfi_fast_decode_attn(prob.shape, prob.d_kv, comp, S, W, prob.d_q, fo, max_tokens=S + k + W + 32,
                                         workspace=sfi.alloc_workspace(prob.shape, prob.B, S + k + W + 32),
                                         dev_status=st, flags=flags)
                sfi.sfi_slow_dense_attn_with_scores(prob.shape, prob.d_kv, S, W, prob.d_q, do, None, sc,
                                                    max_tokens=1516, workspace=sfi.alloc_workspace(prob.shape, prob.B,
                                                                                                   1516),
                                                    dev_status=st, flags=flags)
                outs += [fo, do, sc]
        torch.cuda.synchronize()
        assert st.item() == 0
        return [x.cpu().numpy() for x in outs]

    for a, b in zip(run(0), run(sfi.SFI_ATTN_EARLY_KV_PREFETCH)):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("bounds", ["tight", "underestimated"])
def test_mixed_launch_matches_oracle(bounds):
    """One launch serving fast and slow requests of one batch, the current token fused:
    fast requests against the oracle's fast step, slow ones against dense attention and
    the masked scores. The slow requests are long enough to be split, so their partial
    states merge through the workspace. Token bounds below the real lengths change the
    plan, never the results."""
    sfi = _sfi()
    S, W, k = 4, 32, 64
    lens = [4000, 1200, 3000, 600, 2500, 40]
    prob = Problem(seed=91, lens=lens, Hq=16, Hkv=8, D=128, S=S, W=W, extra_tokens=16,
                   heavy_frac=0.02).to_device()
    fast, slow = [1, 3, 5], [0, 2, 4]
    # an earlier slow step for the fast requests' compact buffers
    stride = int(prob.lens.max()) + 16
    scores0 = torch.full((prob.B, prob.Hkv, stride), float("nan"), device="cuda")
    _dense(prob, scores=scores0)
    comp = _compact_buffers(prob, [k] * prob.B)
    idx = torch.zeros((prob.B, prob.Hkv, k), dtype=torch.int32, device="cuda")
    st = _status()
    sfi.sfi_select_topk(scores0, prob.Hkv, prob.d_kv.seq_lens, S, W, dev_i32([k] * prob.B), idx, comp.count,
                        dev_status=st)
    sfi.sfi_compact_gather(prob.shape, prob.d_kv, idx, comp.count, S, comp, dev_status=st)
    torch.cuda.synchronize()
    ref_idx, ref_count = run_oracle_selection(prob, scores0.cpu().numpy(), [k] * prob.B, k)
    cap = comp.capacity.cpu().numpy()
    compacts = {r: oracle_compact_request(prob, r, ref_idx[r], ref_count[r], cap[r]) for r in fast}
    # the mixed step, one token later
    kn, vn = _grow(prob, syn.rng(403, 1))
    q = syn.normal_bf16(syn.rng(404, 1), (prob.B, 16, 128))
    out = torch.full((prob.B, 16, 128), float("nan"), device="cuda")
    lse = torch.full((prob.B, 16), float("nan"), device="cuda")
    scores = torch.full((prob.B, prob.Hkv, stride), float("nan"), device="cuda")
    mf, md = S + k + W + 32, int(prob.lens.max()) + 16
    if bounds == "underestimated":
        mf, md = 64, 1024
    ws = sfi.alloc_mixed_workspace(prob.shape, prob.B, mf, md)
    assert sfi.sfi_mixed_workspace_size(prob.shape, len(fast), len(slow), mf, md) > 0  # slow units are split
    sfi.sfi_mixed_decode_attn(prob.shape, prob.d_kv, comp, S, W, dev_bf16(q), out, dev_i32(fast), dev_i32(slow),
                              lse=lse, scores=scores, k_new=dev_bf16(kn), v_new=dev_bf16(vn), max_fast_tokens=mf,
                              max_dense_tokens=md, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert counters_zero(ws, prob.B * prob.Hkv)
    for r in range(prob.B):
        oracle.paged_append(prob.kv.k_pool, prob.kv.v_pool, prob.kv.page_table[r], prob.lens[r], kn[r], vn[r],
                            prob.Hkv, prob.D, 16)
    np.testing.assert_array_equal(host_bf16(prob.d_kv.k_pool), prob.kv.k_pool)
    prob.q = q
    o, l, sc = out.cpu().numpy(), lse.cpu().numpy(), scores.cpu().numpy()
    for r in fast:
        rk, rv = compacts[r]
        if prob.lens[r] <= S:
            rk[:, prob.lens[r] - 1], rv[:, prob.lens[r] - 1] = kn[r], vn[r]
        o_ref, l_ref = oracle.fast_attn(q[r], rk, rv, ref_count[r], prob.kv.k_pool, prob.kv.v_pool,
                                        prob.kv.page_table[r], prob.lens[r], S, W, 16, 8, 128, 16)
        assert_close(o[r], o_ref, f"mixed fast r={r}")
        assert_close(l[r], l_ref, f"mixed fast lse r={r}")
        assert np.isnan(sc[r]).all(), "fast requests write no scores"
    for r in slow:
        o_ref, l_ref = prob.oracle_dense(r)
        assert_close(o[r], o_ref, f"mixed slow r={r}")
        assert_close(l[r], l_ref, f"mixed slow lse r={r}")
        L = prob.lens[r]
        ref = prob.oracle_scores(r, stride)
        masked = np.isneginf(ref[:, :L])
        assert np.array_equal(np.isneginf(sc[r, :, :L]), masked)
        err = np.abs(sc[r, :, :L][~masked].astype(np.float64) - ref[:, :L][~masked])
        assert (err <= prob.score_bound(r, stride)[:, :L][~masked]).all()


# ---------------------------------------------------------------------------
# Selector + compaction in one call (sfi_select_compact)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("D,Hq,Hkv,lens,k_per_req,k_cap", [
    (64, 8, 2, [1024, 777, 36, 3, 40], [64, 100, 64, 8, 64], 128),          # L < S, L < S + W, keff < k
    (128, 16, 8, [300, 21000, 530], [400, 1500, 10], 1600),                  # keff == |C|; |C| > 16384 (rounds)
    (128, 32, 8, [4096, 2048], [256, 128], 256),
    (128, 16, 8, [700 + 37 * i for i in range(16)], [8 * i for i in range(16)], 128),  # 128 units, ragged k
])
def test_select_compact_bit_exact(D, Hq, Hkv, lens, k_per_req, k_cap):
    """Selector + compaction in one call equals the oracle Selector (on the GPU-written scores)
    followed by the oracle compaction, byte for byte, and leaves the same counts."""
    sfi = _sfi()
    S, W = 4, 32
    prob = Problem(seed=700 + D + len(lens), lens=lens, Hq=Hq, Hkv=Hkv, D=D, S=S, W=W, heavy_frac=0.03).to_device()
    stride = int(max(lens)) + 8
    scores = torch.full((prob.B, Hkv, stride), float("nan"), device="cuda")
    _dense(prob, scores=scores)
    comp = _compact_buffers(prob, [k_cap] * prob.B)
    idx = torch.full((prob.B, Hkv, k_cap), -7, dtype=torch.int32, device="cuda")
    st = _status()
    sfi.sfi_select_compact(prob.shape, prob.d_kv, scores, S, W, dev_i32(k_per_req), idx, comp, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    sc = scores.cpu().numpy()
    ref_idx, ref_count = run_oracle_selection(prob, sc, k_per_req, k_cap)
    got_idx, got_count = idx.cpu().numpy(), comp.count.cpu().numpy()
    np.testing.assert_array_equal(got_count, ref_count)
    ck, cv = host_bf16(comp.k), host_bf16(comp.v)
    off, cap = comp.row_offset.cpu().numpy(), comp.capacity.cpu().numpy()
    for r in range(prob.B):
        keff = ref_count[r]
        np.testing.assert_array_equal(got_idx[r, :, :keff], ref_idx[r, :, :keff])
        assert (got_idx[r, :, keff:] == -7).all(), "entries past k_eff must not be written"
        rk, rv = oracle_compact_request(prob, r, ref_idx[r], keff, cap[r])
        ns = min(S, lens[r])
        for kvh in range(Hkv):
            base = off[r] + kvh * cap[r]
            for lo, hi in ((0, ns), (S, S + keff)):
                np.testing.assert_array_equal(ck[base + lo:base + hi], rk[kvh, lo:hi], err_msg=f"K r={r} kv={kvh}")
                np.testing.assert_array_equal(cv[base + lo:base + hi], rv[kvh, lo:hi], err_msg=f"V r={r} kv={kvh}")


@pytest.mark.parametrize("B,Hkv", [(3, 2), (16, 8)])
def test_select_compact_subset_and_bad_capacity(B, Hkv):
    """A request subset is handled alone; a request whose capacity is below S + k_eff keeps its
    selection, is not packed, and is reported."""
    sfi = _sfi()
    S, W = 4, 32
    lens = [800 + 100 * (i % 3) for i in range(B)]
    prob = Problem(seed=720 + B, lens=lens, Hq=2 * Hkv, Hkv=Hkv, D=128, S=S, W=W).to_device()
    stride = 1008
    scores = torch.full((prob.B, Hkv, stride), float("nan"), device="cuda")
    _dense(prob, scores=scores)
    comp = _compact_buffers(prob, [8 if r == 1 else 64 for r in range(B)])  # request 1: capacity S + 8 < S + 64
    idx = torch.full((prob.B, Hkv, 64), -7, dtype=torch.int32, device="cuda")
    st = _status()
    subset = [2, 1] if B == 3 else list(range(B - 1, 0, -1))  # every request but 0
    sfi.sfi_select_compact(prob.shape, prob.d_kv, scores, S, W, dev_i32([64] * B), idx, comp,
                           req_ids=dev_i32(subset), dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 4  # SFI_DEV_K_OVERFLOW for request 1
    sc = scores.cpu().numpy()
    ref_idx, ref_count = run_oracle_selection(prob, sc, [64] * B, 64)
    got_idx = idx.cpu().numpy()
    for r in subset:
        np.testing.assert_array_equal(got_idx[r], ref_idx[r])
    assert (got_idx[0] == -7).all()
    ck = host_bf16(comp.k)
    off, cap = comp.row_offset.cpu().numpy(), comp.capacity.cpu().numpy()
    for r in subset:
        if r == 1:
            continue
        rk, _ = oracle_compact_request(prob, r, ref_idx[r], 64, cap[r])
        for kvh in range(Hkv):
            base = off[r] + kvh * cap[r]
            np.testing.assert_array_equal(ck[base:base + S + 64], rk[kvh, :S + 64])
    for kvh in range(Hkv):
        base1 = off[1] + kvh * cap[1]
        assert not ck[base1:base1 + cap[1]].any(), "the request with too small a capacity is not packed"


# ---------------------------------------------------------------------------
# Long units split many ways (the automatic plan of small batches)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("splits", [16, 32])
def test_many_split_workspace_merge(splits):
    """16 and 32 splits per unit (the automatic plan at batch 1-2 for long contexts), merged
    from the workspace: dense attention, the slow step's scores and the fast step against
    the oracle; the counters are left zeroed."""
    sfi = _sfi()
    lens = [8200, 6000, 17, 5100]
    prob = Problem(seed=60 + splits, lens=lens, Hq=16, Hkv=8, D=128, S=4, W=32, heavy_frac=0.02).to_device()
    maxL = 8216
    assert sfi.sfi_plan_splits(prob.shape, prob.B, maxL, splits) == splits
    stride = 8216
    scores = torch.full((prob.B, prob.Hkv, stride), float("nan"), device="cuda")
    out, lse = _dense(prob, num_splits=splits, scores=scores, max_tokens=maxL)
    sc = scores.cpu().numpy()
    for r in range(prob.B):
        o_ref, l_ref = prob.oracle_dense(r)
        assert_close(out[r], o_ref, f"dense out r={r}")
        assert_close(lse[r], l_ref, f"dense lse r={r}")
        L = prob.lens[r]
        ref = prob.oracle_scores(r, stride)
        masked = np.isneginf(ref[:, :L])
        assert np.array_equal(np.isneginf(sc[r, :, :L]), masked)
        err = np.abs(sc[r, :, :L][~masked].astype(np.float64) - ref[:, :L][~masked])
        assert (err <= prob.score_bound(r, stride)[:, :L][~masked]).all(), err.max()
    # the fast step with a selection long enough for the same split count
    _fast_case(70 + splits, [8200, 6000, 5100], 16, 8, 128, 4, 32, [4300, 4100, 4200], 4300, splits=splits)


def test_many_split_workspace_merge_bad_page_and_timeout():
    """32 splits through the workspace: a bad page id (in one split) keeps the unit's
    outputs unwritten, a launch whose waits ran out writes nothing, and the counters are
    left zeroed either way."""
    sfi = _sfi()
    splits = 32
    prob = Problem(seed=81, lens=[8200, 8200], Hq=16, Hkv=8, D=128, S=4, W=32).to_device()
    maxL = 8216
    ws = sfi.alloc_workspace(prob.shape, 2, maxL, splits)
    pt = prob.d_kv.page_table.clone()
    pt[1, 300] = 10_000_000
    bad = sfi.PagedKV(prob.d_kv.k_pool, prob.d_kv.v_pool, pt, prob.d_kv.seq_lens)
    out = torch.full((2, 16, 128), float("nan"), device="cuda")
    lse = torch.full((2, 16), float("nan"), device="cuda")
    st = _status()
    sfi.sfi_slow_dense_attn_with_scores(prob.shape, bad, 4, 32, prob.d_q, out, lse, None, max_tokens=maxL,
                                        num_splits=splits, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 1, f"status {st.item()}"
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    assert np.isnan(o[1]).all() and np.isnan(l[1]).all()
    o_ref, l_ref = prob.oracle_dense(0)
    assert_close(o[0], o_ref, "the healthy request")
    assert counters_zero(ws, 2 * prob.Hkv)
    out.fill_(float("nan"))
    st.zero_()
    sfi.sfi_slow_dense_attn_with_scores(prob.shape, prob.d_kv, 4, 32, prob.d_q, out, None, None, max_tokens=maxL,
                                        num_splits=splits, workspace=ws, dev_status=st,
                                        flags=sfi.SFI_ATTN_TEST_WITHHOLD)
    torch.cuda.synchronize()
    assert st.item() & 16, f"status {st.item()}"
    assert np.isnan(out.cpu().numpy()).all(), "a timed-out launch writes no output"
    assert counters_zero(ws, 2 * prob.Hkv), "split counters must be left zeroed after a timeout"
