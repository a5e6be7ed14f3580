"""Pins of the CPU oracle against what the SFI paper and plain mathematics fix.

None of these tests compares the oracle with a retyped copy of itself. They use
closed forms (one token, equal logits, one dominant logit, a two-token softmax
with a known logit gap), structural encodings (values that spell out their own
position and KV head, so that any wrong index, page, head or set shows up in the
output), algebraic identities between different oracle functions (100% retention
equals dense, as in the paper's Table 1; the sparse state equals dense attention
with every other position masked, as in the Figure 2 caption; split-KV merging
equals one-pass softmax) and brute force on tiny inputs (the Selector against the
dominance definition of a top-k set over every subset).
"""
import itertools
import math

import numpy as np
import pytest

import sfi_synth as syn

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _pool(num_pages, Hkv, P, D, fill=0.0):
    return np.full((num_pages, Hkv, P, D), syn.bf16_bits(np.float32(fill)), np.uint16)


def _set_row(pool, page_row, pos, kv, P, values):
    pool[page_row[pos // P], kv, pos % P] = syn.bf16_bits(values)


# ---------------------------------------------------------------------------
# Softmax closed forms
# ---------------------------------------------------------------------------
def test_single_token_returns_its_value(oracle_lib):
    g = syn.rng(1, 1)
    Hq, Hkv, D, P = 4, 2, 64, 16
    kv = syn.make_paged_kv(g, [1], Hkv, D, P)
    q = syn.normal_bf16(g, (Hq, D))
    out, lse = oracle_lib.dense_attn(q, kv.k_pool, kv.v_pool, kv.page_table[0], 1, Hq, Hkv, D, P)
    for h in range(Hq):
        page = kv.page_table[0, 0]
        v0 = syn.bf16_values(kv.v_pool[page, h // 2, 0])
        k0 = syn.bf16_values(kv.k_pool[page, h // 2, 0])
        assert np.array_equal(out[h], v0)
        assert lse[h] == pytest.approx(float(syn.bf16_values(q[h]) @ k0) / 8.0, rel=1e-14, abs=1e-14)


def test_equal_logits_give_the_mean_and_log_count(oracle_lib):
    g = syn.rng(1, 2)
    Hq, Hkv, D, P, L = 2, 1, 64, 16, 37
    kv = syn.make_paged_kv(g, [L], Hkv, D, P)
    q = np.zeros((Hq, D), np.uint16)  # all logits 0
    out, lse = oracle_lib.dense_attn(q, kv.k_pool, kv.v_pool, kv.page_table[0], L, Hq, Hkv, D, P)
    rows = np.stack([syn.bf16_values(kv.v_pool[kv.page_table[0, j // P], 0, j % P]) for j in range(L)])
    np.testing.assert_allclose(out[0], rows.mean(axis=0), rtol=0, atol=1e-14)
    assert lse[0] == pytest.approx(math.log(L), abs=1e-14)


def test_dominant_logit_selects_its_value(oracle_lib):
    Hq, Hkv, D, P, L = 1, 1, 64, 16, 40
    table = np.arange(3, dtype=np.int32)
    kp, vp = _pool(3, Hkv, P, D), _pool(3, Hkv, P, D)
    g = syn.rng(1, 3)
    for j in range(L):
        _set_row(vp, table, j, 0, P, g.standard_normal(D))
    hot = 23
    kvec = np.zeros(D)
    kvec[0] = 200.0
    _set_row(kp, table, hot, 0, P, kvec)
    q = np.zeros((1, D))
    q[0, 0] = 64.0  # logit of `hot` = 64*200/8 = 1600, all others 0
    out, lse = oracle_lib.dense_attn(syn.bf16_bits(q), kp, vp, table, L, Hq, Hkv, D, P)
    np.testing.assert_array_equal(out[0], syn.bf16_values(vp[1, 0, hot % P]))
    assert lse[0] == pytest.approx(1600.0, abs=1e-9)


def test_two_token_softmax_closed_form(oracle_lib):
    """Logits (0, 1) only if the scale is 1/sqrt(D): p1 = e / (1 + e)."""
    Hq, Hkv, D, P = 1, 1, 64, 16
    table = np.array([0], np.int32)
    kp, vp = _pool(1, Hkv, P, D), _pool(1, Hkv, P, D)
    k1 = np.zeros(D)
    k1[0] = 1.0
    _set_row(kp, table, 1, 0, P, k1)
    v0, v1 = np.full(D, 1.0), np.full(D, -3.0)
    v0[5], v1[5] = 0.5, 2.0
    _set_row(vp, table, 0, 0, P, v0)
    _set_row(vp, table, 1, 0, P, v1)
    q = np.zeros((1, D))
    q[0, 0] = 8.0
    out, lse = oracle_lib.dense_attn(syn.bf16_bits(q), kp, vp, table, 2, Hq, Hkv, D, P)
    e = math.e
    np.testing.assert_allclose(out[0], (v0 + e * v1) / (1 + e), rtol=1e-14, atol=1e-14)
    assert lse[0] == pytest.approx(math.log(1 + e), abs=1e-14)
    gold = dict(l.split("=", 1) for l in open(__file__.replace("test_oracle_pins.py", "golden/two_token_softmax.txt"))
                .read().splitlines() if "=" in l and not l.startswith("#"))
    assert out[0][0] == pytest.approx(float(gold["o_d0"]), abs=1e-15)
    assert out[0][5] == pytest.approx(float(gold["o_d5"]), abs=1e-15)
    assert lse[0] == pytest.approx(float(gold["lse"]), abs=1e-15)


def test_gqa_heads_map_to_contiguous_groups(oracle_lib):
    Hq, Hkv, D, P, L = 8, 2, 64, 16, 5
    table = np.array([0], np.int32)
    kp = syn.normal_bf16(syn.rng(1, 4), (1, Hkv, P, D))
    vp = _pool(1, Hkv, P, D)
    vp[0, 0] = syn.bf16_bits(np.float32(1.0))
    vp[0, 1] = syn.bf16_bits(np.float32(-1.0))
    q = syn.normal_bf16(syn.rng(1, 5), (Hq, D))
    out, _ = oracle_lib.dense_attn(q, kp, vp, table, L, Hq, Hkv, D, P)
    np.testing.assert_allclose(out[:4], 1.0, atol=1e-14)
    np.testing.assert_allclose(out[4:], -1.0, atol=1e-14)


def _position_coded_kv(L, Hkv, D, P, seed, cap=None):
    """Shuffled paged pool whose V row at (pos, kv) is [pos, kv, 0, ...] and K is zero."""
    g = syn.rng(2, seed)
    table, npages = syn.make_page_table(g, [cap or L], P, shuffle=True, spare_pages=3)
    kp, vp = _pool(npages, Hkv, P, D), _pool(npages, Hkv, P, D)
    for kv in range(Hkv):
        for j in range(cap or L):
            row = np.zeros(D)
            row[0], row[1] = j, kv
            _set_row(vp, table[0], j, kv, P, row)
    return table[0], kp, vp


def test_dense_reads_every_position_once_through_the_page_table(oracle_lib):
    Hq, Hkv, D, P, L = 4, 2, 64, 16, 203
    page_row, kp, vp = _position_coded_kv(L, Hkv, D, P, seed=1)
    out, lse = oracle_lib.dense_attn(np.zeros((Hq, D), np.uint16), kp, vp, page_row, L, Hq, Hkv, D, P)
    for h in range(Hq):
        assert out[h, 0] == pytest.approx((L - 1) / 2, abs=1e-11)
        assert out[h, 1] == h // 2
        assert lse[h] == pytest.approx(math.log(L), abs=1e-13)


@pytest.mark.parametrize("L,S,W,sel", [
    (203, 4, 32, [5, 9, 100, 166]),       # sink + selected + recent, recent starts mid-page
    (203, 4, 32, []),                      # k = 0
    (30, 4, 32, []),                       # L <= S + W: the state is all of [0, L)
    (3, 4, 32, []),                        # L < S
    (36, 4, 32, []),                       # L == S + W
    (37, 4, 32, [4]),                      # one candidate, selected
])
def test_fast_step_attends_exactly_sink_selected_recent(oracle_lib, L, S, W, sel):
    """Position-coded V and zero logits: out = mean of the attended positions, lse = ln |state|."""
    Hq, Hkv, D, P = 4, 2, 64, 16
    page_row, kp, vp = _position_coded_kv(L, Hkv, D, P, seed=2 + L)
    k_eff = len(sel)
    cap = S + max(k_eff, 1)
    idx = np.array([sel, sel], np.int32).reshape(Hkv, -1) if k_eff else np.zeros((Hkv, 1), np.int32)
    ck, cv = oracle_lib.compact(kp, vp, page_row, L, S, idx, k_eff, Hkv, D, P, cap)
    out, lse = oracle_lib.fast_attn(np.zeros((Hq, D), np.uint16), ck, cv, k_eff, kp, vp, page_row, L, S, W,
                                    Hq, Hkv, D, P)
    state = sorted(set(range(min(S, L))) | set(sel) | set(range(max(S, L - W), L)))
    assert len(state) == min(S, L) + k_eff + max(0, L - max(S, L - W))  # no overlap between the segments
    for h in range(Hq):
        assert out[h, 0] == pytest.approx(sum(state) / len(state), abs=1e-11)
        assert out[h, 1] == h // 2
        assert lse[h] == pytest.approx(math.log(len(state)), abs=1e-13)


# ---------------------------------------------------------------------------
# Identities between oracle functions
# ---------------------------------------------------------------------------
def _random_request(seed, L, Hq, Hkv, D, P):
    g = syn.rng(3, seed)
    kv = syn.make_paged_kv(g, [L], Hkv, D, P)
    q = syn.normal_bf16(g, (Hq, D))
    return q, kv


@pytest.mark.parametrize("L", [37, 300, 1000])
def test_full_retention_equals_dense(oracle_lib, L):
    """Table 1: 100% retention is the dense computation (speedup 1.00x)."""
    Hq, Hkv, D, P, S, W = 8, 2, 64, 16, 4, 32
    q, kv = _random_request(L, L, Hq, Hkv, D, P)
    pr = kv.page_table[0]
    scores = oracle_lib.group_scores(q, kv.k_pool, pr, L, S, W, Hq, Hkv, D, P)
    nC = max(0, L - S - W)
    idx = np.zeros((Hkv, max(nC, 1)), np.int32)
    for h in range(Hkv):
        sel = oracle_lib.select_topk(scores[h], L, S, W, nC)
        assert len(sel) == nC
        idx[h, :nC] = sel
    ck, cv = oracle_lib.compact(kv.k_pool, kv.v_pool, pr, L, S, idx, nC, Hkv, D, P, S + max(nC, 1))
    fo, fl = oracle_lib.fast_attn(q, ck, cv, nC, kv.k_pool, kv.v_pool, pr, L, S, W, Hq, Hkv, D, P)
    do, dl = oracle_lib.dense_attn(q, kv.k_pool, kv.v_pool, pr, L, Hq, Hkv, D, P)
    np.testing.assert_allclose(fo, do, rtol=0, atol=1e-12)
    np.testing.assert_allclose(fl, dl, rtol=0, atol=1e-12)


def test_sparse_state_equals_masked_dense(oracle_lib):
    """Figure 2: the fast step is dense attention over sink + selected + recent only."""
    Hq, Hkv, D, P, S, W, L, k = 8, 2, 64, 16, 4, 32, 500, 40
    q, kv = _random_request(7, L, Hq, Hkv, D, P)
    pr = kv.page_table[0]
    scores = oracle_lib.group_scores(q, kv.k_pool, pr, L, S, W, Hq, Hkv, D, P)
    idx = np.stack([oracle_lib.select_topk(scores[h], L, S, W, k) for h in range(Hkv)])
    ck, cv = oracle_lib.compact(kv.k_pool, kv.v_pool, pr, L, S, idx, k, Hkv, D, P, S + k)
    fo, fl = oracle_lib.fast_attn(q, ck, cv, k, kv.k_pool, kv.v_pool, pr, L, S, W, Hq, Hkv, D, P)
    pos = np.stack([np.concatenate([np.arange(S), idx[h], np.arange(L - W, L)]) for h in range(Hkv)])
    mo, ml = oracle_lib.index_attn(q, kv.k_pool, kv.v_pool, pr, pos, Hq, Hkv, D, P)
    np.testing.assert_allclose(fo, mo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(fl, ml, rtol=0, atol=1e-12)
    # and it is not the dense result (the selection matters)
    do, _ = oracle_lib.dense_attn(q, kv.k_pool, kv.v_pool, pr, L, Hq, Hkv, D, P)
    assert np.abs(fo - do).max() > 1e-3


@pytest.mark.parametrize("chunks", [1, 2, 3, 7, "L", "empty"])
def test_split_merge_equals_one_pass(oracle_lib, chunks):
    Hq, Hkv, D, P, L = 4, 2, 128, 16, 331
    q, kv = _random_request(11, L, Hq, Hkv, D, P)
    pr = kv.page_table[0]
    do, dl = oracle_lib.dense_attn(q, kv.k_pool, kv.v_pool, pr, L, Hq, Hkv, D, P)
    if chunks == "L":
        bounds = np.arange(L + 1)
    elif chunks == "empty":
        bounds = np.array([0, 0, 100, 100, 100, 250, L])
    else:
        bounds = np.linspace(0, L, chunks + 1).round().astype(int)
    for h in range(Hq):
        o, l = oracle_lib.split_merge_attn(q[h], h // 2, kv.k_pool, kv.v_pool, pr, bounds, Hkv, D, P)
        np.testing.assert_allclose(o, do[h], rtol=0, atol=1e-12)
        assert l == pytest.approx(dl[h], abs=1e-12)


# ---------------------------------------------------------------------------
# Masked group-summed logits
# ---------------------------------------------------------------------------
def test_group_scores_closed_form_and_mask(oracle_lib):
    """q_{kv*G+g} = c_{kv,g} e_g and k_j = [j mod 7, 1, (j mod 3) - 1, 0...]:
    score_kv(j) = (c_{kv,0} (j mod 7) + c_{kv,1}) / 8 on [S, L-W), -inf elsewhere below L."""
    Hq, Hkv, D, P, L, S, W = 4, 2, 64, 16, 90, 5, 20
    G = Hq // Hkv
    c = np.array([[3.0, -2.0], [0.5, 7.0]])
    page_row, kp, _ = _position_coded_kv(L, Hkv, D, P, seed=9)
    for kv in range(Hkv):
        for j in range(L):
            row = np.zeros(D)
            row[0], row[1], row[2] = j % 7, 1.0, (j % 3) - 1
            _set_row(kp, page_row, j, kv, P, row)
    q = np.zeros((Hq, D))
    for kv in range(Hkv):
        for gg in range(G):
            q[kv * G + gg, gg] = c[kv, gg]
    stride = 96
    sc = oracle_lib.group_scores(syn.bf16_bits(q), kp, page_row, L, S, W, Hq, Hkv, D, P, stride=stride)
    for kv in range(Hkv):
        for j in range(stride):
            if j >= L:
                assert np.isnan(sc[kv, j])  # untouched
            elif S <= j < L - W:
                assert sc[kv, j] == np.float32((c[kv, 0] * (j % 7) + c[kv, 1]) / 8.0)
            else:
                assert sc[kv, j] == -np.inf


def test_group_scores_rounds_the_double_sum_once(oracle_lib):
    """The group sum is formed exactly and rounded to fp32 once (nearest-even).

    Head 0 contributes 1 + 2^-24 (a tie that alone would round down to 1), head 1
    contributes 2^-26; the exact sum 1 + 1.25 * 2^-24 rounds up to 1 + 2^-23.
    """
    Hq, Hkv, D, P, L, S, W = 2, 1, 64, 16, 3, 0, 0
    table = np.array([0], np.int32)
    kp = _pool(1, 1, P, D)
    row = np.zeros(D)
    row[0], row[1], row[2] = 1.0, 1.0, 1.0
    _set_row(kp, table, 1, 0, P, row)
    q = np.zeros((2, D))
    q[0, 0], q[0, 2] = 8.0, 8.0 * 2.0 ** -24
    q[1, 1] = 8.0 * 2.0 ** -26
    sc = oracle_lib.group_scores(syn.bf16_bits(q), kp, table, L, S, W, Hq, Hkv, D, P)
    assert sc[0, 1] == np.float32(1.0 + 2.0 ** -23) and sc[0, 0] == 0.0
    q[1, 1] = 0.0  # alone, 1 + 2^-24 is a tie and rounds to even (1.0)
    sc = oracle_lib.group_scores(syn.bf16_bits(q), kp, table, L, S, W, Hq, Hkv, D, P)
    assert sc[0, 1] == np.float32(1.0)


# ---------------------------------------------------------------------------
# Selector
# ---------------------------------------------------------------------------
def _beats(a, b):
    """Total order of the Selector, written as a pairwise rule: does candidate a beat b?
    a, b = (score, position). NaN loses to every number; -0 == +0; equal -> lower position."""
    (sa, ia), (sb, ib) = a, b
    na, nb = math.isnan(sa), math.isnan(sb)
    if na != nb:
        return nb
    if not na and sa != sb:
        return sa > sb
    return ia < ib


def _brute_topk(vals, S, k):
    """The unique k-subset whose every member beats every non-member, found by trying all subsets."""
    items = [(float(v), S + i) for i, v in enumerate(vals)]
    k = min(k, len(items))
    winners = []
    for sub in itertools.combinations(range(len(items)), k):
        inside = set(sub)
        if all(_beats(items[i], items[j]) for i in inside for j in range(len(items)) if j not in inside):
            winners.append(sorted(items[i][1] for i in sub))
    assert len(winners) == 1
    return winners[0]


@pytest.mark.parametrize("trial", range(60))
def test_selector_matches_brute_force_on_tiny_inputs(oracle_lib, trial):
    g = syn.rng(4, trial)
    n = int(g.integers(1, 11))
    palette = np.array([1.5, -0.25, 1.5, 0.0, -0.0, -np.inf, np.nan, 3.0], np.float32)
    pal = palette[: 3 + trial % 6]
    vals = pal[g.integers(0, len(pal), size=n)]
    S, W = int(g.integers(0, 4)), int(g.integers(0, 4))
    L = S + n + W
    row = np.full(L, 77.0, np.float32)  # outside C: must be ignored
    row[S:S + n] = vals
    for k in range(0, n + 2):
        got = oracle_lib.select_topk(row, L, S, W, k)
        assert list(got) == _brute_topk(vals, S, k), (vals, k)


def test_selector_ties_go_to_lower_positions(oracle_lib):
    L, S, W = 100, 4, 8
    row = np.zeros(L, np.float32)
    assert list(oracle_lib.select_topk(row, L, S, W, 10)) == list(range(S, S + 10))
    row[:] = -np.inf
    hot = [90, 17, 55, 4, 60]
    row[hot] = 1.0
    row[95] = 5.0  # in the recent window: not a candidate
    assert list(oracle_lib.select_topk(row, L, S, W, 5)) == sorted(hot)
    assert list(oracle_lib.select_topk(row, L, S, W, 7)) == sorted(hot + [5, 6])
    assert len(oracle_lib.select_topk(row, L, S, W, 1000)) == L - S - W


def test_selector_planted_zipf_ties(oracle_lib):
    """A Zipf profile with the band around rank k tied: the threshold group is cut by position."""
    n, k, S, W = 5000, 400, 64, 256
    g = syn.rng(4, 999)
    vals = syn.zipf_scores_with_ties(g, n, k)
    L = S + n + W
    row = np.full(L, -np.inf, np.float32)
    row[S:S + n] = vals
    got = oracle_lib.select_topk(row, L, S, W, k)
    thr = np.sort(vals)[::-1][k - 1]
    above = [S + i for i in range(n) if vals[i] > thr]
    eq = [S + i for i in range(n) if vals[i] == thr]
    assert len(above) < k <= len(above) + len(eq)
    assert list(got) == sorted(above + eq[:k - len(above)])


# ---------------------------------------------------------------------------
# Compaction and append
# ---------------------------------------------------------------------------
def test_compaction_copies_sink_then_selection_bit_for_bit(oracle_lib):
    Hkv, D, P, L, S = 2, 64, 16, 150, 4
    page_row, _, vp = _position_coded_kv(L, Hkv, D, P, seed=21)
    kp = syn.normal_bf16(syn.rng(5, 1), vp.shape)
    idx = np.array([[7, 8, 40, 99], [4, 50, 51, 113]], np.int32)
    cap = S + 6
    ck, cv = oracle_lib.compact(kp, vp, page_row, L, S, idx, 4, Hkv, D, P, cap)
    for kv in range(Hkv):
        want = list(range(S)) + list(idx[kv])
        for row, pos in enumerate(want):
            assert syn.bf16_values(cv[kv, row, :2]).tolist() == [pos, kv]
            page, slot = page_row[pos // P], pos % P
            assert np.array_equal(ck[kv, row], kp[page, kv, slot])
        assert not ck[kv, S + 4:].any() and not cv[kv, S + 4:].any()  # rows past k_eff untouched


def test_compaction_short_request_copies_partial_sink(oracle_lib):
    Hkv, D, P, L, S = 1, 64, 16, 3, 4
    page_row, kp, vp = _position_coded_kv(L, Hkv, D, P, seed=22)
    ck, cv = oracle_lib.compact(kp, vp, page_row, L, S, np.zeros((1, 1), np.int32), 0, Hkv, D, P, S + 1)
    assert [syn.bf16_values(cv[0, r, 0]) for r in range(3)] == [0, 1, 2]
    assert not cv[0, 3:].any()


def test_append_writes_only_the_last_slot(oracle_lib):
    Hkv, D, P = 2, 64, 16
    g = syn.rng(6, 1)
    kv = syn.make_paged_kv(g, [40], Hkv, D, P, capacity_tokens=[64])
    kp, vp = kv.k_pool.copy(), kv.v_pool.copy()
    kn, vn = syn.normal_bf16(g, (Hkv, D)), syn.normal_bf16(g, (Hkv, D))
    oracle_lib.paged_append(kp, vp, kv.page_table[0], 41, kn, vn, Hkv, D, P)
    page, slot = kv.page_table[0, 40 // P], 40 % P
    assert np.array_equal(kp[page, :, slot], kn) and np.array_equal(vp[page, :, slot], vn)
    kp[page, :, slot] = kv.k_pool[page, :, slot]
    vp[page, :, slot] = kv.v_pool[page, :, slot]
    assert np.array_equal(kp, kv.k_pool) and np.array_equal(vp, kv.v_pool)


# ---------------------------------------------------------------------------
# Schedule
# ---------------------------------------------------------------------------
def test_schedule_interval_and_boundaries(oracle_lib):
    steps, batch = 70, 3
    b = np.zeros((steps, batch), np.uint8)
    b[5, 1] = 1
    b[6, 1] = 1
    b[40, 2] = 1
    m = oracle_lib.schedule(b, 16)
    assert np.flatnonzero(m[:, 0]).tolist() == [0, 16, 32, 48, 64]
    assert np.flatnonzero(m[:, 1]).tolist() == [0, 5, 6, 22, 38, 54]
    assert np.flatnonzero(m[:, 2]).tolist() == [0, 16, 32, 40, 56]


# ---------------------------------------------------------------------------
# Several query tokens: draft over the sparse state, verification over the whole
# context ("A Sparse Glimpse of the Whole", abstract; the T tokens sit at positions
# L - T .. L - 1 and token t sees the context up to its own position)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("L,T", [(203, 1), (203, 5), (40, 3), (16, 16), (37, 9)])
def test_verify_is_causal_prefix_mean(oracle_lib, L, T):
    """Zero logits and position-coded V: token t averages positions 0 .. L - T + t."""
    Hq, Hkv, D, P = 4, 2, 64, 16
    page_row, kp, vp = _position_coded_kv(L, Hkv, D, P, seed=40 + L + T)
    out, lse = oracle_lib.verify_attn(np.zeros((T, Hq, D), np.uint16), kp, vp, page_row, L, T, Hq, Hkv, D, P)
    for t in range(T):
        n = L - T + t + 1
        for h in range(Hq):
            assert out[t, h, 0] == pytest.approx((n - 1) / 2, abs=1e-11)
            assert out[t, h, 1] == h // 2
            assert lse[t, h] == pytest.approx(math.log(n), abs=1e-13)


def test_verify_tokens_see_nothing_after_themselves(oracle_lib):
    """Changing K/V after position L - T + t, or another token's query, leaves token t unchanged."""
    Hq, Hkv, D, P, L, T = 8, 2, 64, 16, 150, 6
    g = syn.rng(3, 77)
    kv = syn.make_paged_kv(g, [L], Hkv, D, P)
    pr = kv.page_table[0]
    q = syn.normal_bf16(g, (T, Hq, D))
    base, base_l = oracle_lib.verify_attn(q, kv.k_pool, kv.v_pool, pr, L, T, Hq, Hkv, D, P)
    t_cut = 2
    kp, vp = kv.k_pool.copy(), kv.v_pool.copy()
    for j in range(L - T + t_cut + 1, L):
        for h in range(Hkv):
            kp[pr[j // P], h, j % P] = syn.normal_bf16(g, (D,))
            vp[pr[j // P], h, j % P] = syn.normal_bf16(g, (D,))
    o2, l2 = oracle_lib.verify_attn(q, kp, vp, pr, L, T, Hq, Hkv, D, P)
    assert np.array_equal(o2[:t_cut + 1], base[:t_cut + 1]) and np.array_equal(l2[:t_cut + 1], base_l[:t_cut + 1])
    assert np.abs(o2[t_cut + 1:] - base[t_cut + 1:]).max() > 1e-3
    q2 = q.copy()
    q2[4] = syn.normal_bf16(g, (Hq, D))
    o3, _ = oracle_lib.verify_attn(q2, kv.k_pool, kv.v_pool, pr, L, T, Hq, Hkv, D, P)
    keep = [t for t in range(T) if t != 4]
    assert np.array_equal(o3[keep], base[keep]) and np.abs(o3[4] - base[4]).max() > 1e-3


@pytest.mark.parametrize("L,T,S,W,sel", [
    (203, 4, 4, 32, [5, 9, 100, 166]),     # windows shift by one position per token
    (203, 6, 4, 3, [5, 9, 100]),           # W < T: every token's window is disjoint from the first's
    (10, 4, 12, 32, []),                   # L - T + 1 < S: the sink grows with the token
    (12, 12, 4, 6, []),                    # T = L
])
def test_fast_multi_attends_each_tokens_sparse_state(oracle_lib, L, T, S, W, sel):
    """Zero logits and position-coded V: token t averages sink + selection + its own recent window."""
    Hq, Hkv, D, P = 4, 2, 64, 16
    page_row, kp, vp = _position_coded_kv(L, Hkv, D, P, seed=60 + L + T)
    k_eff = len(sel)
    cap = S + max(k_eff, 1)
    idx = np.array([sel, sel], np.int32).reshape(Hkv, -1) if k_eff else np.zeros((Hkv, 1), np.int32)
    ck, cv = oracle_lib.compact(kp, vp, page_row, L, S, idx, k_eff, Hkv, D, P, cap)
    out, lse = oracle_lib.fast_multi_attn(np.zeros((T, Hq, D), np.uint16), ck, cv, k_eff, kp, vp, page_row, L, T,
                                          S, W, Hq, Hkv, D, P)
    for t in range(T):
        Lt = L - T + t + 1
        state = sorted(set(range(min(S, Lt))) | set(sel) | set(range(max(S, Lt - W), Lt)))
        for h in range(Hq):
            assert out[t, h, 0] == pytest.approx(sum(state) / len(state), abs=1e-11)
            assert out[t, h, 1] == h // 2
            assert lse[t, h] == pytest.approx(math.log(len(state)), abs=1e-13)


def test_fast_multi_equals_masked_dense_per_token(oracle_lib):
    """Random data: token t equals dense attention restricted to its explicit position set."""
    Hq, Hkv, D, P, S, W, L, T, k = 8, 2, 64, 16, 4, 24, 400, 5, 30
    g = syn.rng(3, 91)
    kv = syn.make_paged_kv(g, [L], Hkv, D, P)
    pr = kv.page_table[0]
    q = syn.normal_bf16(g, (T, Hq, D))
    L0 = L - T + 1
    idx = np.stack([np.sort(g.choice(np.arange(S, L0 - W), k, replace=False)) for _ in range(Hkv)]).astype(np.int32)
    ck, cv = oracle_lib.compact(kv.k_pool, kv.v_pool, pr, L0, S, idx, k, Hkv, D, P, S + k)
    out, lse = oracle_lib.fast_multi_attn(q, ck, cv, k, kv.k_pool, kv.v_pool, pr, L, T, S, W, Hq, Hkv, D, P)
    for t in range(T):
        Lt = L0 + t
        pos = np.stack([np.concatenate([np.arange(S), idx[h], np.arange(Lt - W, Lt)]) for h in range(Hkv)])
        mo, ml = oracle_lib.index_attn(q[t], kv.k_pool, kv.v_pool, pr, pos.astype(np.int32), Hq, Hkv, D, P)
        np.testing.assert_allclose(out[t], mo, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[t], ml, rtol=0, atol=1e-12)


@pytest.mark.parametrize("which", ["first", "last"])
def test_fast_multi_full_retention_meets_verify(oracle_lib, which):
    """Table 1's 100%-retention identity, per token: with every candidate of C(L_t) selected, token t's
    sparse state is all of [0, L_t), so it equals the verification's token t."""
    Hq, Hkv, D, P, S, W, L, T = 8, 2, 64, 16, 4, 24, 300, 6
    g = syn.rng(3, 93)
    kv = syn.make_paged_kv(g, [L], Hkv, D, P)
    pr = kv.page_table[0]
    q = syn.normal_bf16(g, (T, Hq, D))
    t = 0 if which == "first" else T - 1
    Lt = L - T + t + 1
    nC = Lt - W - S
    idx = np.tile(np.arange(S, Lt - W, dtype=np.int32), (Hkv, 1))
    ck, cv = oracle_lib.compact(kv.k_pool, kv.v_pool, pr, Lt, S, idx, nC, Hkv, D, P, S + nC)
    fo, fl = oracle_lib.fast_multi_attn(q, ck, cv, nC, kv.k_pool, kv.v_pool, pr, L, T, S, W, Hq, Hkv, D, P)
    vo, vl = oracle_lib.verify_attn(q, kv.k_pool, kv.v_pool, pr, L, T, Hq, Hkv, D, P)
    np.testing.assert_allclose(fo[t], vo[t], rtol=0, atol=1e-12)
    np.testing.assert_allclose(fl[t], vl[t], rtol=0, atol=1e-12)
    other = T - 1 - t
    assert np.abs(fo[other] - vo[other]).max() > 1e-4  # the others miss part of their context


@pytest.mark.parametrize("T,W", [(5, 2), (4, 40), (1, 20)])
def test_verify_scores_closed_form_and_mask(oracle_lib, T, W):
    """q_{t, kv*G+g} = c_{t,kv,g} e_g and k_j = [j mod 7, 1, 0...]: the statistic of candidate j is
    (sum over the tokens that see j of c_{t,kv,0} (j mod 7) + c_{t,kv,1}) / 8 on [S, L - W)."""
    Hq, Hkv, D, P, L, S = 4, 2, 64, 16, 90, 5
    G = Hq // Hkv
    g = syn.rng(3, 95 + T)
    c = np.round(g.standard_normal((T, Hkv, G)) * 4) / 4  # exact in bf16
    page_row, kp, _ = _position_coded_kv(L, Hkv, D, P, seed=19)
    for kv in range(Hkv):
        for j in range(L):
            row = np.zeros(D)
            row[0], row[1] = j % 7, 1.0
            _set_row(kp, page_row, j, kv, P, row)
    q = np.zeros((T, Hq, D))
    for t in range(T):
        for kv in range(Hkv):
            for gg in range(G):
                q[t, kv * G + gg, gg] = c[t, kv, gg]
    stride = 96
    sc = oracle_lib.verify_scores(syn.bf16_bits(q), kp, page_row, L, T, S, W, Hq, Hkv, D, P, stride=stride)
    for kv in range(Hkv):
        for j in range(stride):
            if j >= L:
                assert np.isnan(sc[kv, j])
            elif S <= j < L - W:
                seers = [t for t in range(T) if j < L - T + t + 1]
                want = sum(c[t, kv, 0] * (j % 7) + c[t, kv, 1] for t in seers) / 8.0
                assert sc[kv, j] == np.float32(want)
            else:
                assert sc[kv, j] == -np.inf
    if T == 1:  # one token: the slow step's statistic
        one = oracle_lib.group_scores(syn.bf16_bits(q[0]), kp, page_row, L, S, W, Hq, Hkv, D, P, stride=stride)
        np.testing.assert_array_equal(sc, one)


def test_append_tokens_writes_exactly_the_last_t_slots(oracle_lib):
    Hkv, D, P, L, T = 2, 64, 16, 45, 7
    g = syn.rng(6, 2)
    kv = syn.make_paged_kv(g, [L - T], Hkv, D, P, capacity_tokens=[64])
    kp, vp = kv.k_pool.copy(), kv.v_pool.copy()
    kn, vn = syn.normal_bf16(g, (T, Hkv, D)), syn.normal_bf16(g, (T, Hkv, D))
    oracle_lib.paged_append_tokens(kp, vp, kv.page_table[0], L, T, kn, vn, Hkv, D, P)
    for t in range(T):
        pos = L - T + t
        page, slot = kv.page_table[0, pos // P], pos % P
        assert np.array_equal(kp[page, :, slot], kn[t]) and np.array_equal(vp[page, :, slot], vn[t])
        kp[page, :, slot] = kv.k_pool[page, :, slot]
        vp[page, :, slot] = kv.v_pool[page, :, slot]
    assert np.array_equal(kp, kv.k_pool) and np.array_equal(vp, kv.v_pool)
