"""Plant plausible mistakes in a copy of the oracle and require the pins to catch each.

Each entry rewrites one line of the oracle's C source (a dropped term, a wrong
index, a flipped comparison, an off-by-one), compiles that copy on the CPU and runs
the pins named beside it against the copy: at least one of them must fail. The
mutated copies live in a temporary directory; the real oracle is never touched.
"""
import pytest

import oracle
from tests import test_oracle_pins as pins

O = oracle


def _fast_set(L, S, W, sel):
    return lambda: pins.test_fast_step_attends_exactly_sink_selected_recent(O, L, S, W, sel)


MUTATIONS = [
    ("scale 1/D instead of 1/sqrt(D)", "1.0 / sqrt((double)D)", "1.0 / (double)D",
     [lambda: pins.test_two_token_softmax_closed_form(O)]),
    ("query head mapped by h % Hkv", "int kv = h / G;", "int kv = h % Hkv;",
     [lambda: pins.test_gqa_heads_map_to_contiguous_groups(O)]),
    ("no max subtraction in softmax", "double p = exp(s[j] - m);", "double p = exp(s[j]) / exp(m);",
     [lambda: pins.test_dominant_logit_selects_its_value(O)]),
    ("lse without the max", "*lse = m + log(l);", "*lse = log(l);",
     [lambda: pins.test_single_token_returns_its_value(O)]),
    ("dense drops the last position", "attend_rows(qd, kr, vr, L, D", "attend_rows(qd, kr, vr, L > 1 ? L - 1 : L, D",
     [lambda: pins.test_dense_reads_every_position_once_through_the_page_table(O)]),
    ("recent window one short", "int rs = (L - W) > S ? (L - W) : S;", "int rs = (L - W) > S ? (L - W) + 1 : S;",
     [_fast_set(203, 4, 32, [5, 9, 100, 166])]),
    ("sink not clamped to L", "int ns = S < L ? S : L;\n    int n_compact", "int ns = S;\n    int n_compact",
     [_fast_set(3, 4, 32, [])]),
    ("selection dropped from the fast step", "int n_compact = ns + count;", "int n_compact = ns;",
     [_fast_set(203, 4, 32, [5, 9, 100, 166])]),
    ("ties go to the higher position", "return (ia > ib) - (ia < ib);", "return (ia < ib) - (ia > ib);",
     [lambda: pins.test_selector_ties_go_to_lower_positions(O)]),
    ("NaN ranked above numbers", "return na ? 1 : -1;", "return na ? -1 : 1;",
     [lambda: [pins.test_selector_matches_brute_force_on_tiny_inputs(O, t) for t in range(60)]]),
    ("recent window counted as candidates", "int n = L - W - S;", "int n = L - S;",
     [lambda: pins.test_selector_ties_go_to_lower_positions(O)]),
    ("scores not scaled", "sigma += scale * acc;", "sigma += acc;",
     [lambda: pins.test_group_scores_closed_form_and_mask(O)]),
    ("scores summed over the wrong heads", "widen_query(q + (size_t)(kv * G + g) * D",
     "widen_query(q + (size_t)(g * Hkv + kv) * D", [lambda: pins.test_group_scores_closed_form_and_mask(O)]),
    ("recent positions not masked in scores", "if (j < c_lo || j >= c_hi) {", "if (j < c_lo) {",
     [lambda: pins.test_group_scores_closed_form_and_mask(O)]),
    ("scores rounded through float per head", "sigma += scale * acc;", "sigma = (float)(sigma + scale * acc);",
     [lambda: pins.test_group_scores_rounds_the_double_sum_once(O)]),
    ("compaction uses head 0's selection", "int pos = idx[(size_t)kv * idx_stride + t];", "int pos = idx[t];",
     [lambda: pins.test_compaction_copies_sink_then_selection_bit_for_bit(O)]),
    ("split merge without rescaling", "double w = exp(mc[c] - m);", "double w = 1.0;",
     [lambda: pins.test_split_merge_equals_one_pass(O, 3)]),
    ("append one slot late", "int pos = L - 1;", "int pos = L;",
     [lambda: pins.test_append_writes_only_the_last_slot(O)]),
    ("verification not causal", "page_row, L - T + t + 1, Hq, Hkv", "page_row, L, Hq, Hkv",
     [lambda: pins.test_verify_is_causal_prefix_mean(O, 40, 3)]),
    ("verification shifted by one position", "page_row, L - T + t + 1, Hq, Hkv", "page_row, L - T + t, Hq, Hkv",
     [lambda: pins.test_verify_is_causal_prefix_mean(O, 40, 3)]),
    ("multi-token draft shares the last token's window", "page_row, L - T + t + 1, S, W,", "page_row, L, S, W,",
     [lambda: pins.test_fast_multi_attends_each_tokens_sparse_state(O, 203, 4, 4, 32, [5, 9, 100, 166])]),
    ("verification statistic ignores causality", "if (j > L - T + t) continue;", "if (j > L) continue;",
     [lambda: pins.test_verify_scores_closed_form_and_mask(O, 5, 2)]),
    ("verification statistic from the last token only", "for (int t = 0; t < T; ++t) {\n                if (j >",
     "for (int t = T - 1; t < T; ++t) {\n                if (j >",
     [lambda: pins.test_verify_scores_closed_form_and_mask(O, 4, 40)]),
    ("token append one slot early", "page_row, L - T + t + 1, k_new", "page_row, L - T + t, k_new",
     [lambda: pins.test_append_tokens_writes_exactly_the_last_t_slots(O)]),
    ("refresh interval off by one", "(t - last_slow >= interval)", "(t - last_slow > interval)",
     [lambda: pins.test_schedule_interval_and_boundaries(O)]),
]


@pytest.mark.parametrize("name,old,new,catchers", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new, catchers):
    src = oracle.source()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    so = oracle.build_variant(src.replace(old, new), str(tmp_path), "mutant")
    caught = 0
    with oracle.use_library(so):
        for run in catchers:
            try:
                run()
            except AssertionError:
                caught += 1
    assert caught > 0, f"no pin caught: {name}"
