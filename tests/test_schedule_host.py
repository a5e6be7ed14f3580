"""Host schedule (slow/fast decisions) and compact layout, against the oracle's
schedule on the seeded boundary process of the ragged mixed-batch workload."""
import numpy as np
import pytest

import sfi_synth as syn


def test_schedule_matches_oracle_on_boundary_process(oracle_lib):
    from sparse_kv_long_sfi_gb300.runtime import SlowFastSchedule
    steps, batch = 300, 64
    b = syn.boundary_draws(syn.rng(50, 1), steps, batch, 0.06)
    want = oracle_lib.schedule(b, 32)
    s = SlowFastSchedule(batch, 32)
    got = np.stack([s.next(b[t]) for t in range(steps)])
    np.testing.assert_array_equal(got, want)
    gaps = [np.diff(np.flatnonzero(want[:, r])) for r in range(batch)]
    assert max(g.max() for g in gaps) == 32          # forced refresh
    assert 10 < np.mean(np.concatenate(gaps)) < 18   # ~1/(p + 1/32) for p = 0.06


def test_fixed_interval_schedule(oracle_lib):
    from sparse_kv_long_sfi_gb300.runtime import SlowFastSchedule
    s = SlowFastSchedule(3, 16)
    modes = np.stack([s.next() for _ in range(40)])
    assert np.flatnonzero(modes[:, 0]).tolist() == [0, 16, 32]
    np.testing.assert_array_equal(modes, oracle_lib.schedule(np.zeros((40, 3), np.uint8), 16))


def test_retention_budgets_match_table1_ratios():
    """Table 1's retention ratios at KV length 16K are token budgets n * 256 (n/64 of 16384)."""
    printed = [1.6, 6.3, 12.5, 25.0, 37.5, 50.0, 75.0, 98.4, 100.0]
    n = [1, 4, 8, 16, 24, 32, 48, 63, 64]
    for pct, m in zip(printed, n):
        assert abs(100 * m / 64 - pct) <= 0.05 + 1e-9  # printed to one decimal
    S, W, L = 64, 256, 16384
    ks = [syn.retention_budget(m / 64, L, S, W) for m in n]
    assert ks == [0, 704, 1728, 3776, 5824, 7872, 11968, 15808, 16064]
