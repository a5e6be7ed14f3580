"""Full-size parity: the five workloads at their real sizes, run through the host
runtime (SFIDecoder: fused append, main + aux streams) in the launch configuration
the benchmark uses, with the CPU oracle recomputing sampled requests one by one.

Selection is checked bit-exactly on every (request, KV head) by running the oracle's
Selector on the GPU-written fp32 scores; compaction bytes and attention outputs are
checked on the sampled requests against the oracle on those requests' pages.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import sfi_synth as syn
from tests.gpu_harness import assert_close, host_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from sparse_kv_long_sfi_gb300 import build
    build.build()
    oracle.build()


class Workload:
    """Seeded device-resident batch: shuffled page table, per-layer pools, queries and
    new tokens for a few steps."""

    def __init__(self, seed, lens, Hq, Hkv, D, S, W, k_per_req, steps=3, layers=1, heavy_frac=0.0,
                 k_cap=None, single_launch_mixed=True, ragged=False):
        import sparse_kv_long_sfi_gb300 as sfi
        self.sfi = sfi
        self.Hq, self.Hkv, self.D, self.P, self.S, self.W = Hq, Hkv, D, 16, S, W
        self.lens0 = np.asarray(lens, np.int64)
        self.B = len(lens)
        self.steps = steps
        self.shape = sfi.AttnShape(Hq, Hkv, D)
        g = syn.rng(seed, 0)
        table, num_pages = syn.make_page_table(g, self.lens0 + steps + 1, 16, shuffle=True)
        self.table = table
        dev = torch.device("cuda")
        self.k_per_req = np.asarray(k_per_req, np.int64)
        k_cap = int(k_cap or max(1, self.k_per_req.max()))
        off, cap = sfi.compact_layout(self.shape, S, [k_cap] * self.B)
        self.batch = sfi.DecodeBatch(torch.as_tensor(table).to(dev), off, cap,
                                     torch.as_tensor(self.k_per_req.astype(np.int32)).to(dev), k_cap,
                                     score_stride=int(self.lens0.max()) + steps + 1)
        self.q = torch.empty((steps, layers, self.B, Hq, D), dtype=torch.bfloat16, device=dev)
        self.kn = torch.empty((steps, layers, self.B, Hkv, D), dtype=torch.bfloat16, device=dev)
        self.vn = torch.empty_like(self.kn)
        syn.device_normal_bf16_(self.q, syn.stream_seed(seed, 1))
        syn.device_normal_bf16_(self.kn, syn.stream_seed(seed, 2))
        syn.device_normal_bf16_(self.vn, syn.stream_seed(seed, 3))
        lens_t = torch.as_tensor(self.lens0.astype(np.int32)).to(dev)

        def init(i, kp, vp):
            syn.device_normal_bf16_(kp, syn.stream_seed(seed, 10, i))
            syn.device_normal_bf16_(vp, syn.stream_seed(seed, 11, i))
            if heavy_frac > 0:
                syn.device_plant_heavy_hitters_(kp, self.batch.page_table, self.q[0, i], lens_t, S, W, heavy_frac,
                                                3.0, syn.stream_seed(seed, 12, i))

        self.layers = sfi.allocate_layers(self.shape, layers, num_pages, self.batch, S, device=dev, pool_init=init)
        self.out = torch.zeros((layers, self.B, Hq, D), dtype=torch.float32, device=dev)
        self.lse = torch.zeros((layers, self.B, Hq), dtype=torch.float32, device=dev)
        self.dec = sfi.SFIDecoder(self.shape, self.layers, self.batch, S, W, max_len=int(self.lens0.max()) + steps + 1,
                                  single_launch_mixed=single_launch_mixed, ragged=ragged)
        self.cur = self.lens0.copy()

    def io(self, t):
        return self.sfi.StepIO(self.q[t], self.kn[t], self.vn[t], self.out, self.lse)

    def seq_lens(self):
        return torch.as_tensor(self.cur.astype(np.int32)).cuda()

    def host_pages(self, layer, r):
        """The request's pages (after every step so far) as a small host pool + local page row."""
        n = int(math.ceil(self.cur[r] / 16))
        pages = torch.as_tensor(self.table[r, :n].astype(np.int64)).cuda()
        Lb = self.layers[layer]
        return (host_bf16(Lb.k_pool[pages]), host_bf16(Lb.v_pool[pages]), np.arange(n, dtype=np.int32))

    def host_q(self, t, layer, r):
        return host_bf16(self.q[t, layer, r])


def _check_slow(w, t, layer, sampled):
    """After a slow step: selection bit-exact everywhere; sampled requests' attention,
    scores and compaction against the oracle."""
    L = w.layers[layer]
    torch.cuda.synchronize()
    assert w.dec.dev_status.item() == 0
    scores = L.scores.cpu().numpy()
    idx = L.idx.cpu().numpy()
    count = L.compact.count.cpu().numpy()
    for r in range(w.B):
        if not w.slow_mask[r]:
            continue
        for h in range(w.Hkv):
            want = oracle.select_topk(scores[r, h], w.cur[r], w.S, w.W, w.k_now[r])
            assert count[r] == len(want)
            np.testing.assert_array_equal(idx[r, h, :len(want)], want, err_msg=f"selection r={r} kv={h}")
    ck, cv = L.compact.k, L.compact.v
    off, cap = L.compact.row_offset.cpu().numpy(), L.compact.capacity.cpu().numpy()
    out, lse = w.out[layer].cpu().numpy(), w.lse[layer].cpu().numpy()
    for r in sampled:
        if not w.slow_mask[r]:
            continue
        kp, vp, pr = w.host_pages(layer, r)
        q = w.host_q(t, layer, r)
        o_ref, l_ref = oracle.dense_attn(q, kp, vp, pr, w.cur[r], w.Hq, w.Hkv, w.D, 16)
        assert_close(out[r], o_ref, f"slow out r={r} t={t}")
        assert_close(lse[r], l_ref, f"slow lse r={r} t={t}")
        keff = count[r]
        rk, rv = oracle.compact(kp, vp, pr, w.cur[r], w.S, idx[r], keff, w.Hkv, w.D, 16, cap[r])
        ns = min(w.S, w.cur[r])
        rows = torch.as_tensor(np.concatenate([np.arange(ns), np.arange(w.S, w.S + keff)]).astype(np.int64))
        for h in range(w.Hkv):
            base = int(off[r] + h * cap[r])
            np.testing.assert_array_equal(host_bf16(ck[base + rows.cuda()]),
                                          np.concatenate([rk[h, :ns], rk[h, w.S:w.S + keff]]))
            np.testing.assert_array_equal(host_bf16(cv[base + rows.cuda()]),
                                          np.concatenate([rv[h, :ns], rv[h, w.S:w.S + keff]]))
        w.oracle_compact[(layer, r)] = (rk, rv, keff)


def _check_fast(w, t, layer, sampled):
    torch.cuda.synchronize()
    assert w.dec.dev_status.item() == 0
    out, lse = w.out[layer].cpu().numpy(), w.lse[layer].cpu().numpy()
    for r in sampled:
        if w.slow_mask[r]:
            continue
        kp, vp, pr = w.host_pages(layer, r)
        rk, rv, keff = w.oracle_compact[(layer, r)]
        o_ref, l_ref = oracle.fast_attn(w.host_q(t, layer, r), rk, rv, keff, kp, vp, pr, w.cur[r], w.S, w.W,
                                        w.Hq, w.Hkv, w.D, 16)
        assert_close(out[r], o_ref, f"fast out r={r} t={t}")
        assert_close(lse[r], l_ref, f"fast lse r={r} t={t}")


def _run_schedule(w, modes, sampled, retention=None, refresh=None):
    """Run len(modes) steps (modes[t][b] = 1 slow / 0 fast) and check every step.
    refresh[t]: layers that take the slow path inside an all-fast step t."""
    w.oracle_compact = {}
    for t, m in enumerate(modes):
        layers_slow = set(refresh[t]) if refresh else set()
        w.cur = w.cur + 1  # the step's token is appended first (fused into the attention kernels)
        w.slow_mask = np.asarray(m, bool)
        if retention is not None:  # k fixed at each slow step from the request's retention ratio
            for r in np.flatnonzero(w.slow_mask):
                w.k_per_req[r] = syn.retention_budget(retention[r], int(w.cur[r]), w.S, w.W)
            w.batch.k_per_req.copy_(torch.as_tensor(w.k_per_req.astype(np.int32)))
        w.k_now = w.k_per_req.copy()
        seq = w.seq_lens()
        if w.slow_mask.all():
            w.dec.slow_step(w.io(t), seq)
        elif not w.slow_mask.any():
            w.dec.fast_step(w.io(t), seq, refresh_layers=layers_slow)
        else:
            w.dec.mixed_step(w.io(t), seq, torch.as_tensor(np.flatnonzero(w.slow_mask).astype(np.int32)).cuda(),
                             torch.as_tensor(np.flatnonzero(~w.slow_mask).astype(np.int32)).cuda())
        w.dec.join()
        step_mask = w.slow_mask
        for layer in range(len(w.layers)):
            w.slow_mask = np.ones_like(step_mask) if layer in layers_slow else step_mask
            _check_slow(w, t, layer, sampled)
            _check_fast(w, t, layer, sampled)
        w.slow_mask = step_mask


def test_qwen3_0_6b_16k_batch16_cycle():
    """16 Q / 8 KV heads, D 128, L 16384, batch 16, 6.25% retention (sink 64, k 704, recent 256),
    two layers: slow step then two fast steps."""
    k = syn.retention_budget(0.0625, 16384, 64, 256)
    w = Workload(2, [16383] * 16, 16, 8, 128, 64, 256, [k] * 16, steps=3, layers=2, heavy_frac=0.02)
    _run_schedule(w, [[1] * 16, [0] * 16, [0] * 16], sampled=[0, 11])


def test_qwen3_0_6b_16k_batch1_full_retention():
    """Batch 1 at 100% retention (every candidate selected), the Table 1 end point; the
    fast step one token later misses only the token that left the recent window."""
    k = 16384 - 64 - 256
    w = Workload(21, [16383], 16, 8, 128, 64, 256, [k], steps=2, layers=1)
    _run_schedule(w, [[1], [0]], sampled=[0])


def test_qwen3_8b_32k_batch32():
    """32 Q / 8 KV heads, D 128, L 32768, batch 32, 6.3% retention (k 1728), slow then fast."""
    k = syn.retention_budget(0.0625, 32768, 64, 256)
    w = Workload(3, [32767] * 32, 32, 8, 128, 64, 256, [k] * 32, steps=2, layers=1, heavy_frac=0.02)
    _run_schedule(w, [[1] * 32, [0] * 32], sampled=[5])


def test_slow_step_stress_64k_zipf_ties():
    """64 Q / 8 KV heads, D 128, L 65536, batch 8, top-4096 per KV head over a Zipf(1.1) logit
    profile with K rows duplicated bit for bit (exact ties through the GPU path)."""
    S, W, k, L = 64, 256, 4096, 65535
    w = Workload(4, [L] * 8, 64, 8, 128, S, W, [k] * 8, steps=1, layers=1)
    n = L + 1 - S - W
    for r in range(8):
        g = syn.rng(4, 100, r)
        lm = syn.zipf_log_mass(g, n)
        beta = lm - lm.mean()
        dup = [(int(S + a), int(S + b)) for a, b in g.integers(0, n, size=(100, 2))]
        syn.device_plant_key_profile_(w.layers[0].k_pool, w.batch.page_table, w.q[0, 0], r, np.arange(S, S + n),
                                      beta, dup)
    _run_schedule(w, [[1] * 8], sampled=[6])
    # the duplicated rows produced exact ties in the GPU scores
    sc = w.layers[0].scores.cpu().numpy()
    assert any(len(np.unique(sc[r, h, S:S + n])) < n for r in range(8) for h in range(8))
    # score values of the sampled request (G = 8 at 64K) against the oracle's fp64 group
    # sums, within the fp32 dot-product bound 2 G D 2^-24 sum |scale q k|
    r, L = 6, int(w.cur[6])
    kp, vp, pr = w.host_pages(0, r)
    q = w.host_q(0, 0, r)
    ref = oracle.group_scores(q, kp, pr, L, S, W, 64, 8, 128, 16, stride=sc.shape[-1])
    masked = np.isneginf(ref[:, :L])
    assert np.array_equal(np.isneginf(sc[r, :, :L]), masked)
    qa = np.abs(syn.bf16_values(q))
    pos = np.arange(L)
    for h in range(8):
        rows = np.abs(syn.bf16_values(kp[pr[pos // 16], h, pos % 16]))
        mag = (rows @ qa[8 * h:8 * h + 8].T).sum(1) / math.sqrt(128)
        bound = 2 * 8 * 128 * 2.0 ** -24 * mag + 1e-30
        ok = ~masked[h]
        err = np.abs(sc[r, h, :L][ok].astype(np.float64) - ref[h, :L][ok])
        assert (err <= bound[ok]).all(), (h, err.max())


@pytest.mark.parametrize("single_launch,ragged", [(True, False), (False, False), (False, True)],
                         ids=["one-launch", "two-launch", "two-launch-ragged-flag"])
def test_ragged_mixed_batch_64_requests(single_launch, ragged):
    """64 requests, lengths log-uniform in [4096, 131072], 32 Q / 8 KV heads, shuffled pages,
    per-request retention from {3, 12.5, 25}%, boundary process p = 0.06 with a forced
    refresh every 32 steps (the first step is slow). The ragged-flag variant plans the
    separate fast and slow launches in length-sized chunks."""
    g = syn.rng(5, 0)
    lens = syn.log_uniform_lengths(g, 64, 4096, 131072) - 1
    ret = g.choice([0.03, 0.125, 0.25], size=64)
    S, W = 64, 256
    k0 = [syn.retention_budget(ret[r], int(lens[r]) + 1, S, W) for r in range(64)]
    k_cap = max(syn.retention_budget(ret[r], int(lens[r]) + 8, S, W) for r in range(64))
    w = Workload(5, lens, 32, 8, 128, S, W, k0, steps=4, layers=1, heavy_frac=0.02, k_cap=k_cap,
                 single_launch_mixed=single_launch, ragged=ragged)
    from sparse_kv_long_sfi_gb300 import SlowFastSchedule
    sched = SlowFastSchedule(64, 32)
    b = syn.boundary_draws(syn.rng(5, 1), 4, 64, 0.3)  # a high rate so that a short run mixes modes
    modes = [sched.next(b[t]) for t in range(4)]
    assert modes[0].all() and 0 < modes[1].sum() < 64
    short, long_ = int(np.argmin(lens)), int(np.argmax(lens))
    slow_then_fast = int(np.flatnonzero(modes[1] == 0)[0])
    _run_schedule(w, modes, sampled=sorted({short, long_, slow_then_fast}), retention=ret)


@pytest.mark.parametrize("single_launch,ragged", [(True, False), (False, True)], ids=["one-launch", "ragged-flag"])
def test_randomized_schedule_small(single_launch, ragged):
    """Twelve decode steps whose kinds are drawn at random (all slow, all fast, fast with
    a refresh layer, mixed) over 6 requests of different lengths, 2 layers, D 64, G 4,
    per-request retention; every request is checked against the oracle after every
    step, so stale compact buffers or mis-ordered side-stream work would show."""
    g = syn.rng(78, 0)  # a draw with every step kind at least twice
    B, steps, S, W = 6, 12, 16, 64
    lens = g.integers(1500, 5000, size=B)
    ret = g.choice([0.05, 0.1, 0.2], size=B)
    k0 = [syn.retention_budget(ret[r], int(lens[r]) + 1, S, W) for r in range(B)]
    k_cap = max(syn.retention_budget(ret[r], int(lens[r]) + steps + 1, S, W) for r in range(B))
    w = Workload(78, lens, 8, 2, 64, S, W, k0, steps=steps, layers=2, heavy_frac=0.02, k_cap=k_cap,
                 single_launch_mixed=single_launch, ragged=ragged)
    modes, refresh = [[1] * B], [()]
    for _ in range(1, steps):
        kind = int(g.integers(0, 4))
        if kind == 3:  # mixed: at least one slow and one fast request
            m = (g.random(B) < 0.4).astype(int)
            m[0], m[1] = 1, 0
            modes.append(list(m))
        else:
            modes.append([1 if kind == 0 else 0] * B)
        refresh.append((1,) if kind == 2 else ())
    assert any(0 < sum(x) < B for x in modes) and any(refresh)
    _run_schedule(w, modes, sampled=list(range(B)), retention=ret, refresh=refresh)


def test_refresh_layer_inside_fast_steps():
    """ASPIRE's intra-draft refresh layer: layer 1 runs the slow path (dense attention,
    scores, Selector, compaction) inside fast steps; the step after uses its fresh
    selection while layer 0 keeps the one of the first slow step."""
    k = syn.retention_budget(0.125, 4096, 64, 256)
    w = Workload(6, [4095] * 4, 16, 8, 128, 64, 256, [k] * 4, steps=4, layers=2, heavy_frac=0.02)
    _run_schedule(w, [[1] * 4, [0] * 4, [0] * 4, [0] * 4], sampled=[0, 3], refresh=[(), (1,), (), (1,)])


def test_speculative_draft_verify_refresh_16k_batch16():
    """Self-speculative decoding over the SFI state ("A Sparse Glimpse of the Whole",
    abstract), Qwen3-0.6B attention at 16K, batch 16, 6.25% retention, two layers:
    slow step, a 4-token draft pass over the sparse state, verification of the same 4
    positions (new K/V, causal dense attention, the recycled statistic), acceptance of a
    seeded number of tokens per request, Selector + compaction from the statistic at the
    accepted lengths, then a fast step on the refreshed state."""
    S, W, T, NL, B = 64, 256, 4, 2, 16
    k = syn.retention_budget(0.0625, 16384, S, W)
    w = Workload(7, [16383] * B, 16, 8, 128, S, W, [k] * B, steps=2 * T + 2, layers=NL, heavy_frac=0.02)
    sampled = [1, 14]
    dev = torch.device("cuda")
    # step 0: slow
    _run_schedule(w, [[1] * B], sampled=sampled)
    oc = dict(w.oracle_compact)
    # draft pass: T tokens over the sparse state
    g = syn.rng(7, 50)
    qd = torch.empty((NL, B, T, 16, 128), dtype=torch.bfloat16, device=dev)
    kd = torch.empty((NL, B, T, 8, 128), dtype=torch.bfloat16, device=dev)
    vd = torch.empty_like(kd)
    for i, t in enumerate((qd, kd, vd)):
        syn.device_normal_bf16_(t, syn.stream_seed(7, 60, i))
    od = torch.full((NL, B, T, 16, 128), float("nan"), device=dev)
    w.cur = w.cur + T
    w.dec.draft_step(w.sfi.StepIO(qd, kd, vd, od), w.seq_lens(), T)
    torch.cuda.synchronize()
    assert w.dec.dev_status.item() == 0
    for layer in range(NL):
        o = od[layer].cpu().numpy()
        for r in sampled:
            kp, vp, pr = w.host_pages(layer, r)
            rk, rv, keff = oc[(layer, r)]
            o_ref, _ = oracle.fast_multi_attn(host_bf16(qd[layer, r]), rk, rv, keff, kp, vp, pr, w.cur[r], T, S, W,
                                              16, 8, 128, 16)
            assert_close(o[r], o_ref, f"draft out layer={layer} r={r}")
    # verification of the same T positions with the full model's K/V and queries
    qv, kv_, vv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    for i, t in enumerate((qv, kv_, vv)):
        syn.device_normal_bf16_(t, syn.stream_seed(7, 70, i))
    ov = torch.full_like(od, float("nan"))
    lv = torch.full((NL, B, T, 16), float("nan"), device=dev)
    for L_ in w.layers:
        L_.scores.fill_(float("nan"))
    w.dec.verify_step(w.sfi.StepIO(qv, kv_, vv, ov, lv), w.seq_lens(), T)
    torch.cuda.synchronize()
    assert w.dec.dev_status.item() == 0
    for layer in range(NL):
        o, l = ov[layer].cpu().numpy(), lv[layer].cpu().numpy()
        sc = w.layers[layer].scores.cpu().numpy()
        for r in sampled:
            kp, vp, pr = w.host_pages(layer, r)
            q = host_bf16(qv[layer, r])
            o_ref, l_ref = oracle.verify_attn(q, kp, vp, pr, w.cur[r], T, 16, 8, 128, 16)
            assert_close(o[r], o_ref, f"verify out layer={layer} r={r}")
            assert_close(l[r], l_ref, f"verify lse layer={layer} r={r}")
            L = int(w.cur[r])
            ref = oracle.verify_scores(q, kp, pr, L, T, S, W, 16, 8, 128, 16, stride=sc.shape[-1])
            masked = np.isneginf(ref[:, :L])
            assert np.array_equal(np.isneginf(sc[r, :, :L]), masked)
            qa = np.abs(syn.bf16_values(q))
            for h in range(8):
                rows = np.abs(syn.bf16_values(kp[pr[np.arange(L) // 16], h, np.arange(L) % 16]))
                mag = (rows @ qa[:, 2 * h:2 * h + 2].reshape(-1, 128).T).sum(1) / math.sqrt(128)
                bound = 2 * T * 2 * 128 * 2.0 ** -24 * mag + 1e-30
                ok = ~masked[h]
                err = np.abs(sc[r, h, :L][ok].astype(np.float64) - ref[h, :L][ok])
                assert (err <= bound[ok]).all(), (layer, r, h, err.max())
    # acceptance: a seeded number of the T tokens per request, then the selection refresh
    accepted = syn.rng(7, 80).integers(0, T + 1, size=B)
    w.cur = w.cur - T + accepted
    w.dec.refresh_selection(w.seq_lens())
    w.dec.join()
    torch.cuda.synchronize()
    assert w.dec.dev_status.item() == 0
    w.oracle_compact = {}
    for layer in range(NL):
        Lb = w.layers[layer]
        sc = Lb.scores.cpu().numpy()
        idx, count = Lb.idx.cpu().numpy(), Lb.compact.count.cpu().numpy()
        cap = Lb.compact.capacity.cpu().numpy()
        for r in range(B):
            for h in range(8):
                want = oracle.select_topk(sc[r, h], w.cur[r], S, W, k)
                assert count[r] == len(want)
                np.testing.assert_array_equal(idx[r, h, :len(want)], want, err_msg=f"layer={layer} r={r} kv={h}")
        for r in sampled:
            kp, vp, pr = w.host_pages(layer, r)
            rk, rv = oracle.compact(kp, vp, pr, w.cur[r], S, idx[r], count[r], 8, 128, 16, cap[r])
            w.oracle_compact[(layer, r)] = (rk, rv, count[r])
    # a fast step on the refreshed state
    w.cur = w.cur + 1
    w.slow_mask = np.zeros(B, bool)
    w.dec.fast_step(w.io(1), w.seq_lens())
    w.dec.join()
    for layer in range(NL):
        _check_fast(w, 1, layer, sampled)


def test_schedule_without_join_between_steps():
    """Nine decode steps (slow, fast, fast with a refresh layer, mixed, ...) issued back to
    back with no join between them, so a step's fast attention of layer i may be queued
    while layer i's Selector and compaction from the previous step are still running on
    the side stream: only the per-layer events order them (Figure 3 (A) of the SFI
    paper). Each step's outputs, scores and selections are snapshotted on the stream
    that wrote them; after one final join every step of every request is checked
    against the oracle (attention within tolerance, selection bit-exact)."""
    B, NL, S, W = 6, 2, 16, 64
    g = syn.rng(91, 0)
    lens = g.integers(2000, 5000, size=B)
    k = [int(x) for x in g.integers(100, 400, size=B)]
    steps = 9
    w = Workload(91, lens, 16, 8, 128, S, W, k, steps=steps, layers=NL, heavy_frac=0.02, k_cap=max(k))
    # per step: request modes (1 slow / 0 fast) and refresh layers inside an all-fast step
    modes = [[1] * B, [0] * B, [0] * B, [1, 0, 0, 1, 0, 0], [0] * B, [1] * B, [0] * B, [0, 1, 0, 0, 0, 1], [0] * B]
    refresh = [(), (), (1,), (), (0,), (), (), (), ()]
    dec = w.dec
    keep = []  # device tensors the side stream may still read
    snaps = []
    cur = w.cur.copy()
    for t in range(steps):
        cur = cur + 1
        seq = torch.as_tensor(cur.astype(np.int32)).cuda()
        keep.append(seq)
        m = np.asarray(modes[t], bool)
        if m.all():
            dec.slow_step(w.io(t), seq)
        elif not m.any():
            dec.fast_step(w.io(t), seq, refresh_layers=refresh[t])
        else:
            sid = torch.as_tensor(np.flatnonzero(m).astype(np.int32)).cuda()
            fid = torch.as_tensor(np.flatnonzero(~m).astype(np.int32)).cuda()
            keep += [sid, fid]
            dec.mixed_step(w.io(t), seq, sid, fid)
        snap = {"cur": cur.copy()}
        with torch.cuda.stream(dec.main):  # written by the main stream
            snap["out"] = w.out.clone()
            snap["lse"] = w.lse.clone()
            snap["scores"] = [L.scores.clone() for L in w.layers]
        with torch.cuda.stream(dec.aux):  # written by the side stream (no join)
            snap["idx"] = [L.idx.clone() for L in w.layers]
            snap["count"] = [L.compact.count.clone() for L in w.layers]
        snaps.append(snap)
    dec.join()
    torch.cuda.synchronize()
    assert dec.dev_status.item() == 0
    oracle_state = {}  # (layer, request) -> oracle compact rows of the latest slow step
    n_checked = 0
    for t in range(steps):
        sn = snaps[t]
        w.cur = sn["cur"]
        out, lse = sn["out"].cpu().numpy(), sn["lse"].cpu().numpy()
        for layer in range(NL):
            slow = np.asarray(modes[t], bool) | (layer in refresh[t])
            sc = sn["scores"][layer].cpu().numpy()
            idx, count = sn["idx"][layer].cpu().numpy(), sn["count"][layer].cpu().numpy()
            cap = w.layers[layer].compact.capacity.cpu().numpy()
            for r in range(B):
                kp, vp, pr = w.host_pages(layer, r)
                q = w.host_q(t, layer, r)
                L = int(w.cur[r])
                if slow[r]:
                    o_ref, l_ref = oracle.dense_attn(q, kp, vp, pr, L, w.Hq, w.Hkv, w.D, 16)
                    for h in range(w.Hkv):
                        want = oracle.select_topk(sc[r, h], L, S, W, k[r])
                        assert count[r] == len(want), (t, layer, r)
                        np.testing.assert_array_equal(idx[r, h, :len(want)], want,
                                                      err_msg=f"selection t={t} layer={layer} r={r} kv={h}")
                    rk, rv = oracle.compact(kp, vp, pr, L, S, idx[r], count[r], w.Hkv, w.D, 16, cap[r])
                    oracle_state[(layer, r)] = (rk, rv, count[r])
                else:
                    rk, rv, keff = oracle_state[(layer, r)]
                    o_ref, l_ref = oracle.fast_attn(q, rk, rv, keff, kp, vp, pr, L, S, W, w.Hq, w.Hkv, w.D, 16)
                assert_close(out[layer, r], o_ref, f"out t={t} layer={layer} r={r} slow={bool(slow[r])}")
                assert_close(lse[layer, r], l_ref, f"lse t={t} layer={layer} r={r}")
                n_checked += 1
    assert n_checked == steps * NL * B
