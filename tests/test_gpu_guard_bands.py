"""Guard bands: every buffer the kernels write is an interior view of a larger allocation
whose margins hold a sentinel, and the regions the C ABI leaves unwritten (score entries
j >= L, Selector indices past k_eff, compact rows past min(S, L) and S + count) start
with it too. After the slow step, the Selector, the compaction, the fast step (with the
fused append) and a T-token draft, every sentinel must still be there, bit for bit, for
the cluster merges (per-warp and per-CTA pushes, and the pull), the workspace merge and
a single split. Written values are checked against the oracle elsewhere; here the
question is only where the kernels write."""
import numpy as np
import pytest
import torch

import sfi_synth as syn
from tests.gpu_harness import Problem, dev_bf16, dev_i32

pytestmark = pytest.mark.gpu

PAD = 1024  # guard elements on each side of every buffer (keeps every view 16-byte aligned)
# sentinels no kernel output can equal (attention outputs and KV rows are O(1), indices >= 0)
F32, BF16, I32 = -7.0e30, -1.0e38, -7
BF16_STORED = float(torch.tensor(BF16, dtype=torch.bfloat16).float())


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from sparse_kv_long_sfi_gb300 import build
    build.build()


def _sfi():
    import sparse_kv_long_sfi_gb300 as sfi
    return sfi


class Guarded:
    """An interior view `v` of shape `shape` inside a sentinel-filled allocation."""

    def __init__(self, shape, dtype, fill):
        n = int(np.prod(shape))
        self.fill = fill
        self.full = torch.full((n + 2 * PAD,), fill, dtype=dtype, device="cuda")
        self.v = self.full[PAD:PAD + n].view(*shape)

    def margins_intact(self):
        ref = torch.full((PAD,), self.fill, dtype=self.full.dtype, device="cuda")
        return torch.equal(self.full[:PAD], ref) and torch.equal(self.full[-PAD:], ref)


def _workspace(nbytes):
    """A zero-filled workspace (as the ABI requires) between 0xA5 guard bands."""
    g = Guarded((max(256, nbytes),), torch.uint8, 0xA5)
    g.v.zero_()
    return g


def _run(Hq, Hkv, splits, T):
    sfi = _sfi()
    S, W, D = 4, 32, 128
    lens = [3, 17, 300, 1500]
    k_per_req = [0, 0, 100, 700]
    k_cap = 768
    prob = Problem(seed=900 + Hq + splits, lens=lens, Hq=Hq, Hkv=Hkv, D=D, S=S, W=W, extra_tokens=16).to_device()
    B = prob.B
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    checks = []

    # slow step: dense attention and the masked scores
    stride = max(lens) + 40
    out = Guarded((B, Hq, D), torch.float32, F32)
    lse = Guarded((B, Hq), torch.float32, F32)
    scores = Guarded((B, Hkv, stride), torch.float32, F32)
    max_l = max(lens) + 16
    ws = _workspace(sfi.sfi_workspace_size(prob.shape, B, max_l, splits))
    sfi.sfi_slow_dense_attn_with_scores(prob.shape, prob.d_kv, S, W, prob.d_q, out.v, lse.v, scores.v,
                                        max_tokens=max_l, num_splits=splits, workspace=ws.v, dev_status=st)
    checks += [("slow out", out), ("slow lse", lse), ("scores", scores), ("slow workspace", ws)]

    # Selector and compaction
    idx = Guarded((B, Hkv, k_cap), torch.int32, I32)
    count = Guarded((B,), torch.int32, I32)
    sfi.sfi_select_topk(scores.v, Hkv, prob.d_kv.seq_lens, S, W, dev_i32(k_per_req), idx.v, count.v, dev_status=st)
    off, cap = sfi.compact_layout(prob.shape, S, k_per_req)
    rows = int((off[-1] + Hkv * cap[-1]).item())
    ck = Guarded((rows, D), torch.bfloat16, BF16)
    cv = Guarded((rows, D), torch.bfloat16, BF16)
    comp = sfi.CompactKV(ck.v, cv.v, off, cap, count.v)
    sfi.sfi_compact_gather(prob.shape, prob.d_kv, idx.v, count.v, S, comp, dev_status=st)
    checks += [("idx", idx), ("count", count), ("compact k", ck), ("compact v", cv)]

    # fast step with the current token appended in the same launch
    g = syn.rng(907, Hq + splits)
    lens1 = [L + 1 for L in lens]
    prob.set_lens(lens1)
    kn, vn = dev_bf16(syn.normal_bf16(g, (B, Hkv, D))), dev_bf16(syn.normal_bf16(g, (B, Hkv, D)))
    out2 = Guarded((B, Hq, D), torch.float32, F32)
    lse2 = Guarded((B, Hq), torch.float32, F32)
    mt = max(S + k_cap + W + 32, 1600)  # a bound large enough that 12 splits are not clamped
    ws2 = _workspace(sfi.sfi_workspace_size(prob.shape, B, mt, splits))
    sfi.sfi_fast_decode_attn(prob.shape, prob.d_kv, comp, S, W, prob.d_q, out2.v, lse2.v, k_new=kn, v_new=vn,
                             max_tokens=mt, num_splits=splits, workspace=ws2.v, dev_status=st)
    checks += [("fast out", out2), ("fast lse", lse2), ("fast workspace", ws2)]

    # T-token draft over the same state (its own query tokens and append)
    lensT = [L + T for L in lens1]
    prob.set_lens(lensT)
    qT = dev_bf16(syn.normal_bf16(g, (B, T, Hq, D)))
    knT, vnT = dev_bf16(syn.normal_bf16(g, (B, T, Hkv, D))), dev_bf16(syn.normal_bf16(g, (B, T, Hkv, D)))
    out3 = Guarded((B, T, Hq, D), torch.float32, F32)
    lse3 = Guarded((B, T, Hq), torch.float32, F32)
    mtT = max(S + k_cap + W + T + 32, 1600)
    ws3 = _workspace(sfi.sfi_multi_workspace_size(prob.shape, B, T, mtT, splits))
    draft_ids = [1, 2, 3]  # request 0 is left out: its outputs must keep their sentinel
    sfi.sfi_sparse_draft_attn(prob.shape, prob.d_kv, comp, S, W, qT, T, out3.v, lse3.v,
                              req_ids=dev_i32(draft_ids), max_tokens=mtT, num_splits=splits, workspace=ws3.v,
                              dev_status=st, k_new=knT, v_new=vnT)
    checks += [("draft out", out3), ("draft lse", lse3), ("draft workspace", ws3)]
    torch.cuda.synchronize()
    assert st.item() == 0

    for name, gbuf in checks:
        assert gbuf.margins_intact(), f"{name}: a write landed in the guard band"

    # regions the ABI leaves unwritten
    sc = scores.v.cpu().numpy()
    for r, L in enumerate(lens):
        assert (sc[r, :, L:] == np.float32(F32)).all(), f"scores past L written, r={r}"
        assert (sc[r, :, :L] != np.float32(F32)).all(), f"scores below L not written, r={r}"
    ix, cnt = idx.v.cpu().numpy(), count.v.cpu().numpy()
    c = ck.v.float().cpu().numpy()
    offs, caps = off.cpu().numpy(), cap.cpu().numpy()
    for r, L in enumerate(lens):
        keff = int(cnt[r])
        assert 0 <= keff <= k_per_req[r]
        assert (ix[r, :, keff:] == I32).all(), f"Selector indices past k_eff written, r={r}"
        for kvh in range(Hkv):
            base = int(offs[r]) + kvh * int(caps[r])
            blk = c[base:base + int(caps[r])]
            written = np.zeros(int(caps[r]), bool)
            written[:min(S, L)] = True
            written[S:S + keff] = True
            assert (blk[~written] == BF16_STORED).all(), f"compact rows outside the sink and selection written, r={r}"
            assert (blk[written] != BF16_STORED).all(), f"compact rows not written, r={r}"
    # outputs of requests left out of the draft keep their sentinel
    o3 = out3.v.cpu().numpy()
    for r in range(B):
        if r not in draft_ids:
            assert (o3[r] == np.float32(F32)).all()
        else:
            assert (o3[r] != np.float32(F32)).all()


@pytest.mark.parametrize("Hq,Hkv,splits", [
    (16, 8, 1),   # one split
    (16, 8, 3),   # cluster: per-warp partials from the other CTAs
    (64, 8, 3),   # cluster: one partial per CTA (G = 8)
    (64, 8, 6),   # cluster: rank 0 pulls the partials
    (16, 8, 12),  # workspace merge
    (16, 8, 0),   # automatic plans
])
def test_kernels_write_nothing_outside_their_buffers(Hq, Hkv, splits):
    _run(Hq, Hkv, splits, T=2 if Hq // Hkv == 8 else 4)
