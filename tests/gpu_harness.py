"""Helpers for the GPU parity tests: seeded problems, host<->device copies, and the
oracle run request by request. Inputs come from sfi_synth only; expected values
come from the oracle only."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import sfi_synth as syn

# Attention tolerance of the parity bar (allclose form): |gpu - oracle| <= ATOL + RTOL * |oracle|.
ATOL, RTOL = 2e-3, 1e-2


def dev_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).cuda()


def host_bf16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dev_i32(a) -> torch.Tensor:
    return torch.as_tensor(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def dev_i64(a) -> torch.Tensor:
    return torch.as_tensor(np.ascontiguousarray(a, dtype=np.int64)).cuda()


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str, atol=ATOL, rtol=RTOL):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.isfinite(gpu).all(), f"{what}: non-finite GPU values"
    err = np.abs(gpu - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {err.size} outside tolerance; worst at {i}: "
                             f"gpu {gpu[i]!r} oracle {ref[i]!r} (max abs err {err.max():.3e})")


class Problem:
    """A seeded batch: host paged KV, queries, and the decode geometry."""

    def __init__(self, seed, lens, Hq, Hkv, D, S, W, extra_tokens=0, heavy_frac=0.0, heavy_beta=3.0,
                 shuffle=True):
        self.Hq, self.Hkv, self.D, self.P, self.S, self.W = Hq, Hkv, D, 16, S, W
        self.G = Hq // Hkv
        g = syn.rng(100, seed)
        self.lens = np.asarray(lens, np.int32)
        self.B = len(lens)
        self.kv = syn.make_paged_kv(g, self.lens, Hkv, D, 16, capacity_tokens=self.lens + extra_tokens,
                                    shuffle=shuffle)
        self.q = syn.normal_bf16(g, (self.B, Hq, D))
        if heavy_frac > 0:
            for r in range(self.B):
                L = int(self.lens[r])
                nC = max(0, L - S - W)
                n_hot = int(round(heavy_frac * nC))
                if n_hot == 0:
                    continue
                for kvh in range(Hkv):
                    pos = S + g.choice(nC, size=n_hot, replace=False)
                    u = syn.group_direction(self.q[r], kvh, self.G)
                    # K += beta * u raises the group-summed scaled logit, whose std over
                    # N(0, 1) keys is |qbar| / sqrt(D), by exactly beta standard deviations.
                    step = heavy_beta
                    syn.plant_key_bias(self.kv, r, kvh, pos, u, step)
        self.shape = None

    # ---- device views ----
    def to_device(self):
        import sparse_kv_long_sfi_gb300 as sfi
        self.shape = sfi.AttnShape(self.Hq, self.Hkv, self.D)
        self.d_kv = sfi.PagedKV(dev_bf16(self.kv.k_pool), dev_bf16(self.kv.v_pool), dev_i32(self.kv.page_table),
                                dev_i32(self.kv.seq_lens))
        self.d_q = dev_bf16(self.q)
        return self

    def set_lens(self, lens):
        self.lens = np.asarray(lens, np.int32)
        self.kv.seq_lens = self.lens.copy()
        if self.shape is not None:
            self.d_kv.seq_lens.copy_(torch.as_tensor(self.lens))

    # ---- oracle, request by request ----
    def oracle_dense(self, r):
        return oracle.dense_attn(self.q[r], self.kv.k_pool, self.kv.v_pool, self.kv.page_table[r], self.lens[r],
                                 self.Hq, self.Hkv, self.D, self.P)

    def oracle_scores(self, r, stride):
        return oracle.group_scores(self.q[r], self.kv.k_pool, self.kv.page_table[r], self.lens[r], self.S, self.W,
                                   self.Hq, self.Hkv, self.D, self.P, stride=stride)

    def score_bound(self, r, stride):
        """fp32 dot-product error bound per score: 2*G*D*2^-24 * sum_{g,d} |scale q k| (+ tiny slack)."""
        L = int(self.lens[r])
        scale = 1.0 / math.sqrt(self.D)
        out = np.zeros((self.Hkv, stride))
        qa = np.abs(syn.bf16_values(self.q[r]))
        for kvh in range(self.Hkv):
            rows = np.stack([np.abs(syn.bf16_values(
                self.kv.k_pool[self.kv.page_table[r, j // 16], kvh, j % 16])) for j in range(L)])
            mag = (rows @ qa[kvh * self.G:(kvh + 1) * self.G].T).sum(1) * scale
            out[kvh, :L] = 2 * self.G * self.D * 2.0 ** -24 * mag + 1e-30
        return out


def run_oracle_selection(prob: Problem, scores_host: np.ndarray, k_per_req, k_cap):
    """Oracle Selector on given fp32 score rows -> (idx [B][Hkv][k_cap] with -1 fill, count [B])."""
    B, Hkv = prob.B, prob.Hkv
    idx = np.full((B, Hkv, max(k_cap, 1)), -1, np.int32)
    count = np.zeros(B, np.int32)
    for r in range(B):
        for kvh in range(Hkv):
            sel = oracle.select_topk(scores_host[r, kvh], prob.lens[r], prob.S, prob.W, k_per_req[r])
            idx[r, kvh, :len(sel)] = sel
            count[r] = len(sel)
    return idx, count


def oracle_compact_request(prob: Problem, r, idx_r, keff, cap):
    return oracle.compact(prob.kv.k_pool, prob.kv.v_pool, prob.kv.page_table[r], prob.lens[r], prob.S,
                          np.where(idx_r < 0, 0, idx_r), keff, prob.Hkv, prob.D, prob.P, cap)
