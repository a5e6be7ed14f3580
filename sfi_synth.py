"""Seeded synthetic inputs for the SFI decode-attention path.

This module is the only code shared by the CUDA path's tests and benchmark and by
the CPU oracle's callers. It holds input recipes only (random numbers, bf16
rounding of the draws, page tables, planted structure) and none of the method's
arithmetic: no attention, no scores, no selection, no compaction.

Every draw comes from numpy's PCG64 seeded by a SeedSequence over
(base seed, tag, *keys), so each tensor of each workload has its own stream.
Device-side variants (for workloads too large to draw on the host) use a seeded
torch.Generator on the target device.

Recipes (Slow-Fast Inference, Xie et al. 2026: Table 1 fixes bf16 KV, KV length
16K and batch 16 for the kernel-level measurement; Figure 3 fixes the paged KV and
the compact buffer; the shapes are those of Qwen3 attention layers):
  * Q, K, V are N(0, 1) drawn in fp64, rounded to fp32, then to bf16 with
    round-to-nearest-even.
  * Pages hold P tokens of one KV head; a request's pages are a seeded random
    subset of the pool in random order (a shuffled page table).
  * Heavy hitters: K rows at chosen positions get ``+ beta * u`` where u is a unit
    vector (the direction of the group-summed query), which raises the
    group-summed logit of those positions by beta of its standard deviations.
  * Selector score profiles: Zipf(1.1) mass over a seeded permutation of the
    candidates, score = fp32(ln mass), with exact ties planted.
  * Ragged batches: lengths log-uniform in [lo, hi]; per-request retention drawn
    from a small set; boundary events Bernoulli(p) per request and step.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

BASE_SEED = 20260312


def rng(*keys: int) -> np.random.Generator:
    """Independent seeded stream for (BASE_SEED, *keys)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([BASE_SEED, *[int(k) for k in keys]])))


def stream_seed(*keys: int) -> int:
    """A 63-bit seed derived from (BASE_SEED, *keys), for torch generators."""
    ss = np.random.SeedSequence([BASE_SEED, *[int(k) for k in keys]])
    return int(ss.generate_state(1, dtype=np.uint64)[0] & np.uint64((1 << 63) - 1))


# ---------------------------------------------------------------------------
# bf16 materialisation of the draws
# ---------------------------------------------------------------------------
def bf16_bits(x) -> np.ndarray:
    """Round values to bf16 bit patterns (uint16): fp64 -> fp32 (RNE) -> bf16 (RNE).

    Non-finite inputs are not produced by the recipes and are not handled specially.
    """
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_values(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64 (used to plant structure)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def normal_bf16(g: np.random.Generator, shape) -> np.ndarray:
    return bf16_bits(g.standard_normal(shape))


# ---------------------------------------------------------------------------
# Paged KV
# ---------------------------------------------------------------------------
@dataclass
class PagedKV:
    """Host copy of a paged bf16 KV cache.

    k_pool, v_pool: uint16 [num_pages][Hkv][P][D] (bf16 bits)
    page_table:     int32  [B][max_pages]   (-1 = unused slot)
    seq_lens:       int32  [B]
    """
    k_pool: np.ndarray
    v_pool: np.ndarray
    page_table: np.ndarray
    seq_lens: np.ndarray
    page_size: int

    @property
    def num_pages(self) -> int:
        return self.k_pool.shape[0]


def make_page_table(g: np.random.Generator, capacity_tokens, page_size: int, shuffle: bool = True,
                    spare_pages: int = 0):
    """Assign pages for requests able to hold capacity_tokens[r] tokens.

    Returns (page_table int32 [B][max_pages], num_pages). With shuffle, the pages of
    all requests are a seeded permutation of the pool (pages of one request are
    scattered and out of order); unused table slots are -1.
    """
    caps = [int(c) for c in capacity_tokens]
    npg = [(c + page_size - 1) // page_size for c in caps]
    total = sum(npg) + spare_pages
    max_pages = max(1, max(npg) if npg else 1)
    order = g.permutation(total) if shuffle else np.arange(total)
    table = np.full((len(caps), max_pages), -1, dtype=np.int32)
    at = 0
    for r, n in enumerate(npg):
        table[r, :n] = order[at:at + n]
        at += n
    return table, total


def make_paged_kv(g: np.random.Generator, seq_lens, num_kv_heads: int, head_dim: int, page_size: int = 16,
                  capacity_tokens=None, shuffle: bool = True) -> PagedKV:
    """Random N(0,1) bf16 K/V in a shuffled paged pool.

    capacity_tokens (default seq_lens) sizes each request's page list, so that later
    appends have room.
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    cap = seq_lens if capacity_tokens is None else np.asarray(capacity_tokens)
    table, num_pages = make_page_table(g, cap, page_size, shuffle)
    shape = (num_pages, num_kv_heads, page_size, head_dim)
    k_pool = normal_bf16(g, shape)
    v_pool = normal_bf16(g, shape)
    return PagedKV(k_pool, v_pool, table, seq_lens.copy(), page_size)


def pool_slot(kv: PagedKV, r: int, pos: int):
    """(page, slot) holding position pos of request r."""
    return int(kv.page_table[r, pos // kv.page_size]), pos % kv.page_size


def plant_key_bias(kv: PagedKV, r: int, kv_head: int, positions, direction: np.ndarray, beta) -> None:
    """K rows at positions += beta * direction (rounded back to bf16), in place.

    beta may be a scalar or one value per position.
    """
    d = np.asarray(direction, dtype=np.float64)
    betas = np.broadcast_to(np.asarray(beta, dtype=np.float64), (len(positions),))
    for pos, b in zip(positions, betas):
        page, slot = pool_slot(kv, r, int(pos))
        row = bf16_values(kv.k_pool[page, kv_head, slot]) + b * d
        kv.k_pool[page, kv_head, slot] = bf16_bits(row)


def copy_key_row(kv: PagedKV, r: int, kv_head: int, src_pos: int, dst_pos: int) -> None:
    """Duplicate a K row bit for bit (plants exact logit ties)."""
    sp, ss = pool_slot(kv, r, src_pos)
    dp, ds = pool_slot(kv, r, dst_pos)
    kv.k_pool[dp, kv_head, ds] = kv.k_pool[sp, kv_head, ss]


def group_direction(q_bits: np.ndarray, kv_head: int, group: int) -> np.ndarray:
    """Unit vector along the sum of the query rows of one GQA group (kv_head*G .. +G)."""
    qs = bf16_values(q_bits[kv_head * group:(kv_head + 1) * group]).sum(axis=0)
    n = np.linalg.norm(qs)
    return qs / n if n > 0 else np.eye(q_bits.shape[-1])[0]


def group_sigma(q_bits: np.ndarray, kv_head: int, group: int, head_dim: int) -> float:
    """Standard deviation, over N(0,1) keys, of the group-summed scaled logit: |sum_g q_g| / sqrt(D)."""
    qs = bf16_values(q_bits[kv_head * group:(kv_head + 1) * group]).sum(axis=0)
    return float(np.linalg.norm(qs)) / math.sqrt(head_dim)


# ---------------------------------------------------------------------------
# Selector inputs
# ---------------------------------------------------------------------------
def zipf_log_mass(g: np.random.Generator, n: int, s: float = 1.1) -> np.ndarray:
    """ln of a Zipf(s) mass profile (mass ~ rank^-s) over a seeded permutation of n slots."""
    ranks = g.permutation(n) + 1
    return -s * np.log(ranks.astype(np.float64))


def zipf_scores_with_ties(g: np.random.Generator, n: int, k: int, s: float = 1.1, band: int = 16,
                          groups: int = 32) -> np.ndarray:
    """fp32 selector scores over n candidates: fp32(ln Zipf mass) with exact ties.

    Ranks k-band .. k+band (1-based ranks around the k-th) all get the k-th rank's
    exact fp32 value; `groups` random groups of 2..8 slots are set equal to one of
    their members.
    """
    ranks = g.permutation(n) + 1
    vals = (-s * np.log(ranks.astype(np.float64))).astype(np.float32)
    if 0 < k <= n:
        kth = np.float32(-s * math.log(k))
        lo, hi = max(1, k - band), min(n, k + band)
        vals[(ranks >= lo) & (ranks <= hi)] = kth
    for _ in range(groups):
        m = int(g.integers(2, 9))
        members = g.choice(n, size=min(m, n), replace=False)
        vals[members] = vals[members[0]]
    return vals


# ---------------------------------------------------------------------------
# Ragged batches and schedules
# ---------------------------------------------------------------------------
def log_uniform_lengths(g: np.random.Generator, n: int, lo: int, hi: int) -> np.ndarray:
    return np.floor(np.exp(g.uniform(math.log(lo), math.log(hi), size=n))).astype(np.int32).clip(lo, hi)


def boundary_draws(g: np.random.Generator, steps: int, batch: int, p: float) -> np.ndarray:
    """uint8 [steps][batch]: 1 where a boundary event fires (Bernoulli(p))."""
    return (g.random((steps, batch)) < p).astype(np.uint8)


def retention_budget(retention: float, length: int, sink: int, recent: int) -> int:
    """Selected-token count k for a retention ratio: max(0, round(r * L) - sink - recent)."""
    return max(0, int(round(retention * length)) - sink - recent)


# ---------------------------------------------------------------------------
# Device-side draws (large workloads), torch only imported here
# ---------------------------------------------------------------------------
def device_normal_bf16_(t, seed: int):
    """Fill a CUDA bf16 tensor in place with N(0,1) draws (fp32 draw, RNE to bf16) from a seeded generator."""
    import torch
    gen = torch.Generator(device=t.device)
    gen.manual_seed(int(seed))
    flat = t.view(-1)
    chunk = 1 << 28
    for s in range(0, flat.numel(), chunk):
        e = min(flat.numel(), s + chunk)
        flat[s:e].copy_(torch.randn(e - s, generator=gen, device=t.device, dtype=torch.float32))
    return t


def device_plant_heavy_hitters_(k_pool, page_table, q, seq_lens, sink: int, recent: int, frac: float, beta: float,
                                seed: int):
    """Heavy-hitter keys on the device: for each (request, KV head), a seeded 'frac'
    share of the candidate positions [sink, L - recent) gets K += beta * u, u the unit
    vector along the group-summed query q (bf16 [B][Hq][D]). In place on k_pool
    (bf16 [pages][Hkv][P][D]); page_table int32 [B][max_pages] and seq_lens are
    device tensors."""
    import torch
    B, Hq, D = q.shape
    Hkv, P = k_pool.shape[1], k_pool.shape[2]
    G = Hq // Hkv
    gen = torch.Generator(device=q.device)
    gen.manual_seed(int(seed))
    qbar = q.float().view(B, Hkv, G, D).sum(2)
    u = qbar / qbar.norm(dim=-1, keepdim=True).clamp_min(1e-12)          # [B][Hkv][D]
    flat = k_pool.view(-1, D)
    lens = seq_lens.cpu().tolist()
    for r in range(B):
        n = lens[r] - sink - recent
        m = int(round(frac * n))
        if m <= 0:
            continue
        pos = sink + torch.stack([torch.randperm(n, generator=gen, device=q.device)[:m] for _ in range(Hkv)])
        pages = page_table[r].long()[pos // P]                              # [Hkv][m]
        kvh = torch.arange(Hkv, device=q.device).view(Hkv, 1)
        rows = (pages * Hkv + kvh) * P + pos % P
        vals = flat[rows.view(-1)].float().view(Hkv, m, D) + beta * u[r].view(Hkv, 1, D)
        flat[rows.view(-1)] = vals.view(-1, D).to(k_pool.dtype)
    return k_pool


def device_plant_key_profile_(k_pool, page_table, q, r: int, positions, betas, dup_pairs=()):
    """K rows of request r at `positions` (host ints) get K += beta_j * u (u along the
    group-summed query of each KV head), then K rows are copied bit for bit for each
    (src, dst) in dup_pairs (exact logit ties). In place on the device pool."""
    import torch
    B, Hq, D = q.shape
    Hkv, P = k_pool.shape[1], k_pool.shape[2]
    G = Hq // Hkv
    qbar = q[r].float().view(Hkv, G, D).sum(1)
    u = qbar / qbar.norm(dim=-1, keepdim=True).clamp_min(1e-12)            # [Hkv][D]
    flat = k_pool.view(-1, D)
    pos = torch.as_tensor(np.asarray(positions, np.int64), device=q.device)
    beta = torch.as_tensor(np.asarray(betas, np.float32), device=q.device)
    pages = page_table[r].long()[pos // P]
    kvh = torch.arange(Hkv, device=q.device).view(Hkv, 1)
    rows = ((pages.view(1, -1) * Hkv + kvh) * P + (pos % P).view(1, -1)).view(-1)
    vals = flat[rows].float().view(Hkv, -1, D) + beta.view(1, -1, 1) * u.view(Hkv, 1, D)
    flat[rows] = vals.view(-1, D).to(k_pool.dtype)
    for src, dst in dup_pairs:
        for h in range(Hkv):
            sr = (int(page_table[r, src // P]) * Hkv + h) * P + src % P
            dr = (int(page_table[r, dst // P]) * Hkv + h) * P + dst % P
            flat[dr] = flat[sr]
    return k_pool
