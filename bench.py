#!/usr/bin/env python3
"""Benchmark of the SFI decode-attention path on one GB300 (replicas on N GPUs).

Workload (the paper's Table 1 setting with Qwen3-0.6B attention shapes): 16 query
heads / 8 KV heads, head_dim 128, 28 layers, bf16 paged KV (page 16), KV length
16384, batch 16, sink 64 + selected + recent 256. Seeded N(0,1) Q/K/V on the device
with heavy-hitter keys on 2% of the candidates.

One bench step = one SFI refresh cycle of 16 decode steps over all 28 layers: a slow
step (append, dense attention + masked group-summed scores on the main stream,
Selector + compaction on the aux stream overlapped with the next layers), then 15
fast steps (append, sparse attention over sink + selected + recent) at 6.25%
retention (k = 704). The whole cycle is one CUDA graph replay. `value` is the
decode-attention time per decode step (cycle time / 16, all 28 layers).

Also reported: the end-to-end time through the public API with host buffers (per
decode step: H2D of q/k/v, D2H of the outputs), the roofline of the dominant kernel,
the CPU oracle timed on a bounded sample (the reference arm: --impl reference), and
these sections (--sections):
  overlap          the side stream's overlap: the cycle with the Selector and
                   compaction on the main stream against the two-stream cycle, the
                   side work alone, and the first fast step's penalty against the
                   side work's own HBM time;
  retention        Table 1's retention sweep against the dense decode kernel;
  speculative      verification and draft passes of T = 1, 2, 4, 8 tokens;
  batch1           the same cycle and retention sweep at batch 1;
  qwen3_8b         the Qwen3-8B-shaped workload as a full cycle: 36 layers, batch 32,
                   KV 32K, 6.25% retention, one slow step every 16;
  other            per-launch times of the 64-query-head, KV 64K, top-4096 slow step;
  ragged           one step of the ragged 64-request batch, one vs two launches;
  ragged_schedule  the ragged batch under its seeded boundary process for 64 steps.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attn µs/step & achieved HBM GB/s vs ~8 TB/s; sparse/dense speedup at 16K"
UNIT = "us/step"
WL = dict(workload="qwen3-0.6b-attn kv16k b16 sfi-cycle", num_q_heads=16, num_kv_heads=8, head_dim=128,
          page_size=16, layers=28, batch=16, kv_len=16384, sink=64, recent=256, retention=0.0625,
          refresh_interval=16, heavy_hitter_frac=0.02, heavy_hitter_beta=3.0)
# Table 1 retention points at 16K: n/64 of the KV length (n = 1 is below sink + recent: recent 192, k = 0)
SWEEP_N = [1, 4, 8, 16, 24, 32, 48, 63, 64]
TABLE1 = {1: 10.67, 4: 9.56, 8: 7.15, 16: 3.96, 24: 2.75, 32: 2.10, 48: 1.43, 63: 1.10, 64: 1.00}


SECTIONS = ("overlap", "retention", "speculative", "batch1", "qwen3_8b", "other", "ragged", "ragged_schedule")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["sfi", "reference"], default="sfi")
    ap.add_argument("--no-sweep", action="store_true", help="skip the retention and speculative sweeps")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline leg")
    ap.add_argument("--layers", type=int, default=WL["layers"])
    ap.add_argument("--batch", type=int, default=WL["batch"])
    ap.add_argument("--kv-len", type=int, default=WL["kv_len"])
    ap.add_argument("--sections", default=",".join(SECTIONS),
                    help="comma list of the sections after the headline: " + ", ".join(SECTIONS))
    ap.add_argument("--ragged-requests", type=int, default=64, help="requests of the ragged mixed-step section")
    ap.add_argument("--spec-tokens", default="1,2,4,8", help="comma list of draft/verify token counts (speculative)")
    args = ap.parse_args()
    args.sections = [x for x in args.sections.split(",") if x]
    args.spec_tokens = [int(x) for x in args.spec_tokens.split(",") if x]
    unknown = set(args.sections) - set(SECTIONS)
    if unknown:
        ap.error(f"unknown sections {sorted(unknown)}")
    return args


# ---------------------------------------------------------------------------
# ranks
# ---------------------------------------------------------------------------
def rank_info():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


class Ranks:
    def __init__(self):
        self.rank, self.world, self.local = rank_info()
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
            self.dist = dist

    def barrier(self):
        if self.world > 1:
            self.dist.barrier()

    def max(self, x: float) -> float:
        if self.world == 1:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.world > 1:
            self.dist.destroy_process_group()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------
def fast_bytes(B, Hq, Hkv, D, P, n_ret, W):
    """K/V rows of sink + selected + recent, q in, o out (fp32) and lse, recent page ids."""
    return B * Hkv * n_ret * 4 * D + B * Hq * D * (2 + 4) + B * Hq * 4 + B * (math.ceil(W / P) + 1) * 4


def dense_bytes(B, Hq, Hkv, D, P, L, scores):
    b = B * Hkv * L * 4 * D + B * math.ceil(L / P) * 4 + B * Hq * D * (2 + 4) + B * Hq * 4
    if scores:
        b += B * Hkv * L * 4
    return b


def select_bytes(B, Hkv, nC, k):
    return B * Hkv * nC * 4 + B * Hkv * k * 4


def compact_bytes(B, Hkv, D, S, k):
    return 2 * B * Hkv * (S + k) * 4 * D + B * Hkv * k * 4


def append_bytes(B, Hkv, D):
    return 2 * 2 * B * Hkv * D * 2


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
# DRAM bytes (read + write) per launch from `ncu --set full` captures of the attention
# kernel at the benchmark's per-launch shape (16 requests x 8 KV heads at KV 16K; the
# summaries under profiles/ give the commands). They describe the kernel built from
# the sources whose hash is recorded here and are dropped (null) once those change.
PROFILED_SOURCES = ("sparse_kv_long_sfi_gb300/csrc/attn_kernel.cuh", "sparse_kv_long_sfi_gb300/csrc/attn_decode.cu",
                    "sparse_kv_long_sfi_gb300/csrc/sfi_device.cuh", "sparse_kv_long_sfi_gb300/csrc/sfi_internal.h",
                    "sparse_kv_long_sfi_gb300/csrc/sfi_api.cu")
PROFILED_TRAFFIC = {"sha256_16": "b1a619051ccb121b", "fast": 68_289_280 + 574_208, "slow": 1_073_954_560 + 6_764_800}


def profiled_traffic(kind):
    import hashlib
    h = hashlib.sha256()
    for f in PROFILED_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return PROFILED_TRAFFIC[kind] if h.hexdigest()[:16] == PROFILED_TRAFFIC["sha256_16"] else None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


class Cycle:
    """One SFI refresh cycle of a uniform batch, resident in HBM: 1 slow + (cyc - 1) fast
    decode steps over NL layers through SFIDecoder (main + side stream), replayable as
    one CUDA graph. Every layer has its own paged pools, compact buffers and scores."""

    def __init__(self, dev, seed0, Hq, Hkv, NL, B, L0, retention, cyc, D=128, P=16, S=64, W=256, heavy=True,
                 k_cap=None):
        import torch
        import sfi_synth as syn
        import sparse_kv_long_sfi_gb300 as sfi
        self.dev, self.Hq, self.Hkv, self.NL, self.B, self.L0 = dev, Hq, Hkv, NL, B, L0
        self.D, self.P, self.S, self.W, self.cyc = D, P, S, W, cyc
        self.shape = sfi.AttnShape(Hq, Hkv, D, P)
        self.k = syn.retention_budget(retention, L0, S, W)
        k_cap = self.k if k_cap is None else max(self.k, k_cap)
        g = syn.rng(seed0, 1)
        table, num_pages = syn.make_page_table(g, [L0 + cyc] * B, P, shuffle=True)
        self.page_table = torch.as_tensor(table).to(dev)
        off, cap = sfi.compact_layout(self.shape, S, [k_cap] * B, device=dev)
        self.batch = sfi.DecodeBatch(self.page_table, off, cap, torch.full((B,), self.k, dtype=torch.int32, device=dev),
                                     k_cap, score_stride=L0 + cyc)
        self.seq_steps = torch.tensor([[L0 + t] * B for t in range(cyc)], dtype=torch.int32, device=dev)
        self.q_all = torch.empty((cyc, NL, B, Hq, D), dtype=torch.bfloat16, device=dev)
        self.kn_all = torch.empty((cyc, NL, B, Hkv, D), dtype=torch.bfloat16, device=dev)
        self.vn_all = torch.empty_like(self.kn_all)
        syn.device_normal_bf16_(self.q_all, syn.stream_seed(seed0, 2))
        syn.device_normal_bf16_(self.kn_all, syn.stream_seed(seed0, 3))
        syn.device_normal_bf16_(self.vn_all, syn.stream_seed(seed0, 4))
        self.out = torch.zeros((NL, B, Hq, D), dtype=torch.float32, device=dev)

        def pool_init(i, kp, vp):
            syn.device_normal_bf16_(kp, syn.stream_seed(seed0, 10, i))
            syn.device_normal_bf16_(vp, syn.stream_seed(seed0, 11, i))
            if heavy:
                syn.device_plant_heavy_hitters_(kp, self.page_table, self.q_all[0, i], self.seq_steps[0], S, W,
                                                WL["heavy_hitter_frac"], WL["heavy_hitter_beta"],
                                                syn.stream_seed(seed0, 12, i))

        t0 = time.time()
        self.layers = sfi.allocate_layers(self.shape, NL, num_pages, self.batch, S, device=dev, pool_init=pool_init)
        torch.cuda.synchronize()
        self.alloc_s = time.time() - t0
        self.dec = sfi.SFIDecoder(self.shape, self.layers, self.batch, S, W, max_len=L0 + cyc, device=dev, k_max=self.k)
        self.ios = [sfi.StepIO(self.q_all[t], self.kn_all[t], self.vn_all[t], self.out) for t in range(cyc)]
        # algorithmic bytes: per launch (the fused append included) and per cycle
        self.by_fast = fast_bytes(B, Hq, Hkv, D, P, S + self.k + W, W) + append_bytes(B, Hkv, D)
        self.by_slow = dense_bytes(B, Hq, Hkv, D, P, L0, scores=True) + append_bytes(B, Hkv, D)
        self.by_aux = select_bytes(B, Hkv, L0 - S - W, self.k) + compact_bytes(B, Hkv, D, S, self.k)
        self.by_cycle = NL * (self.by_slow + self.by_aux) + (cyc - 1) * NL * self.by_fast
        self.launches_per_cycle = NL * 3 + (cyc - 1) * NL  # slow + Selector + compaction, then fast

    def run(self, dec=None, marks=None):
        """Issue one cycle on dec's streams; with marks, record timing events at the decode-
        step boundaries of the main stream as ("slow"|"fast", start, end)."""
        import torch
        dec = dec or self.dec

        def mark():
            ev = torch.cuda.Event(enable_timing=True, external=True)
            ev.record(dec.main)
            return ev
        for t in range(self.cyc):
            a = mark() if marks is not None else None
            if t == 0:
                dec.slow_step(self.ios[0], self.seq_steps[0])
            else:
                dec.fast_step(self.ios[t], self.seq_steps[t])
            if marks is not None:
                marks.append(("slow" if t == 0 else "fast", a, mark()))
        dec.join()

    def graph(self, fn):
        import torch
        with torch.cuda.stream(self.dec.main):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.dec.main):
            fn()
        return g

    def replay_ms(self, g, reps, warmup):
        import torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.dec.main):
            for _ in range(warmup):
                g.replay()
            e0.record(self.dec.main)
            for _ in range(reps):
                g.replay()
            e1.record(self.dec.main)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    def step_durations(self, reps, warmup):
        """Per-layer durations of the slow step and of each fast step (µs), from events at
        the decode-step boundaries captured as graph nodes, read after the last replay."""
        marks = []
        g = self.graph(lambda: (marks.clear(), self.run(marks=marks)))
        ms = self.replay_ms(g, reps, warmup)
        dur = {"slow": [], "fast": []}
        for kind, a, b in marks:
            dur[kind].append(a.elapsed_time(b) * 1e3 / self.NL)
        return dur, ms

    def aux_alone_us(self, reps=5):
        """The side stream's work of one slow step (Selector + compaction of every layer)
        timed alone, as one graph on one stream, per layer."""
        import sparse_kv_long_sfi_gb300 as sfi
        d = self.dec

        def aux():
            for i, Lb in enumerate(self.layers):
                kv = sfi.PagedKV(Lb.k_pool, Lb.v_pool, self.page_table, self.seq_steps[0])
                sfi.sfi_select_compact(self.shape, kv, Lb.scores, self.S, self.W, self.batch.k_per_req, Lb.idx,
                                       Lb.compact, stream=d.main)
        g = self.graph(aux)
        return self.replay_ms(g, reps, 2) * 1e3 / self.NL

    def free(self):
        import torch
        del self.layers, self.dec, self.ios, self.q_all, self.kn_all, self.vn_all, self.out
        torch.cuda.synchronize()
        torch.cuda.empty_cache()


def cycle_report(cy, dur, ms_cycle, peak):
    """Amortised decode step and per-launch figures of a measured cycle."""
    fast_wait = dur["fast"][:1]
    fast_clean = dur["fast"][1:] or dur["fast"]
    t_fast = statistics.mean(fast_clean)
    t_first = statistics.mean(fast_wait)
    t_slow = statistics.mean(dur["slow"])
    gbps = lambda by, us: round(by / (us * 1e-6) / 1e9, 1)
    return {"us_per_step": round(ms_cycle * 1e3 / cy.cyc, 3),
            "tokens_per_s": round(cy.B * cy.cyc / (ms_cycle * 1e-3), 1),
            "hbm_GBps_cycle": gbps(cy.by_cycle, ms_cycle * 1e3),
            "frac_of_peak_cycle": round(cy.by_cycle / (ms_cycle * 1e-3) / 1e9 / peak, 3),
            "bytes_per_cycle": cy.by_cycle,
            "fast_us_per_launch": round(t_fast, 3), "fast_bytes_per_launch": cy.by_fast,
            "fast_GBps": gbps(cy.by_fast, t_fast), "fast_frac_of_peak": round(cy.by_fast / (t_fast * 1e-6) / 1e9 / peak, 3),
            "slow_us_per_launch": round(t_slow, 3), "slow_bytes_per_launch": cy.by_slow,
            "slow_GBps": gbps(cy.by_slow, t_slow), "slow_frac_of_peak": round(cy.by_slow / (t_slow * 1e-6) / 1e9 / peak, 3),
            "first_fast_step_us_per_layer": round(t_first, 3)}


def overlap_report(cy, dur, ms_cycle, peak, reps):
    """The side stream's overlap (SFI Figure 3 (A)): the same cycle with the Selector and
    compaction issued on the main stream (serial) against the two-stream cycle, the side
    work timed alone, and the first fast step's penalty against its HBM floor."""
    import sparse_kv_long_sfi_gb300 as sfi
    d = cy.dec
    serial = sfi.SFIDecoder(cy.shape, cy.layers, cy.batch, cy.S, cy.W, max_len=cy.L0 + cy.cyc, device=cy.dev,
                            main_stream=d.main, aux_stream=d.main, k_max=cy.k)
    g = cy.graph(lambda: cy.run(dec=serial))
    ms_serial = cy.replay_ms(g, reps, 2)
    del g
    aux_us = cy.aux_alone_us()
    t_fast = statistics.mean(dur["fast"][1:] or dur["fast"])
    t_first = statistics.mean(dur["fast"][:1])
    floor_us = cy.by_aux / (peak * 1e3)  # the side work's own bytes at the measured copy bandwidth
    saved = (ms_serial - ms_cycle) * 1e3 / cy.NL  # per layer of the slow step
    return {"serial_cycle_ms": round(ms_serial, 4), "overlapped_cycle_ms": round(ms_cycle, 4),
            "aux_alone_us_per_layer": round(aux_us, 3), "saved_us_per_layer": round(saved, 3),
            "overlap_efficiency": round(saved / aux_us, 3) if aux_us > 0 else None,
            "first_fast_step_us_per_layer": round(t_first, 3), "fast_step_us_per_layer": round(t_fast, 3),
            "first_fast_step_ratio": round(t_first / t_fast, 3),
            "aux_bytes_per_layer": cy.by_aux, "aux_hbm_floor_us_per_layer": round(floor_us, 3),
            "first_fast_penalty_us_per_layer": round(t_first - t_fast, 3),
            "penalty_over_floor": round((t_first - t_fast) / floor_us, 3),
            "note": "efficiency = (serial - overlapped) / side work alone; the first fast step after a slow step "
                    "waits for the side work layer by layer, and its extra time is compared with the side work's "
                    "own HBM bytes (Selector reads, compaction reads and writes) at the measured copy bandwidth"}


def run_gpu(args, ranks: Ranks):
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import sparse_kv_long_sfi_gb300 as sfi

    dev = torch.device("cuda", ranks.local)
    torch.cuda.set_device(dev)
    Hq, Hkv, D, P = WL["num_q_heads"], WL["num_kv_heads"], WL["head_dim"], WL["page_size"]
    NL, B, L0 = args.layers, args.batch, args.kv_len
    S, W, cyc = WL["sink"], WL["recent"], WL["refresh_interval"]
    seed0 = 1000 + 97 * ranks.rank
    sections = [] if args.no_sweep else args.sections
    peak, peak_kind = measured_peaks()

    # room in the compact buffers for the 100% point of the retention sweep
    cy = Cycle(dev, seed0, Hq, Hkv, NL, B, L0, WL["retention"], cyc, D, P, S, W, heavy=True,
               k_cap=(L0 - S - W) if "retention" in sections else None)
    dec, k_main = cy.dec, cy.k

    # eager warm-up (sets kernel attributes; checks status)
    with torch.cuda.stream(dec.main):
        cy.run()
    torch.cuda.synchronize()
    assert dec.dev_status.item() == 0, f"device status {dec.dev_status.item()}"

    # headline graph: the cycle with no timing nodes
    g_cycle = cy.graph(cy.run)
    with torch.cuda.stream(dec.main):
        for _ in range(args.warmup):
            g_cycle.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    ranks.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(dec.main):
        e0.record(dec.main)
        for _ in range(args.steps):
            g_cycle.replay()
        e1.record(dec.main)
    torch.cuda.synchronize()
    ranks.barrier()
    clk = clocks.stop()
    ms_cycle = ranks.max(e0.elapsed_time(e1) / args.steps)
    assert dec.dev_status.item() == 0, f"device status {dec.dev_status.item()}"

    # per-kernel averages: the same cycle with timing events (graph nodes) at the step
    # boundaries only; each step's main stream is NL back-to-back attention launches
    reps = max(3, min(args.steps, 10))
    try:
        dur, ms_marked = cy.step_durations(reps, args.warmup)
        timing_method = (f"events at decode-step boundaries (graph nodes), {NL} back-to-back launches per step, "
                         f"last of {reps} replays after the headline region; the fast kernel's average over the "
                         f"{cyc - 2} fast steps that do not follow the slow step")
    except RuntimeError as exc:
        dur, ms_marked = None, None
        timing_method = f"unavailable: {exc}"

    us_step = ms_cycle * 1e3 / cyc
    roofline = None
    if dur:
        # The first fast step after the slow step also waits, layer by layer, for the
        # side stream's Selector and compaction, so the fast kernel's own duration is
        # taken from the other fast steps; the first one is reported on its own.
        rep = cycle_report(cy, dur, ms_marked, peak)
        t_fast, t_slow, t_first = rep["fast_us_per_launch"], rep["slow_us_per_launch"], rep["first_fast_step_us_per_layer"]
        share_fast = (t_fast * (cyc - 2) + t_first) * NL / (ms_marked * 1e3)
        share_slow = t_slow * NL / (ms_marked * 1e3)
        if share_slow >= share_fast:
            name, per, tl, sh = "attn_decode_kernel<128,dense,scores> (slow step)", cy.by_slow, t_slow, share_slow
        else:
            name, per, tl, sh = "attn_decode_kernel<128,fast> (fast step)", cy.by_fast, t_fast, share_fast
        ach = per / (tl * 1e-6) / 1e9
        roofline = {"bound": "hbm", "kernel": name, "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(ach / peak, 4), "peak_kind": f"{peak_kind} hbm_gbs (burst copy)",
                    "traffic": profiled_traffic("fast" if "fast" in name else "slow"), "bytes_per_launch": per,
                    "avg_launch_us": round(tl, 3), "time_share": round(sh, 4), "timing": timing_method,
                    "other": {"fast_avg_us": t_fast, "fast_GBps": rep["fast_GBps"], "fast_share": round(share_fast, 4),
                              "first_fast_step_us_per_layer": t_first,
                              "first_fast_step_note": "waits for the side stream's Selector and compaction",
                              "slow_avg_us": t_slow, "slow_GBps": rep["slow_GBps"], "slow_share": round(share_slow, 4)}}

    result = {
        "metric": METRIC, "value": round(us_step, 3), "unit": UNIT, "n_gpus": ranks.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_cycle, 4), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {**WL, "layers": NL, "batch": B, "kv_len": L0, "k": k_main,
                   "step": f"1 slow + {cyc - 1} fast decode steps x {NL} layers (one CUDA graph)",
                   "l2": f"inputs larger than L2: {NL} distinct layers, {cy.by_cycle / cyc / 1e9:.2f} GB per decode step",
                   "parallelism": f"replicas x{ranks.world}"},
        "us_per_step_with_step_timing_nodes": round(ms_marked * 1e3 / cyc, 3) if ms_marked else None,
        "tokens_per_s": round(ranks.world * B * cyc / (ms_cycle * 1e-3), 1),
        "hbm_GBps_cycle": round(cy.by_cycle / (ms_cycle * 1e-3) / 1e9, 1),
        "bytes_per_cycle": cy.by_cycle,
        "gpu_launches": cy.launches_per_cycle * args.steps,
        "clocks": clk,
        "roofline": roofline,
        "alloc_s": round(cy.alloc_s, 1),
    }

    # ---- end to end through the public API with host buffers ----
    result["e2e"] = e2e_cycle(args, dec, cy.ios, cy.seq_steps, cyc, NL, B, Hq, Hkv, D, dev, ranks)

    if "overlap" in sections and dur:
        result["overlap"] = overlap_report(cy, dur, ms_cycle, peak, reps=max(3, min(args.steps, 5)))
    if "retention" in sections:
        result["retention_sweep"] = retention_sweep(cy, dev, peak)
    if "speculative" in sections:
        result["speculative_sweep"] = speculative_sweep(dec, cy.layers, cy.batch, cy.shape, cy.q_all, cy.seq_steps,
                                                        NL, B, Hq, Hkv, D, P, L0, S, W, k_main, dev, peak, seed0,
                                                        tokens=args.spec_tokens)
    cy.free()
    del cy, dec, g_cycle
    torch.cuda.empty_cache()
    if "batch1" in sections:
        result["batch1"] = batch_one(args, dev, peak, seed0)
    if "qwen3_8b" in sections:
        result["qwen3_8b_cycle"] = qwen3_8b_cycle(args, dev, peak, seed0)
    if "other" in sections:
        result["other_workloads"] = other_workloads(dev, peak, seed0)
    if "ragged" in sections:
        result["ragged_mixed_step"] = ragged_mixed_step(dev, peak, seed0, B=args.ragged_requests)
    if "ragged_schedule" in sections:
        result["ragged_schedule"] = ragged_schedule(dev, peak, seed0, B=args.ragged_requests)
    return result


def batch_one(args, dev, peak, seed0):
    """Config 2's other batch: the same Qwen3-0.6B cycle and Table 1 retention sweep at batch 1."""
    import torch
    reps = max(3, min(args.steps, 10))
    cy = Cycle(dev, seed0 + 5, WL["num_q_heads"], WL["num_kv_heads"], args.layers, 1, args.kv_len, WL["retention"],
               WL["refresh_interval"], heavy=True, k_cap=args.kv_len - WL["sink"] - WL["recent"])
    with torch.cuda.stream(cy.dec.main):
        cy.run()
    torch.cuda.synchronize()
    g = cy.graph(cy.run)
    ms = cy.replay_ms(g, max(3, args.steps), args.warmup)
    dur, _ = cy.step_durations(reps, 2)
    rep = cycle_report(cy, dur, ms, peak)
    rep["retention_sweep"] = retention_sweep(cy, dev, peak)
    assert cy.dec.dev_status.item() == 0
    cy.free()
    return {"workload": f"qwen3-0.6b-attn kv{args.kv_len} b1 sfi-cycle, {args.layers} layers", **rep}


def qwen3_8b_cycle(args, dev, peak, seed0, NL=36, B=32, L0=32768):
    """The Qwen3-8B-shaped workload as stated: 32 Q / 8 KV heads, 36 layers, batch 32, KV
    32K, fast steps at 6.25% retention with one slow step every 16 (its Selector and
    compaction on the side stream, overlapped with the next layers), as one graph."""
    import torch
    free, total = torch.cuda.mem_get_info(dev)
    need = 2 * NL * B * (L0 + 32) * 8 * 128 * 2 * 1.08
    if need > free:
        return {"skipped": f"needs about {need / 1e9:.0f} GB of device memory, {free / 1e9:.0f} GB free"}
    reps = 3
    cy = Cycle(dev, seed0 + 7, 32, 8, NL, B, L0, 0.0625, WL["refresh_interval"], heavy=False)
    with torch.cuda.stream(cy.dec.main):
        cy.run()
    torch.cuda.synchronize()
    g = cy.graph(cy.run)
    ms = cy.replay_ms(g, reps, 1)
    dur, _ = cy.step_durations(reps, 1)
    rep = cycle_report(cy, dur, ms, peak)
    del g
    ov = overlap_report(cy, dur, ms, peak, reps=2)
    assert cy.dec.dev_status.item() == 0
    alloc = cy.alloc_s
    kv_gb = 2 * NL * cy.layers[0].k_pool.numel() * 2 / 1e9
    cy.free()
    return {"workload": f"qwen3-8b-attn kv{L0} b{B} sfi-cycle, {NL} layers, k {cy.k}", "kv_GB": round(kv_gb, 1),
            **rep, "overlap": ov, "alloc_s": round(alloc, 1),
            "note": "one graph per refresh cycle (1 slow + 15 fast decode steps x 36 layers); amortised per decode "
                    "step; Q/K/V N(0,1)"}


def ragged_schedule(dev, peak, seed0, B=64, steps=64, p_boundary=0.06, interval=32):
    """Config 5 as a schedule: B (64) requests with lengths log-uniform in [4096, 131072],
    32 Q / 8 KV heads, shuffled pages, per-request retention from {3, 12.5, 25}%, and a
    seeded boundary process (slow with p = 0.06 per token, forced every 32 steps, the first
    step slow) run for `steps` decode steps of one layer. Each step is one attention
    launch (fast and slow requests together) plus, for the slow requests, the Selector and
    compaction on the side stream; k is fixed at each slow step from the request's
    retention. The whole run is one graph."""
    import numpy as np
    import torch
    import sfi_synth as syn
    import sparse_kv_long_sfi_gb300 as sfi

    Hq, Hkv, D, P, S, W = 32, 8, 128, 16, 64, 256
    shape = sfi.AttnShape(Hq, Hkv, D, P)
    g = syn.rng(seed0, 60)
    lens = syn.log_uniform_lengths(g, B, 4096, 131072) - 1
    ret = g.choice([0.03, 0.125, 0.25], size=B)
    k_cap = max(syn.retention_budget(ret[r], int(lens[r]) + steps, S, W) for r in range(B))
    caps = [syn.retention_budget(ret[r], int(lens[r]) + steps, S, W) for r in range(B)]
    table, num_pages = syn.make_page_table(g, lens + steps + 1, P, shuffle=True)
    pt = torch.as_tensor(table).to(dev)
    off, cap = sfi.compact_layout(shape, S, caps, device=dev)
    k_now = np.array([syn.retention_budget(ret[r], int(lens[r]) + 1, S, W) for r in range(B)], np.int32)
    batch = sfi.DecodeBatch(pt, off, cap, torch.as_tensor(k_now).to(dev), k_cap,
                            score_stride=int(lens.max()) + steps + 1)
    lens_t = torch.as_tensor((lens + 1).astype(np.int32)).to(dev)

    q = torch.empty((steps, 1, B, Hq, D), dtype=torch.bfloat16, device=dev)
    kn = torch.empty((steps, 1, B, Hkv, D), dtype=torch.bfloat16, device=dev)
    vn = torch.empty_like(kn)
    for t_, tag in ((q, 61), (kn, 62), (vn, 63)):
        syn.device_normal_bf16_(t_, syn.stream_seed(seed0, tag))

    def init(i, kp, vp):
        syn.device_normal_bf16_(kp, syn.stream_seed(seed0, 64))
        syn.device_normal_bf16_(vp, syn.stream_seed(seed0, 65))
        syn.device_plant_heavy_hitters_(kp, pt, q[0, 0], lens_t, S, W, WL["heavy_hitter_frac"],
                                        WL["heavy_hitter_beta"], syn.stream_seed(seed0, 66))

    layers = sfi.allocate_layers(shape, 1, num_pages, batch, S, device=dev, pool_init=init)
    out = torch.zeros((1, B, Hq, D), dtype=torch.float32, device=dev)
    dec = sfi.SFIDecoder(shape, layers, batch, S, W, max_len=int(lens.max()) + steps + 1, device=dev)
    # the seeded schedule and every step's lengths, ids and k (precomputed on the host)
    sched = sfi.SlowFastSchedule(B, interval)
    draws = syn.boundary_draws(syn.rng(seed0, 67), steps, B, p_boundary)
    plan = []
    cur = lens.astype(np.int64).copy()
    k_host = k_now.copy()
    by_total = 0
    for t in range(steps):
        cur = cur + 1
        m = sched.next(draws[t]).astype(bool)
        for r in np.flatnonzero(m):
            k_host[r] = syn.retention_budget(ret[r], int(cur[r]), S, W)
        sid = torch.as_tensor(np.flatnonzero(m).astype(np.int32)).to(dev)
        fid = torch.as_tensor(np.flatnonzero(~m).astype(np.int32)).to(dev)
        plan.append((m, torch.as_tensor(cur.astype(np.int32)).to(dev), sid, fid,
                     torch.as_tensor(k_host.copy()).to(dev)))
        for r in np.flatnonzero(m):  # slow requests: dense + scores, then the side work
            L = int(cur[r])
            by_total += (dense_bytes(1, Hq, Hkv, D, P, L, scores=True) +
                         select_bytes(1, Hkv, max(0, L - S - W), int(k_host[r])) +
                         compact_bytes(1, Hkv, D, S, int(k_host[r])))
    # fast-step bytes use the selection a request holds at that step (its last slow step's k)
    held = np.zeros(B, np.int64)
    by_fast_total = 0
    for m, _, _, _, kt in plan:
        k_t = kt.cpu().numpy()
        held[m] = k_t[m]
        for r in np.flatnonzero(~m):
            by_fast_total += fast_bytes(1, Hq, Hkv, D, P, S + int(held[r]) + W, W)
    by_total += by_fast_total + steps * append_bytes(B, Hkv, D)

    def run():
        for t, (m, seq, sid, fid, kt) in enumerate(plan):
            dec.batch.k_per_req = kt
            io = sfi.StepIO(q[t], kn[t], vn[t], out)
            if m.all():
                dec.slow_step(io, seq)
            elif not m.any():
                dec.fast_step(io, seq)
            else:
                dec.mixed_step(io, seq, sid, fid)
        dec.join()

    with torch.cuda.stream(dec.main):
        run()
    torch.cuda.synchronize()
    assert dec.dev_status.item() == 0, f"device status {dec.dev_status.item()}"
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=dec.main):
        run()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 5
    with torch.cuda.stream(dec.main):
        gr.replay()
        e0.record(dec.main)
        for _ in range(reps):
            gr.replay()
        e1.record(dec.main)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    n_slow = [int(x[0].sum()) for x in plan]
    del gr, layers, dec, q, kn, vn, out
    torch.cuda.empty_cache()
    return {"workload": f"ragged {B} requests, kv 4K-128K log-uniform, 32q/8kv heads, retention {{3,12.5,25}}%, "
                        f"boundary p={p_boundary}, refresh forced every {interval} steps, {steps} steps, 1 layer",
            "steps": steps, "total_kv_tokens": int(lens.sum()), "us_per_step": round(ms * 1e3 / steps, 2),
            "bytes_per_run": by_total, "GBps": round(by_total / (ms * 1e-3) / 1e9, 1),
            "frac_of_peak": round(by_total / (ms * 1e-3) / 1e9 / peak, 3),
            "slow_requests_per_step_mean": round(float(np.mean(n_slow)), 2),
            "slow_requests_first_step": n_slow[0], "slow_requests_max_after_first": max(n_slow[1:]) if steps > 1 else 0,
            "note": "one graph of all steps; each step: one mixed attention launch (append fused) + Selector and "
                    "compaction of its slow requests on the side stream; bytes include the side work"}


def e2e_cycle(args, dec, ios, seq_steps, cyc, NL, B, Hq, Hkv, D, dev, ranks):
    """The same cycle with every decode step's q/k_new/v_new copied in from pinned
    host memory and its outputs copied back, all inside one captured graph. The copies
    run on their own stream: all steps' inputs go up at the start of the cycle (each step
    waits for its own), and each step's output comes back while the next steps run
    (one output buffer per step)."""
    import torch
    import sparse_kv_long_sfi_gb300 as sfi
    h_q = [io.q.cpu().pin_memory() for io in ios]
    h_k = [io.k_new.cpu().pin_memory() for io in ios]
    h_v = [io.v_new.cpu().pin_memory() for io in ios]
    h_out = [torch.empty(ios[0].out.shape, dtype=torch.float32, pin_memory=True) for _ in range(cyc)]
    eios = [sfi.StepIO(io.q, io.k_new, io.v_new, torch.empty_like(io.out)) for io in ios]
    copy = torch.cuda.Stream(device=dev)

    def cycle():
        copy.wait_stream(dec.main)
        ready = []
        with torch.cuda.stream(copy):
            for t in range(cyc):
                eios[t].q.copy_(h_q[t], non_blocking=True)
                eios[t].k_new.copy_(h_k[t], non_blocking=True)
                eios[t].v_new.copy_(h_v[t], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy)
                ready.append(ev)
        for t in range(cyc):
            dec.main.wait_event(ready[t])
            if t == 0:
                dec.slow_step(eios[0], seq_steps[0])
            else:
                dec.fast_step(eios[t], seq_steps[t])
            done = torch.cuda.Event()
            done.record(dec.main)
            copy.wait_event(done)
            with torch.cuda.stream(copy):
                h_out[t].copy_(eios[t].out, non_blocking=True)
        dec.join()
        dec.main.wait_stream(copy)

    with torch.cuda.stream(dec.main):
        cycle()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=dec.main):
        cycle()
    with torch.cuda.stream(dec.main):
        for _ in range(max(1, args.warmup)):
            g.replay()
    torch.cuda.synchronize()
    n = max(3, args.steps // 2)
    ranks.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(dec.main):
        e0.record(dec.main)
        for _ in range(n):
            g.replay()
        e1.record(dec.main)
    torch.cuda.synchronize()
    ranks.barrier()
    ms = ranks.max(e0.elapsed_time(e1) / n)
    # the copies of one cycle (cyc decode steps), per decode step
    h2d = sum(x.numel() * x.element_size() for x in h_q + h_k + h_v) // cyc
    d2h = sum(x.numel() * x.element_size() for x in h_out) // cyc
    return {"value": round(ms * 1e3 / cyc, 3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": n, "path": "SFIDecoder (libsfi C ABI), pinned host inputs/outputs copied on a side stream, one graph per cycle"}


def retention_sweep(cy, dev, peak):
    """Fast decode steps (all layers) at Table 1's retention points vs the dense decode kernel."""
    import torch
    import sparse_kv_long_sfi_gb300 as sfi

    reps = 20
    dec, layers, batch, shape = cy.dec, cy.layers, cy.batch, cy.shape
    NL, B, Hq, Hkv, D, P, L0, S = cy.NL, cy.B, cy.Hq, cy.Hkv, cy.D, cy.P, cy.L0, cy.S
    q_all, kn_all, vn_all, out, seq_steps = cy.q_all, cy.kn_all, cy.vn_all, cy.out, cy.seq_steps
    L1 = L0 + 1
    seq = seq_steps[1]

    def time_graph(fn):
        g = cy.graph(fn)
        return cy.replay_ms(g, reps, 3) * 1e3

    ws_dense = dec.ws_dense

    def dense_step():
        for i, Lb in enumerate(layers):
            kv = sfi.PagedKV(Lb.k_pool, Lb.v_pool, batch.page_table, seq)
            sfi.sfi_slow_dense_attn_with_scores(shape, kv, S, 0, q_all[1, i], out[i], None, None,
                                                k_new=kn_all[1, i], v_new=vn_all[1, i], max_tokens=L1 + P,
                                                workspace=ws_dense, stream=dec.main, flags=dec.attn_flags)

    us_dense = time_graph(dense_step)
    by_dense = dense_bytes(B, Hq, Hkv, D, P, L1, scores=False) + append_bytes(B, Hkv, D)
    rows = []
    for n in SWEEP_N:
        W = 192 if n == 1 else 256
        k = max(0, n * 256 - S - W) if n < 64 else L0 - S - W
        kreq = torch.full((B,), k, dtype=torch.int32, device=dev)
        # slow step at L0 fills the compact buffers for this retention
        for i, Lb in enumerate(layers):
            kv = sfi.PagedKV(Lb.k_pool, Lb.v_pool, batch.page_table, seq_steps[0])
            sfi.sfi_slow_dense_attn_with_scores(shape, kv, S, W, q_all[0, i], out[i], None, Lb.scores,
                                                max_tokens=L0 + P, workspace=ws_dense, stream=dec.main)
            sfi.sfi_select_topk(Lb.scores, Hkv, seq_steps[0], S, W, kreq, Lb.idx, Lb.compact.count, stream=dec.main)
            sfi.sfi_compact_gather(shape, kv, Lb.idx, Lb.compact.count, S, Lb.compact, stream=dec.main)
        max_tok = S + k + W + 2 * P
        ws_fast = sfi.alloc_workspace(shape, B, max_tok, device=dev)

        def fast_step():
            for i, Lb in enumerate(layers):
                kv = sfi.PagedKV(Lb.k_pool, Lb.v_pool, batch.page_table, seq)
                sfi.sfi_fast_decode_attn(shape, kv, Lb.compact, S, W, q_all[1, i], out[i], None,
                                         k_new=kn_all[1, i], v_new=vn_all[1, i], max_tokens=max_tok,
                                         workspace=ws_fast, stream=dec.main, flags=dec.attn_flags)

        us = time_graph(fast_step)
        n_ret = S + k + W
        by = NL * (fast_bytes(B, Hq, Hkv, D, P, n_ret, W) + append_bytes(B, Hkv, D))
        rows.append({"retention_pct": round(100 * n_ret / L1, 2), "n_over_64": n, "sink": S, "k": k, "recent": W,
                     "us_per_step": round(us, 2), "GBps": round(by / (us * 1e-6) / 1e9, 1),
                     "frac_of_peak": round(by / (us * 1e-6) / 1e9 / peak, 3),
                     "speedup_vs_dense": round(us_dense / us, 3), "table1_speedup_context": TABLE1[n]})
    # Latency floor of a fast launch: the same graph over the smallest state (16 sink rows,
    # no selected rows, one recent page: 32 tokens per (request, KV head)), where the
    # bytes are negligible and the launch costs its fixed start-up and merge.
    Sf, Wf = 16, 16
    k0 = torch.zeros((B,), dtype=torch.int32, device=dev)
    for i, Lb in enumerate(layers):
        kv = sfi.PagedKV(Lb.k_pool, Lb.v_pool, batch.page_table, seq_steps[0])
        sfi.sfi_slow_dense_attn_with_scores(shape, kv, Sf, Wf, q_all[0, i], out[i], None, Lb.scores,
                                            max_tokens=L0 + P, workspace=ws_dense, stream=dec.main)
        sfi.sfi_select_topk(Lb.scores, Hkv, seq_steps[0], Sf, Wf, k0, Lb.idx, Lb.compact.count, stream=dec.main)
        sfi.sfi_compact_gather(shape, kv, Lb.idx, Lb.compact.count, Sf, Lb.compact, stream=dec.main)
    max_tok_f = Sf + Wf + 2 * P
    ws_floor = sfi.alloc_workspace(shape, B, max_tok_f, device=dev)

    def floor_step():
        for i, Lb in enumerate(layers):
            kv = sfi.PagedKV(Lb.k_pool, Lb.v_pool, batch.page_table, seq)
            sfi.sfi_fast_decode_attn(shape, kv, Lb.compact, Sf, Wf, q_all[1, i], out[i], None,
                                     k_new=kn_all[1, i], v_new=vn_all[1, i], max_tokens=max_tok_f,
                                     workspace=ws_floor, stream=dec.main, flags=dec.attn_flags)

    floor_us = time_graph(floor_step) / NL
    for r in rows:
        per = r["us_per_step"] / NL
        by_launch = r["GBps"] * 1e9 * per * 1e-6
        r["us_per_launch"] = round(per, 3)
        r["bytes_at_peak_us_per_launch"] = round(by_launch / (peak * 1e3), 3)
        r["over_latency_floor_us_per_launch"] = round(per - floor_us, 3)
    # restore the main cycle's selection state
    dec.pending = [False] * len(layers)
    return {"batch": B, "dense_us_per_step": round(us_dense, 2),
            "dense_GBps": round(NL * by_dense / (us_dense * 1e-6) / 1e9, 1),
            "dense_frac_of_peak": round(NL * by_dense / (us_dense * 1e-6) / 1e9 / peak, 3),
            "latency_floor_us_per_launch": round(floor_us, 3),
            "latency_floor_state": f"sink {Sf}, k 0, recent {Wf}: {Sf + Wf} tokens per (request, KV head)",
            "points": rows, "note": f"fast and dense steps include the (fused) paged append; {NL} layers per step; "
                                    "Table 1 speedups are the paper's (hardware unstated), context only; "
                                    "latency_floor_us_per_launch is a fast launch over the smallest state (its fixed "
                                    "start-up and merge cost), bytes_at_peak the point's bytes at the measured copy "
                                    "bandwidth: a point is latency-bound where its time sits near the floor plus that"}


def speculative_sweep(dec, layers, batch, shape, q_all, seq_steps, NL, B, Hq, Hkv, D, P, L0, S, W, k_main, dev, peak,
                      seed0, tokens=(1, 2, 4, 8)):
    """Self-speculative decoding's two passes over all layers ("A Sparse Glimpse of the
    Whole", abstract): verification of T tokens (T-token append + causal dense
    attention + the recycled statistic) and a T-token draft pass over the sparse state
    at the main workload's retention, each as one graph of NL layers."""
    import torch
    import sfi_synth as syn
    import sparse_kv_long_sfi_gb300 as sfi

    reps = 20

    def time_graph(fn):
        with torch.cuda.stream(dec.main):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=dec.main):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(dec.main):
            for _ in range(3):
                g.replay()
            e0.record(dec.main)
            for _ in range(reps):
                g.replay()
            e1.record(dec.main)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    # the main workload's selection (k_main at L0) in every layer's compact buffer
    kreq = torch.full((B,), k_main, dtype=torch.int32, device=dev)
    scratch = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    for i, Lb in enumerate(layers):
        kv = sfi.PagedKV(Lb.k_pool, Lb.v_pool, batch.page_table, seq_steps[0])
        sfi.sfi_slow_dense_attn_with_scores(shape, kv, S, W, q_all[0, i], scratch, None, Lb.scores,
                                            max_tokens=L0 + P, workspace=dec.ws_dense, stream=dec.main)
        sfi.sfi_select_topk(Lb.scores, Hkv, seq_steps[0], S, W, kreq, Lb.idx, Lb.compact.count, stream=dec.main)
        sfi.sfi_compact_gather(shape, kv, Lb.idx, Lb.compact.count, S, Lb.compact, stream=dec.main)
    torch.cuda.synchronize()
    rows = []
    for T in tokens:
        L = L0 + T
        seq = torch.full((B,), L, dtype=torch.int32, device=dev)
        q = torch.empty((NL, B, T, Hq, D), dtype=torch.bfloat16, device=dev)
        kn = torch.empty((NL, B, T, Hkv, D), dtype=torch.bfloat16, device=dev)
        vn = torch.empty_like(kn)
        syn.device_normal_bf16_(q, syn.stream_seed(seed0, 30, T))
        syn.device_normal_bf16_(kn, syn.stream_seed(seed0, 31, T))
        syn.device_normal_bf16_(vn, syn.stream_seed(seed0, 32, T))
        o = torch.empty((NL, B, T, Hq, D), dtype=torch.float32, device=dev)
        ws_v = sfi.alloc_multi_workspace(shape, B, T, L + P, device=dev)
        max_draft = S + k_main + W + T + 2 * P
        ws_d = sfi.alloc_multi_workspace(shape, B, T, max_draft, device=dev)

        def verify():
            for i, Lb in enumerate(layers):
                kv = sfi.PagedKV(Lb.k_pool, Lb.v_pool, batch.page_table, seq)
                sfi.sfi_dense_verify_attn(shape, kv, S, W, q[i], T, o[i], None, Lb.scores, max_tokens=L + P,
                                          workspace=ws_v, stream=dec.main, flags=dec.attn_flags, k_new=kn[i],
                                          v_new=vn[i])

        def draft():
            for i, Lb in enumerate(layers):
                kv = sfi.PagedKV(Lb.k_pool, Lb.v_pool, batch.page_table, seq)
                sfi.sfi_sparse_draft_attn(shape, kv, Lb.compact, S, W, q[i], T, o[i], None, max_tokens=max_draft,
                                          workspace=ws_d, stream=dec.main, flags=dec.attn_flags, k_new=kn[i],
                                          v_new=vn[i])

        us_v, us_d = time_graph(verify), time_graph(draft)
        qo = B * T * Hq * (D * (2 + 4) + 4)
        app = 2 * 2 * B * T * Hkv * D * 2
        by_v = NL * (B * Hkv * L * 4 * D + B * math.ceil(L / P) * 4 + B * Hkv * L * 4 + qo + app)
        by_d = NL * (B * Hkv * (S + k_main + W + T - 1) * 4 * D + qo + app)
        rows.append({"tokens": T,
                     "verify_us_per_pass": round(us_v, 2), "verify_us_per_token": round(us_v / T, 2),
                     "verify_GBps": round(by_v / (us_v * 1e-6) / 1e9, 1),
                     "verify_frac_of_peak": round(by_v / (us_v * 1e-6) / 1e9 / peak, 3),
                     "draft_us_per_pass": round(us_d, 2), "draft_us_per_token": round(us_d / T, 2),
                     "draft_GBps": round(by_d / (us_d * 1e-6) / 1e9, 1),
                     "draft_frac_of_peak": round(by_d / (us_d * 1e-6) / 1e9 / peak, 3)})
    dec.pending = [False] * len(layers)
    return {"points": rows, "retention_pct_of_draft": round(100 * (S + k_main + W) / L0, 2),
            "note": f"{NL} layers per pass, batch {B}, KV {L0} + T; each pass includes the T-token paged append "
                    "(fused into the attention kernel); "
                    "verification writes the recycled statistic (masked logits summed over the group and the "
                    "tokens) for every layer"}


OTHER_WORKLOADS = [
    dict(workload="64q/8kv-heads kv64k b8 top-4096", num_q_heads=64, num_kv_heads=8, kv_len=65536, batch=8, k=4096,
         fast=False),
]


def other_workloads(dev, peak, seed0, layers=4, reps=10):
    """Per-launch times of the larger workloads: the slow step's three kernels and (where
    the workload has one) the fast step, each as a graph over `layers` distinct layers
    (every layer's KV exceeds L2), with the append fused as in the decode cycle."""
    import torch
    import sfi_synth as syn
    import sparse_kv_long_sfi_gb300 as sfi

    S, W, D, P = 64, 256, 128, 16
    stream = torch.cuda.Stream(device=dev)

    def timed(fn):
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps / layers

    out_rows = []
    for cfg in OTHER_WORKLOADS:
        Hq, Hkv, L0, B = cfg["num_q_heads"], cfg["num_kv_heads"], cfg["kv_len"], cfg["batch"]
        shape = sfi.AttnShape(Hq, Hkv, D, P)
        k = cfg.get("k") or syn.retention_budget(cfg["retention"], L0, S, W)
        g = syn.rng(seed0, 40, Hq)
        table, num_pages = syn.make_page_table(g, [L0 + 2] * B, P, shuffle=True)
        pt = torch.as_tensor(table).to(dev)
        off, cap = sfi.compact_layout(shape, S, [k] * B, device=dev)
        batch = sfi.DecodeBatch(pt, off, cap, torch.full((B,), k, dtype=torch.int32, device=dev), k,
                                score_stride=L0 + 2)

        def init(i, kp, vp):
            syn.device_normal_bf16_(kp, syn.stream_seed(seed0, 41, Hq, i))
            syn.device_normal_bf16_(vp, syn.stream_seed(seed0, 42, Hq, i))

        lays = sfi.allocate_layers(shape, layers, num_pages, batch, S, device=dev, pool_init=init)
        q = torch.empty((layers, B, Hq, D), dtype=torch.bfloat16, device=dev)
        kn = torch.empty((layers, B, Hkv, D), dtype=torch.bfloat16, device=dev)
        vn = torch.empty_like(kn)
        for t, tag in ((q, 43), (kn, 44), (vn, 45)):
            syn.device_normal_bf16_(t, syn.stream_seed(seed0, tag, Hq))
        o = torch.empty((layers, B, Hq, D), dtype=torch.float32, device=dev)
        seq0 = torch.full((B,), L0, dtype=torch.int32, device=dev)
        seq1 = torch.full((B,), L0 + 1, dtype=torch.int32, device=dev)
        ws_d = sfi.alloc_workspace(shape, B, L0 + 2 * P, device=dev)
        max_fast = S + k + W + 2 * P
        ws_f = sfi.alloc_workspace(shape, B, max_fast, device=dev)
        flags = sfi.SFI_ATTN_EARLY_KV_PREFETCH

        def slow():
            for i, Lb in enumerate(lays):
                kv = sfi.PagedKV(Lb.k_pool, Lb.v_pool, pt, seq0)
                sfi.sfi_slow_dense_attn_with_scores(shape, kv, S, W, q[i], o[i], None, Lb.scores, max_tokens=L0 + 2 * P,
                                                    workspace=ws_d, stream=stream, flags=flags)

        def select():
            for i, Lb in enumerate(lays):
                sfi.sfi_select_topk(Lb.scores, Hkv, seq0, S, W, batch.k_per_req, Lb.idx, Lb.compact.count,
                                    stream=stream)

        def compact():
            for i, Lb in enumerate(lays):
                kv = sfi.PagedKV(Lb.k_pool, Lb.v_pool, pt, seq0)
                sfi.sfi_compact_gather(shape, kv, Lb.idx, Lb.compact.count, S, Lb.compact, stream=stream)

        def fast():
            for i, Lb in enumerate(lays):
                kv = sfi.PagedKV(Lb.k_pool, Lb.v_pool, pt, seq1)
                sfi.sfi_fast_decode_attn(shape, kv, Lb.compact, S, W, q[i], o[i], None, k_new=kn[i], v_new=vn[i],
                                         max_tokens=max_fast, workspace=ws_f, stream=stream, flags=flags)

        t_slow, t_sel, t_cmp = timed(slow), timed(select), timed(compact)
        nC = L0 - S - W
        by_slow = dense_bytes(B, Hq, Hkv, D, P, L0, scores=True)
        row = {"workload": cfg["workload"], "k": k, "layers_timed": layers,
               "slow_us_per_launch": round(t_slow, 2), "slow_GBps": round(by_slow / (t_slow * 1e-6) / 1e9, 1),
               "slow_frac_of_peak": round(by_slow / (t_slow * 1e-6) / 1e9 / peak, 3),
               "select_us_per_launch": round(t_sel, 2), "compact_us_per_launch": round(t_cmp, 2),
               "compact_GBps": round(compact_bytes(B, Hkv, D, S, k) / (t_cmp * 1e-6) / 1e9, 1)}
        if cfg["fast"]:
            t_fast = timed(fast)
            by_fast = fast_bytes(B, Hq, Hkv, D, P, S + k + W, W) + append_bytes(B, Hkv, D)
            row.update({"fast_us_per_launch": round(t_fast, 2),
                        "fast_GBps": round(by_fast / (t_fast * 1e-6) / 1e9, 1),
                        "fast_frac_of_peak": round(by_fast / (t_fast * 1e-6) / 1e9 / peak, 3),
                        "dense_over_fast": round(t_slow / t_fast, 2)})
        out_rows.append(row)
        del lays, q, kn, vn, o, ws_d, ws_f
        torch.cuda.empty_cache()
    return {"points": out_rows, "note": "per launch = one layer; slow = dense attention + masked scores (no append), "
                                        "fast = the sparse step with the fused append; Selector and compaction as in "
                                        "the slow step; bytes as in the main workload's roofline"}


def ragged_mixed_step(dev, peak, seed0, reps=20, n_slow=5, B=64):
    """One decode step of a ragged batch where a few requests take the slow step and the
    rest the fast step (ASPIRE's mixed forward; SFI's per-request boundaries): B (64)
    requests with lengths log-uniform in [4096, 131072], 32 Q / 8 KV heads, retention
    per request from {3, 12.5, 25}%, `n_slow` slow requests. Times the attention of the
    step (appends fused) as one mixed launch and as two launches."""
    import numpy as np
    import torch
    import sfi_synth as syn
    import sparse_kv_long_sfi_gb300 as sfi

    Hq, Hkv, D, P, S, W = 32, 8, 128, 16, 64, 256
    n_slow = min(n_slow, B)
    shape = sfi.AttnShape(Hq, Hkv, D, P)
    g = syn.rng(seed0, 50)
    lens = syn.log_uniform_lengths(g, B, 4096, 131072)
    ret = g.choice([0.03, 0.125, 0.25], size=B)
    ks = [syn.retention_budget(ret[r], int(lens[r]), S, W) for r in range(B)]
    k_cap = max(ks)
    table, num_pages = syn.make_page_table(g, lens + 2, P, shuffle=True)
    pt = torch.as_tensor(table).to(dev)
    off, cap = sfi.compact_layout(shape, S, ks, device=dev)
    batch = sfi.DecodeBatch(pt, off, cap, torch.as_tensor(np.asarray(ks, np.int32)).to(dev), k_cap,
                            score_stride=int(lens.max()) + 2)

    def init(i, kp, vp):
        syn.device_normal_bf16_(kp, syn.stream_seed(seed0, 51))
        syn.device_normal_bf16_(vp, syn.stream_seed(seed0, 52))

    (lay,) = sfi.allocate_layers(shape, 1, num_pages, batch, S, device=dev, pool_init=init)
    q = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    kn = torch.empty((B, Hkv, D), dtype=torch.bfloat16, device=dev)
    vn = torch.empty_like(kn)
    for t, tag in ((q, 53), (kn, 54), (vn, 55)):
        syn.device_normal_bf16_(t, syn.stream_seed(seed0, tag))
    o = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    seq0 = torch.as_tensor(lens.astype(np.int32)).to(dev)
    seq1 = seq0 + 1
    max_dense = int(lens.max()) + 2 * P
    max_fast = S + k_cap + W + 2 * P
    stream = torch.cuda.Stream(device=dev)
    # every request's selection from a slow step at its length
    ws_d = sfi.alloc_workspace(shape, B, max_dense, device=dev)
    with torch.cuda.stream(stream):
        kv0 = sfi.PagedKV(lay.k_pool, lay.v_pool, pt, seq0)
        sfi.sfi_slow_dense_attn_with_scores(shape, kv0, S, W, q, o, None, lay.scores, max_tokens=max_dense,
                                            workspace=ws_d, stream=stream)
        sfi.sfi_select_compact(shape, kv0, lay.scores, S, W, batch.k_per_req, lay.idx, lay.compact, stream=stream)
    torch.cuda.synchronize()
    slow = np.sort(g.choice(B, size=n_slow, replace=False)).astype(np.int32)
    fast = np.setdiff1d(np.arange(B, dtype=np.int32), slow)
    slow_ids, fast_ids = torch.as_tensor(slow).to(dev), torch.as_tensor(fast).to(dev)
    kv1 = sfi.PagedKV(lay.k_pool, lay.v_pool, pt, seq1)
    ws_m = sfi.alloc_mixed_workspace(shape, B, max_fast, max_dense, device=dev)
    ws_f = sfi.alloc_workspace(shape, B, max_fast, device=dev)
    ws_fr = sfi.alloc_ragged_workspace(shape, B, max_fast, device=dev)
    ws_dr = sfi.alloc_ragged_workspace(shape, B, max_dense, dense=True, device=dev)
    flags = sfi.SFI_ATTN_EARLY_KV_PREFETCH
    rflags = flags | sfi.SFI_ATTN_RAGGED

    def one_launch():
        sfi.sfi_mixed_decode_attn(shape, kv1, lay.compact, S, W, q, o, fast_ids, slow_ids, scores=lay.scores,
                                  k_new=kn, v_new=vn, max_fast_tokens=max_fast, max_dense_tokens=max_dense,
                                  flags=flags, workspace=ws_m, stream=stream)

    def two_launches():
        sfi.sfi_fast_decode_attn(shape, kv1, lay.compact, S, W, q, o, None, k_new=kn, v_new=vn, req_ids=fast_ids,
                                 batch=len(fast), max_tokens=max_fast, workspace=ws_f, stream=stream, flags=flags)
        sfi.sfi_slow_dense_attn_with_scores(shape, kv1, S, W, q, o, None, lay.scores, k_new=kn, v_new=vn,
                                            req_ids=slow_ids, batch=len(slow), max_tokens=max_dense,
                                            workspace=ws_d, stream=stream, flags=flags)

    def timed(fn):
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            gr.replay()
            e0.record(stream)
            for _ in range(reps):
                gr.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    def two_launches_ragged():
        sfi.sfi_fast_decode_attn(shape, kv1, lay.compact, S, W, q, o, None, k_new=kn, v_new=vn, req_ids=fast_ids,
                                 batch=len(fast), max_tokens=max_fast, workspace=ws_fr, stream=stream, flags=rflags)
        sfi.sfi_slow_dense_attn_with_scores(shape, kv1, S, W, q, o, None, lay.scores, k_new=kn, v_new=vn,
                                            req_ids=slow_ids, batch=len(slow), max_tokens=max_dense,
                                            workspace=ws_dr, stream=stream, flags=rflags)

    # the whole batch in a fast step: the same split count for every request, or
    # chunks sized by each request's own length (SFI_ATTN_RAGGED)
    def fast_only_even():
        sfi.sfi_fast_decode_attn(shape, kv1, lay.compact, S, W, q, o, None, k_new=kn, v_new=vn, max_tokens=max_fast,
                                 workspace=ws_f, stream=stream, flags=flags)

    def fast_only_ragged():
        sfi.sfi_fast_decode_attn(shape, kv1, lay.compact, S, W, q, o, None, k_new=kn, v_new=vn, max_tokens=max_fast,
                                 workspace=ws_fr, stream=stream, flags=rflags)

    t1, t2, t2r = timed(one_launch), timed(two_launches), timed(two_launches_ragged)
    tf_even, tf_chunk = timed(fast_only_even), timed(fast_only_ragged)
    by_fast_only = sum(fast_bytes(1, Hq, Hkv, D, P, S + ks[r] + W, W) + append_bytes(1, Hkv, D) for r in range(B))
    by = 0
    for r in range(B):
        L = int(lens[r]) + 1
        if r in set(slow.tolist()):
            by += dense_bytes(1, Hq, Hkv, D, P, L, scores=True)
        else:
            by += fast_bytes(1, Hq, Hkv, D, P, S + ks[r] + W, W)
        by += append_bytes(1, Hkv, D)
    del lay
    torch.cuda.empty_cache()
    return {"workload": f"ragged {B} requests, kv 4K-128K log-uniform, 32q/8kv heads, retention {{3,12.5,25}}%",
            "slow_requests": int(n_slow), "total_kv_tokens": int(lens.sum()), "bytes": by,
            "one_launch_us": round(t1, 2), "one_launch_GBps": round(by / (t1 * 1e-6) / 1e9, 1),
            "one_launch_frac_of_peak": round(by / (t1 * 1e-6) / 1e9 / peak, 3),
            "two_launch_us": round(t2, 2), "two_launch_GBps": round(by / (t2 * 1e-6) / 1e9, 1),
            "two_launch_ragged_us": round(t2r, 2),
            "all_fast_bytes": by_fast_only,
            "all_fast_even_splits_us": round(tf_even, 2),
            "all_fast_ragged_us": round(tf_chunk, 2),
            "all_fast_ragged_frac_of_peak": round(by_fast_only / (tf_chunk * 1e-6) / 1e9 / peak, 3)}


# ---------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------
_SAMPLE = {}


def host_cpu():
    """(logical CPUs of this host, CPU model name) from os and /proc/cpuinfo."""
    model = "unknown"
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":", 1)[0].strip().lower()
                if key in ("model name", "cpu model", "hardware") and ":" in line:
                    model = line.split(":", 1)[1].strip()
                    break
        if model == "unknown":  # Arm hosts: no model name line; report the part number
            with open("/proc/cpuinfo") as f:
                parts = {line.split(":", 1)[1].strip() for line in f if line.lower().startswith("cpu part")}
            if parts:
                model = "Arm CPU part " + "/".join(sorted(parts))
    except OSError:
        pass
    return os.cpu_count() or 1, model


def oracle_sample_us_per_step(min_seconds: float, layers: int, batch: int, kv_len: int):
    """Time the CPU oracle on a bounded sample of the workload and scale it.

    Sample: one request, one layer, 2 of the 8 KV heads (4 of the 16 query heads; the
    heads are independent and cost the same), one refresh cycle's work: a slow step
    (dense attention + masked scores + Selector + compaction) and a fast step. Scaled
    by 4 for the heads, by batch x layers, and to a decode step as
    (slow + (cycle - 1) * fast) / cycle. Returns a dict with the scaled value, the
    measured sample times and the scale factor, so the figure can be reproduced."""
    import numpy as np
    import oracle
    import sfi_synth as syn

    Hq_all, Hkv_all = WL["num_q_heads"], WL["num_kv_heads"]
    Hq, Hkv, D, P = 4, 2, WL["head_dim"], WL["page_size"]
    S, W, cyc = WL["sink"], WL["recent"], WL["refresh_interval"]
    L0 = kv_len
    k = syn.retention_budget(WL["retention"], L0, S, W)
    key = (L0,)
    if key not in _SAMPLE:
        oracle.build()
        g = syn.rng(7000, 1)
        _SAMPLE[key] = (syn.make_paged_kv(g, [L0], Hkv, D, P), syn.normal_bf16(g, (Hq, D)))
    kvh, q = _SAMPLE[key]
    pr = kvh.page_table[0]
    t_slow, t_fast, n = 0.0, 0.0, 0
    t_begin = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        oracle.dense_attn(q, kvh.k_pool, kvh.v_pool, pr, L0, Hq, Hkv, D, P)
        sc = oracle.group_scores(q, kvh.k_pool, pr, L0, S, W, Hq, Hkv, D, P)
        idx = np.stack([oracle.select_topk(sc[h], L0, S, W, k) for h in range(Hkv)])
        ck, cv = oracle.compact(kvh.k_pool, kvh.v_pool, pr, L0, S, idx, k, Hkv, D, P, S + k)
        t1 = time.perf_counter()
        oracle.fast_attn(q, ck, cv, k, kvh.k_pool, kvh.v_pool, pr, L0, S, W, Hq, Hkv, D, P)
        t2 = time.perf_counter()
        t_slow += t1 - t0
        t_fast += t2 - t1
        n += 1
        if time.perf_counter() - t_begin >= min_seconds:
            break
    head_scale = Hkv_all / Hkv
    slow_s, fast_s = t_slow / n, t_fast / n
    sample_s = (slow_s + (cyc - 1) * fast_s) / cyc  # one decode step of the sample (1 request, 1 layer, 2 heads)
    factor = head_scale * batch * layers
    us_step = sample_s * factor * 1e6
    nproc, model = host_cpu()
    sample = (f"{n} x (one slow step: dense + scores + Selector + compaction, and one fast step) of one request, "
              f"one layer, {Hkv} of {Hkv_all} KV heads ({Hq} of {Hq_all} query heads), L={L0}; scaled x{head_scale:g} "
              f"heads x{batch} requests x{layers} layers, (slow + {cyc - 1} fast)/{cyc} per decode step")
    return {"value": us_step, "sample": sample, "wall_s": time.perf_counter() - t_begin,
            "sample_slow_step_s": round(slow_s, 6), "sample_fast_step_s": round(fast_s, 6),
            "sample_decode_step_us": round(sample_s * 1e6, 3), "extrapolation_factor": factor,
            "extrapolation": f"value = sample_decode_step_us x {factor:g} ({head_scale:g} heads x {batch} requests "
                             f"x {layers} layers)",
            "cores": 1, "host_cpus": nproc, "cpu_model": model,
            "cores_note": f"1 core used of {nproc} ({model}); the oracle is single-threaded"}


def cpu_baseline_entry(r, extra=""):
    return {"value": round(r["value"], 1), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": r["sample"] + extra, "host_cpus": r["host_cpus"], "cpu_model": r["cpu_model"],
            "cores_note": r["cores_note"], "sample_decode_step_us": r["sample_decode_step_us"],
            "sample_slow_step_s": r["sample_slow_step_s"], "sample_fast_step_s": r["sample_fast_step_s"],
            "extrapolation_factor": r["extrapolation_factor"], "extrapolation": r["extrapolation"]}


def run_reference(args, ranks: Ranks):
    if ranks.rank != 0:
        return None
    times = []
    last = None
    for _ in range(args.warmup):
        oracle_sample_us_per_step(0.0, args.layers, args.batch, args.kv_len)
    t_all = time.perf_counter()
    for _ in range(args.steps):
        last = oracle_sample_us_per_step(0.0, args.layers, args.batch, args.kv_len)
        times.append(last["value"])
    wall = time.perf_counter() - t_all
    us = statistics.mean(times)
    cpu = cpu_baseline_entry({**last, "value": us},
                             f"; one sample per step, {wall:.1f} s wall for {args.steps} steps")
    return {
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": UNIT, "n_gpus": ranks.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(wall / max(1, args.steps) * 1e3, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {**WL, "layers": args.layers, "batch": args.batch, "kv_len": args.kv_len,
                   "parallelism": "rank 0 only"},
        "timed_region_note": (f"one step of this arm is one bounded sample of the workload, timed on the host "
                              f"({wall:.1f} s of wall time for {args.steps} steps; ms_per_step is that wall time per "
                              f"step); value extrapolates the sample by {last['extrapolation_factor']:g} to the "
                              f"time of one full decode step"),
        "cpu_baseline": cpu,
        "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    ranks = Ranks()
    try:
        if args.impl == "reference":
            res = run_reference(args, ranks)
        else:
            res = run_gpu(args, ranks)
            if res is not None and ranks.rank == 0 and ranks.world == 1 and not args.no_cpu:
                r = oracle_sample_us_per_step(12.0, args.layers, args.batch, args.kv_len)
                res["cpu_baseline"] = cpu_baseline_entry(r, f"; {r['wall_s']:.1f} s of CPU time")
        if res is not None and ranks.rank == 0:
            print(json.dumps(res), flush=True)
    finally:
        ranks.close()


if __name__ == "__main__":
    main()
