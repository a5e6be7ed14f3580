// Split-KV decode attention for SFI on sm_103a (kernel template, included by the
// translation units that instantiate it): the fast step over the two-segment sparse
// state, the slow step's dense attention with masked group-summed logits, the dense
// full-KV baseline, and their multi-token forms (several query tokens per request:
// drafting over the sparse state, verification over the whole context).
//
// Method: Slow-Fast Inference (Xie et al., 2026), Figure 2 caption (fast steps over
// sink + selected + recent; slow steps run dense attention and collect masked
// logits over the candidate set) and Figure 3 caption (B) (sink + selected packed
// in a contiguous compact buffer, recent tokens read in place from paged KV). The
// multi-token forms follow "A Sparse Glimpse of the Whole: Train-Free Self-Speculative
// Decoding", abstract (drafts from the sparse, recallable KV state; full-context
// verification whose per-head statistics are recycled as the importance signal).
//
// Design (HBM-bound: every K/V byte is read once per step):
//  * Grid (split, KV head, request), two CTAs per SM. A (request, KV head) unit's
//    token stream is cut into 16-token sub-blocks: compact rows first (fast mode),
//    then the pages of the recent window (fast) or of [0, L) (dense). Split c owns a
//    contiguous range of sub-blocks.
//  * One producer warp issues TMA tensor loads (2-D tiled, 128-byte swizzle, L2
//    evict-first) of K and V sub-blocks into a 96 KB ring of shared-memory stages;
//    completion is tracked by mbarriers (transaction bytes). Page ids are fetched a
//    chunk of 32 sub-blocks ahead by the whole producer warp.
//  * Four consumer warps each own one sub-block per stage. QK^T and PV run on the
//    tensor cores with mma.sync m16n8k16 (bf16 in, fp32 accumulate): the G <= 8
//    query rows of the KV head form the M = 16 tile, so K and V never pass through
//    CUDA-core unpacking. Online softmax in fp32 on the C fragments. The multi-token
//    form (MQ) fills all 16 rows with T tokens x G heads (row = t * G + g), each row
//    with its own causal / window bounds, at the same number of mma instructions.
//  * The slow step sums the C fragments over the group's rows with warp shuffles and
//    writes the fp32 masked scores.
//  * With k_new/v_new the consumer warp owning position L - 1 (the positions of the T
//    query tokens, multi-token form) stages the new K/V in shared memory before the
//    stream, writes it to the page early in the stream and into its tile when the
//    sub-block arrives (the append fused into the attention).
//  * Warps merge through shared memory in two passes (per-row weights, then 4-float
//    chunks). Splits of a unit merge in-kernel: with up to 8 splits the unit's CTAs
//    form one thread-block cluster and the other ranks store their partial (m, l, o)
//    states into rank 0's shared memory with asynchronous stores that complete on rank
//    0's mbarrier (one partial per warp, without their own warp merge, when those fit;
//    rank 0 reads them through distributed shared memory when even one per CTA does
//    not fit); with more, the last CTA of the unit (atomic
//    counter, self-resetting) merges them from a global workspace.
//  * Every wait on the pipeline or on a peer CTA is bounded and reports
//    SFI_DEV_TIMEOUT instead of hanging.
#pragma once

#include <atomic>

#include "sfi_device.cuh"
#include "sfi_internal.h"

namespace sfi {

template <int D>
struct AttnTile {
    static constexpr int kBoxes = D / 64;                        // 128-byte boxes per row
    static constexpr int kSubBytes = kSubTokens * D * 2;         // K (or V) of one sub-block
    static constexpr int kStageBytes = kConsumerWarps * 2 * kSubBytes;
    static constexpr int kRingBytes = 96 * 1024;                 // two CTAs per SM
    static constexpr int kStages = kRingBytes / kStageBytes;
    // After the ring: where the other CTAs of a cluster push their partial results.
    static constexpr int kRecvOffset = kStages * kStageBytes;
    static constexpr int kRecvBytes = 13 * 1024;
    // Multi-token kernels keep the 16-row query tile in the last kQBytes of the receive
    // region (128-byte rows swizzled in 16-byte chunks), out of reach of the pushes.
    static constexpr int kQBytes = kMaxRows * D * 2;
    static constexpr int kSmemBytes = kRecvOffset + kRecvBytes + 1024;  // + alignment slack
    static constexpr int kKSteps = D / 16;                       // mma k-steps of QK^T
    static constexpr int kNTiles = D / 8;                        // mma n-tiles of PV
    static constexpr int kMergeStride = D + 4;                   // padded rows of the warp-merge scratch
};

constexpr int kAttnThreads = (kConsumerWarps + 1) * 32;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ void consumer_bar_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// Barrier over the consumer threads that also returns whether any of them passed true.
__device__ __forceinline__ bool consumer_bar_or(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, 1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(kConsumerWarps * 32)
        : "memory");
    return r != 0;
}

// Whether any page id of positions [0, L) of request r lies outside the pool, checked by
// every consumer thread before the first score write of a unit, so a unit with a bad
// page writes none of its scores (the pages are checked again as they are streamed).
// In two parts: pages_first issues this thread's first eight loads (the first 1024
// pages), which can happen before the grid dependency wait; pages_bad finishes the
// check (the rest of the pages, then a barrier reduction over the consumer threads).
constexpr int kPageCheckLoads = 8;
__device__ __forceinline__ void pages_first(const AttnParams &p, int r, int L, int (&pg)[kPageCheckLoads]) {
    const int32_t *ptab = p.page_table + (int64_t)r * p.max_pages;
    const int npg = (L + kSubTokens - 1) / kSubTokens;
#pragma unroll
    for (int j = 0; j < kPageCheckLoads; ++j) {
        const int i = threadIdx.x + j * kConsumerWarps * 32;
        pg[j] = i < npg ? __ldg(ptab + i) : 0;
    }
}
__device__ __forceinline__ bool pages_bad(const AttnParams &p, int r, int L, const int (&first)[kPageCheckLoads]) {
    const int32_t *ptab = p.page_table + (int64_t)r * p.max_pages;
    const int npg = (L + kSubTokens - 1) / kSubTokens;
    bool bad = false;
#pragma unroll
    for (int j = 0; j < kPageCheckLoads; ++j) bad |= first[j] < 0 || first[j] >= p.num_pages;
    for (int i0 = threadIdx.x + kPageCheckLoads * kConsumerWarps * 32; i0 < npg;
         i0 += kPageCheckLoads * kConsumerWarps * 32) {
        int pg[kPageCheckLoads];
#pragma unroll
        for (int j = 0; j < kPageCheckLoads; ++j) {  // eight independent loads in flight
            const int i = i0 + j * kConsumerWarps * 32;
            pg[j] = i < npg ? __ldg(ptab + i) : 0;
        }
#pragma unroll
        for (int j = 0; j < kPageCheckLoads; ++j) bad |= pg[j] < 0 || pg[j] >= p.num_pages;
    }
    return consumer_bar_or(bad);
}

// Geometry of one (request, KV head) unit's token stream.
struct UnitStream {
    int L;         // current length (all query tokens appended)
    int L0;        // length seen by the first query token: L - tokens + 1
    int cnt;       // selected rows in the compact buffer (fast mode)
    int n1;        // compact rows streamed (fast mode)
    int nb1;       // compact sub-blocks (fast mode)
    int page0;     // first page of the paged segment
    int lo_pos;    // first valid position of the paged segment
    int nb;        // total sub-blocks
    int64_t crow0; // first compact row of this KV head (fast mode)
    int sb_app;    // sub-block holding position L - 1 (the current token)
    int row_app;   // its row inside that sub-block
};

// `lead` marks one CTA per request, which reports the request's errors.
__device__ __forceinline__ bool unit_stream(const AttnParams &p, int r, int kvh, bool fast, bool lead,
                                            UnitStream &u) {
    // All per-request metadata is loaded up front, in one round trip.
    u.L = p.seq_lens[r];
    u.L0 = u.L - p.tokens + 1;
    const int cnt = fast ? p.c_count[r] : 0;
    u.cnt = cnt;
    const int cap = fast ? p.c_capacity[r] : 0;
    const int64_t off = fast ? p.c_row_offset[r] : 0;
    lead = lead && threadIdx.x == 0 && kvh == 0;
    if (u.L0 < 1 || u.L > p.max_pages * kSubTokens) {
        if (lead) report(p.dev_status, SFI_DEV_BAD_LEN);
        return false;
    }
    if (fast) {
        const int ns = min(p.sink, u.L);
        if (cnt < 0 || cnt > cap - p.sink || (cnt > 0 && u.L0 < p.sink)) {
            if (lead) report(p.dev_status, SFI_DEV_K_OVERFLOW);
            return false;
        }
        if (off < 0 || off + (int64_t)p.hkv * cap > p.c_total_rows) {
            if (lead) report(p.dev_status, SFI_DEV_BAD_COMPACT);
            return false;
        }
        u.crow0 = off + (int64_t)kvh * cap;
        u.n1 = ns + cnt;
        u.nb1 = (u.n1 + kSubTokens - 1) / kSubTokens;
        const int rs = max(p.sink, u.L0 - p.recent);  // the first token's window starts lowest
        if (rs < u.L) {
            u.lo_pos = rs;
            u.page0 = rs / kSubTokens;
            u.nb = u.nb1 + ((u.L - 1) / kSubTokens - u.page0 + 1);
            u.sb_app = u.nb1 + ((u.L - 1) / kSubTokens - u.page0);  // last page of the recent window
        } else {
            u.lo_pos = u.L;
            u.page0 = 0;
            u.nb = u.nb1;
            u.sb_app = (u.L - 1) / kSubTokens;  // L <= S: the current token is a sink row
        }
    } else {
        u.crow0 = 0;
        u.n1 = 0;
        u.nb1 = 0;
        u.lo_pos = 0;
        u.page0 = 0;
        u.nb = (u.L + kSubTokens - 1) / kSubTokens;
        u.sb_app = u.nb - 1;
    }
    u.row_app = (u.L - 1) % kSubTokens;
    return true;
}

// Process one 16-token sub-block held in shared memory (K at kaddr, V at vaddr,
// each kBoxes boxes of [16 rows][128 B] with the 128-byte swizzle).
// The G <= 8 query rows sit in rows 0-7 of the M = 16 tile. In PV, rows 8-15 of the A
// fragment carry the low bf16 part of the same probabilities, so o[nt][0..1] (rows g)
// accumulate P_hi V and o[nt][2..3] (rows g + 8) P_lo V; the caller adds the halves.
template <int D, bool SCORES>
__device__ __forceinline__ void consume_sub_block(uint32_t kaddr, uint32_t vaddr, int lo, int hi, int pos0,
                                                  const uint32_t (&qa)[D / 16][2], float (&o)[D / 8][4],
                                                  float &m_run, float &l_run, const AttnParams &p, float *score_row,
                                                  int L, int lane) {
    using T = AttnTile<D>;
    const int g = lane >> 2, t = lane & 3;
    const int mi = lane >> 3, r8 = lane & 7;

    // S = Q K^T for 16 tokens: two n-tiles (tokens 0-7 and 8-15), one accumulation chain
    // each. (Splitting each into even and odd k-steps was measured: no change, and it
    // made the kernel spill.)
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
        const int tok = ((mi >> 1) << 3) + r8;
        const uint32_t row_addr = kaddr + tok * 128;
#pragma unroll
        for (int ks = 0; ks < T::kKSteps; ++ks) {
            const int box = ks >> 2;
            const int chunk = ((ks & 3) << 1) + (mi & 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(row_addr + box * (kSubTokens * 128) + ((chunk ^ r8) << 4), b0, b1, b2, b3);
            mma_bf16_16816(s[0], qa[ks][0], 0u, qa[ks][1], 0u, b0, b1);
            mma_bf16_16816(s[1], qa[ks][0], 0u, qa[ks][1], 0u, b2, b3);
        }
    }
    const int tk0 = 2 * t, tk1 = 2 * t + 1, tk2 = 8 + 2 * t, tk3 = 9 + 2 * t;

    if (SCORES) {
        // Group sum over the 8 query rows (rows >= G hold zero queries, so they add 0).
        float v0 = s[0][0], v1 = s[0][1], v2 = s[1][0], v3 = s[1][1];
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            v0 += __shfl_xor_sync(0xffffffffu, v0, off);
            v1 += __shfl_xor_sync(0xffffffffu, v1, off);
            v2 += __shfl_xor_sync(0xffffffffu, v2, off);
            v3 += __shfl_xor_sync(0xffffffffu, v3, off);
        }
        // Every lane of a column group holds the sums now; lanes g < 4 store one token each,
        // so the sub-block's 16 scores leave in one coalesced 64-byte store.
        if (g < 4 && score_row != nullptr) {
            const int c_lo = p.sink, c_hi = L - p.recent;
            const float vg = (g & 2) ? ((g & 1) ? v3 : v2) : ((g & 1) ? v1 : v0);
            const int pos = pos0 + (g >> 1) * 8 + 2 * t + (g & 1);  // tk0 .. tk3
            if (pos < L) score_row[pos] = (pos >= c_lo && pos < c_hi) ? vg * p.scale : -INFINITY;
        }
    }

    const bool full = (lo == 0 && hi == kSubTokens);
    float x0 = s[0][0] * p.scale_log2, x1 = s[0][1] * p.scale_log2;
    float x2 = s[1][0] * p.scale_log2, x3 = s[1][1] * p.scale_log2;
    uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
    if (!full) {
        const bool ok0 = tk0 >= lo && tk0 < hi, ok1 = tk1 >= lo && tk1 < hi;
        const bool ok2 = tk2 >= lo && tk2 < hi, ok3 = tk3 >= lo && tk3 < hi;
        x0 = ok0 ? x0 : -INFINITY;
        x1 = ok1 ? x1 : -INFINITY;
        x2 = ok2 ? x2 : -INFINITY;
        x3 = ok3 ? x3 : -INFINITY;
        // V rows of masked tokens may hold anything (even NaN): zero them in the B fragments.
        vm0 = (ok0 ? 0x0000ffffu : 0u) | (ok1 ? 0xffff0000u : 0u);
        vm1 = (ok2 ? 0x0000ffffu : 0u) | (ok3 ? 0xffff0000u : 0u);
    }
    float mt = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
    const float m_new = fmaxf(m_run, mt);
    const float base = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = fast_exp2(m_run - base);
    const float p0 = fast_exp2(x0 - base), p1 = fast_exp2(x1 - base);
    const float p2 = fast_exp2(x2 - base), p3 = fast_exp2(x3 - base);
    l_run = l_run * alpha + ((p0 + p1) + (p2 + p3));
    m_run = m_new;
    if (__any_sync(0xffffffffu, alpha != 1.f)) {  // the running max moved for some row
#pragma unroll
        for (int nt = 0; nt < T::kNTiles; ++nt) {
            o[nt][0] *= alpha;
            o[nt][1] *= alpha;
            o[nt][2] *= alpha;
            o[nt][3] *= alpha;
        }
    }
    // P enters the PV product as two bf16 terms, hi = bf16(p) and lo = bf16(p - hi), so
    // the weights carry about 16 significant bits instead of bf16's 8; hi fills the A
    // fragment's rows 0-7, lo its rows 8-15.
    const __nv_bfloat162 h01 = __floats2bfloat162_rn(p0, p1);
    const __nv_bfloat162 h23 = __floats2bfloat162_rn(p2, p3);
    const __nv_bfloat162 l01 = __floats2bfloat162_rn(p0 - __low2float(h01), p1 - __high2float(h01));
    const __nv_bfloat162 l23 = __floats2bfloat162_rn(p2 - __low2float(h23), p3 - __high2float(h23));
    const uint32_t pa0 = *reinterpret_cast<const uint32_t *>(&h01);
    const uint32_t pa2 = *reinterpret_cast<const uint32_t *>(&h23);
    const uint32_t pl0 = *reinterpret_cast<const uint32_t *>(&l01);
    const uint32_t pl2 = *reinterpret_cast<const uint32_t *>(&l23);

    // O += P V: V sub-block as the B operand via ldmatrix.trans.
    {
        const int tok = ((mi & 1) << 3) + r8;
        const uint32_t row_addr = vaddr + tok * 128;
#pragma unroll
        for (int j = 0; j < T::kNTiles / 2; ++j) {
            const int box = j >> 2;
            const int chunk = ((j & 3) << 1) + (mi >> 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_trans(row_addr + box * (kSubTokens * 128) + ((chunk ^ r8) << 4), b0, b1, b2, b3);
            if (!full) {
                b0 &= vm0;
                b1 &= vm1;
                b2 &= vm0;
                b3 &= vm1;
            }
            mma_bf16_16816(o[2 * j], pa0, pl0, pa2, pl2, b0, b1);
            mma_bf16_16816(o[2 * j + 1], pa0, pl0, pa2, pl2, b2, b3);
        }
    }
}

// Multi-token form of the fused append: the query tokens at positions [L - T, L) that
// fall in this paged sub-block (positions [pos0, pos0 + 16)) replace their rows of the
// tile and are written to the page (k_new/v_new: [request][T][Hkv][D]).
template <int D>
__device__ __forceinline__ void fuse_tokens(uint8_t *tile, const AttnParams &p, int r, int kvh, int L, int pos0,
                                            int lane, int *s_bad) {
    using T = AttnTile<D>;
    constexpr int kChunks = D / 8;
    const int ntok = p.tokens;
    const int first = max(L - ntok, pos0), last = min(L, pos0 + kSubTokens);
    const int page = p.page_table[(int64_t)r * p.max_pages + pos0 / kSubTokens];
    const bool page_ok = page >= 0 && page < p.num_pages;
    if (lane < 2 * kChunks) {
        const bool is_v = lane >= kChunks;
        const int c = is_v ? lane - kChunks : lane;
        const __nv_bfloat16 *src0 = (is_v ? p.v_new : p.k_new) + (int64_t)kvh * D + c * 8;
        __nv_bfloat16 *dst0 = (is_v ? p.v_pool_w : p.k_pool_w) + ((int64_t)page * p.hkv + kvh) * kSubTokens * D + c * 8;
        uint8_t *base0 = tile + (is_v ? T::kSubBytes : 0) + (c >> 3) * (kSubTokens * 128);
        // up to 8 tokens per round, every load of a round issued before its stores
        for (int pos8 = first; pos8 < last; pos8 += 8) {
            int4 val[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int tok = pos8 + j - (L - ntok);
                if (pos8 + j < last)
                    val[j] = *reinterpret_cast<const int4 *>(src0 + ((int64_t)r * ntok + tok) * p.hkv * D);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int row = pos8 + j - pos0;
                if (pos8 + j < last) {
                    *reinterpret_cast<int4 *>(base0 + row * 128 + (((c & 7) ^ (row & 7)) << 4)) = val[j];
                    if (page_ok) *reinterpret_cast<int4 *>(dst0 + (int64_t)row * D) = val[j];
                }
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (!page_ok && lane == 0) {
        report(p.dev_status, SFI_DEV_BAD_PAGE);
        *s_bad = 1;  // the unit writes no output
    }
    __syncwarp();
}

// Bounds [lo, hi) of the tokens of a 16-token sub-block that one query row sees.
struct RowSpan {
    int lo, hi;
};

// Multi-token form of consume_sub_block: all 16 rows of the tile are query rows; this
// lane holds rows g (span ra) and g + 8 (span rb). `full` (warp-uniform) says every
// row sees all 16 tokens; [lo, hi) is the union of the rows' spans.
template <int D, bool SCORES>
__device__ __forceinline__ void consume_sub_block_mq(uint32_t kaddr, uint32_t vaddr, int lo, int hi, bool full,
                                                     RowSpan ra, RowSpan rb, int pos0, uint32_t qtile,
                                                     float (&o)[D / 8][4],
                                                     float (&m_run)[2], float (&l_run)[2], const AttnParams &p,
                                                     float *score_row, int L, int lane) {
    using T = AttnTile<D>;
    const int g = lane >> 2, t = lane & 3;
    const int mi = lane >> 3, r8 = lane & 7;

    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
        const int tok = ((mi >> 1) << 3) + r8;
        const uint32_t row_addr = kaddr + tok * 128;
        // A fragments from the query tile: lane l addresses row (l & 7) + 8 * ((l >> 3) & 1)
        // and the k-half l >> 4 of each 16-column step
        const int qr = r8 + ((mi & 1) << 3);
        const uint32_t qrow_addr = qtile + qr * (D * 2);
#pragma unroll
        for (int ks = 0; ks < T::kKSteps; ++ks) {
            const int box = ks >> 2;
            const int chunk = ((ks & 3) << 1) + (mi & 1);
            uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
            ldsm_x4(qrow_addr + (((2 * ks + (mi >> 1)) ^ r8) << 4), a0, a1, a2, a3);
            ldsm_x4(row_addr + box * (kSubTokens * 128) + ((chunk ^ r8) << 4), b0, b1, b2, b3);
            mma_bf16_16816(s[0], a0, a1, a2, a3, b0, b1);
            mma_bf16_16816(s[1], a0, a1, a2, a3, b2, b3);
        }
    }
    // this lane's tokens, and its elements of rows g (xa) and g + 8 (xb)
    const int tk[4] = {2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t};
    float xa[4] = {s[0][0], s[0][1], s[1][0], s[1][1]};
    float xb[4] = {s[0][2], s[0][3], s[1][2], s[1][3]};
    bool oka[4], okb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        oka[i] = full || (tk[i] >= ra.lo && tk[i] < ra.hi);
        okb[i] = full || (tk[i] >= rb.lo && tk[i] < rb.hi);
    }

    if (SCORES) {
        // Sum over every (token, head) row that sees the position (padding rows hold
        // zero queries and add 0).
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = (oka[i] ? xa[i] : 0.f) + (okb[i] ? xb[i] : 0.f);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], off);
        }
        // one token per lane g < 4 (every lane of a column group holds the sums)
        if (g < 4 && score_row != nullptr) {
            const int c_lo = p.sink, c_hi = L - p.recent;
            const float vg = (g & 2) ? ((g & 1) ? v[3] : v[2]) : ((g & 1) ? v[1] : v[0]);
            const int pos = pos0 + (g >> 1) * 8 + 2 * t + (g & 1);  // tk[g]
            if (pos < L) score_row[pos] = (pos >= c_lo && pos < c_hi) ? vg * p.scale : -INFINITY;
        }
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        xa[i] = oka[i] ? xa[i] * p.scale_log2 : -INFINITY;
        xb[i] = okb[i] ? xb[i] * p.scale_log2 : -INFINITY;
    }
    uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
    if (!full) {
        // V rows outside every row's span may hold anything (even NaN): zero them.
        const bool u0 = tk[0] >= lo && tk[0] < hi, u1 = tk[1] >= lo && tk[1] < hi;
        const bool u2 = tk[2] >= lo && tk[2] < hi, u3 = tk[3] >= lo && tk[3] < hi;
        vm0 = (u0 ? 0x0000ffffu : 0u) | (u1 ? 0xffff0000u : 0u);
        vm1 = (u2 ? 0x0000ffffu : 0u) | (u3 ? 0xffff0000u : 0u);
    }
    if (p.rows <= kMaxGroup) {
        // At most 8 query rows: rows g + 8 of the tile are padding, so (as in the one-token
        // consume_sub_block) they carry the low bf16 half of row g's probabilities and one
        // mma per n-tile computes both halves; the caller adds o[.][0..1] and o[.][2..3].
        float ma = fmaxf(fmaxf(xa[0], xa[1]), fmaxf(xa[2], xa[3]));
        ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
        ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 2));
        const float na = fmaxf(m_run[0], ma);
        const float ba = (na == -INFINITY) ? 0.f : na;
        const float alpha = fast_exp2(m_run[0] - ba);
        float pa[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) pa[i] = fast_exp2(xa[i] - ba);
        l_run[0] = l_run[0] * alpha + ((pa[0] + pa[1]) + (pa[2] + pa[3]));
        m_run[0] = na;
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
            for (int nt = 0; nt < T::kNTiles; ++nt) {
                o[nt][0] *= alpha;
                o[nt][1] *= alpha;
                o[nt][2] *= alpha;
                o[nt][3] *= alpha;
            }
        }
        const __nv_bfloat162 h01 = __floats2bfloat162_rn(pa[0], pa[1]);
        const __nv_bfloat162 h23 = __floats2bfloat162_rn(pa[2], pa[3]);
        const __nv_bfloat162 l01 = __floats2bfloat162_rn(pa[0] - __low2float(h01), pa[1] - __high2float(h01));
        const __nv_bfloat162 l23 = __floats2bfloat162_rn(pa[2] - __low2float(h23), pa[3] - __high2float(h23));
        const uint32_t a0 = *reinterpret_cast<const uint32_t *>(&h01);
        const uint32_t a1 = *reinterpret_cast<const uint32_t *>(&l01);
        const uint32_t a2 = *reinterpret_cast<const uint32_t *>(&h23);
        const uint32_t a3 = *reinterpret_cast<const uint32_t *>(&l23);
        const int tok = ((mi & 1) << 3) + r8;
        const uint32_t row_addr = vaddr + tok * 128;
#pragma unroll
        for (int j = 0; j < T::kNTiles / 2; ++j) {
            const int box = j >> 2;
            const int chunk = ((j & 3) << 1) + (mi >> 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_trans(row_addr + box * (kSubTokens * 128) + ((chunk ^ r8) << 4), b0, b1, b2, b3);
            if (!full) {
                b0 &= vm0;
                b1 &= vm1;
                b2 &= vm0;
                b3 &= vm1;
            }
            mma_bf16_16816(o[2 * j], a0, a1, a2, a3, b0, b1);
            mma_bf16_16816(o[2 * j + 1], a0, a1, a2, a3, b2, b3);
        }
        return;
    }
    float ma = fmaxf(fmaxf(xa[0], xa[1]), fmaxf(xa[2], xa[3]));
    float mb = fmaxf(fmaxf(xb[0], xb[1]), fmaxf(xb[2], xb[3]));
    ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
    ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 2));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
    const float na = fmaxf(m_run[0], ma), nb = fmaxf(m_run[1], mb);
    const float ba = (na == -INFINITY) ? 0.f : na, bb = (nb == -INFINITY) ? 0.f : nb;
    const float alpha_a = fast_exp2(m_run[0] - ba), alpha_b = fast_exp2(m_run[1] - bb);
    float pa[4], pb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        pa[i] = fast_exp2(xa[i] - ba);
        pb[i] = fast_exp2(xb[i] - bb);
    }
    l_run[0] = l_run[0] * alpha_a + ((pa[0] + pa[1]) + (pa[2] + pa[3]));
    l_run[1] = l_run[1] * alpha_b + ((pb[0] + pb[1]) + (pb[2] + pb[3]));
    m_run[0] = na;
    m_run[1] = nb;
    if (__any_sync(0xffffffffu, alpha_a != 1.f || alpha_b != 1.f)) {  // some row's running max moved
#pragma unroll
        for (int nt = 0; nt < T::kNTiles; ++nt) {
            o[nt][0] *= alpha_a;
            o[nt][1] *= alpha_a;
            o[nt][2] *= alpha_b;
            o[nt][3] *= alpha_b;
        }
    }
    // P as two bf16 terms (hi + lo), rows g and g + 8 in the A fragment's halves.
    uint32_t ph[4], pl[4];
    {
        const __nv_bfloat162 ha01 = __floats2bfloat162_rn(pa[0], pa[1]);
        const __nv_bfloat162 hb01 = __floats2bfloat162_rn(pb[0], pb[1]);
        const __nv_bfloat162 ha23 = __floats2bfloat162_rn(pa[2], pa[3]);
        const __nv_bfloat162 hb23 = __floats2bfloat162_rn(pb[2], pb[3]);
        const __nv_bfloat162 la01 = __floats2bfloat162_rn(pa[0] - __low2float(ha01), pa[1] - __high2float(ha01));
        const __nv_bfloat162 lb01 = __floats2bfloat162_rn(pb[0] - __low2float(hb01), pb[1] - __high2float(hb01));
        const __nv_bfloat162 la23 = __floats2bfloat162_rn(pa[2] - __low2float(ha23), pa[3] - __high2float(ha23));
        const __nv_bfloat162 lb23 = __floats2bfloat162_rn(pb[2] - __low2float(hb23), pb[3] - __high2float(hb23));
        ph[0] = *reinterpret_cast<const uint32_t *>(&ha01);
        ph[1] = *reinterpret_cast<const uint32_t *>(&hb01);
        ph[2] = *reinterpret_cast<const uint32_t *>(&ha23);
        ph[3] = *reinterpret_cast<const uint32_t *>(&hb23);
        pl[0] = *reinterpret_cast<const uint32_t *>(&la01);
        pl[1] = *reinterpret_cast<const uint32_t *>(&lb01);
        pl[2] = *reinterpret_cast<const uint32_t *>(&la23);
        pl[3] = *reinterpret_cast<const uint32_t *>(&lb23);
    }
    {
        const int tok = ((mi & 1) << 3) + r8;
        const uint32_t row_addr = vaddr + tok * 128;
#pragma unroll
        for (int j = 0; j < T::kNTiles / 2; ++j) {
            const int box = j >> 2;
            const int chunk = ((j & 3) << 1) + (mi >> 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_trans(row_addr + box * (kSubTokens * 128) + ((chunk ^ r8) << 4), b0, b1, b2, b3);
            if (!full) {
                b0 &= vm0;
                b1 &= vm1;
                b2 &= vm0;
                b3 &= vm1;
            }
            mma_bf16_16816(o[2 * j], ph[0], ph[1], ph[2], ph[3], b0, b1);
            mma_bf16_16816(o[2 * j + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
            mma_bf16_16816(o[2 * j], pl[0], pl[1], pl[2], pl[3], b0, b1);
            mma_bf16_16816(o[2 * j + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
        }
    }
}

// Fused append of the current token (k_new/v_new of this KV head, position L - 1), in
// three steps by the warp that owns its sub-block: stage_current_token starts
// asynchronous copies of the token's K/V chunks and its page id into shared memory
// before the stream; store_current_token writes them to the page early in the stream;
// fuse_current_token puts them into the sub-block's tile when it arrives.
template <int D>
__device__ __forceinline__ void stage_current_token(const AttnParams &p, int r, int kvh, const UnitStream &u,
                                                    int lane, int4 *s_val, int *s_page) {
    constexpr int kChunks = D / 8;
    if (lane < 2 * kChunks) {
        const bool is_v = lane >= kChunks;
        const int c = is_v ? lane - kChunks : lane;
        const __nv_bfloat16 *src = (is_v ? p.v_new : p.k_new) + ((int64_t)r * p.hkv + kvh) * D + c * 8;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(smem_u32(&s_val[lane])), "l"(src)
                     : "memory");
    }
    if (lane == 0) {
        const int32_t *src = p.page_table + (int64_t)r * p.max_pages + (u.L - 1) / kSubTokens;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(s_page)), "l"(src) : "memory");
    }
}

// Write the staged current token's K/V into the paged cache at position L - 1: done by
// the warp that owns the token's sub-block early in the stream, so the writes drain
// during the stream instead of at its end. A bad page id is reported and makes the
// unit write no output.
template <int D>
__device__ __forceinline__ void store_current_token(const AttnParams &p, int kvh, const UnitStream &u, int lane,
                                                    const int4 *s_val, const int *s_page, int *s_bad) {
    constexpr int kChunks = D / 8;
    // the copies issued by stage_current_token have landed (each lane waits for its own)
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();
    const int page = *s_page;
    if (page < 0 || page >= p.num_pages) {
        if (lane == 0) {
            report(p.dev_status, SFI_DEV_BAD_PAGE);
            *s_bad = 1;  // the unit writes no output
        }
    } else if (lane < 2 * kChunks) {
        const bool is_v = lane >= kChunks;
        const int c = is_v ? lane - kChunks : lane;
        const int pos = u.L - 1;
        __nv_bfloat16 *dst = (is_v ? p.v_pool_w : p.k_pool_w) +
                             (((int64_t)page * p.hkv + kvh) * kSubTokens + pos % kSubTokens) * D + c * 8;
        *reinterpret_cast<int4 *>(dst) = s_val[lane];
    }
}

// The staged current token's K/V replace row u.row_app of the swizzled K and V tiles at
// `tile` (the attention sees the cache after the append). One 16-byte chunk per lane;
// the writing lanes then order their generic-proxy shared-memory writes before later
// TMA (async-proxy) writes into the same stage.
template <int D>
__device__ __forceinline__ void fuse_current_token(uint8_t *tile, const UnitStream &u, int lane, const int4 *s_val) {
    using T = AttnTile<D>;
    constexpr int kChunks = D / 8;
    if (lane < 2 * kChunks) {
        const bool is_v = lane >= kChunks;
        const int c = is_v ? lane - kChunks : lane;
        const int row = u.row_app;
        uint8_t *base = tile + (is_v ? T::kSubBytes : 0) + (c >> 3) * (kSubTokens * 128) + row * 128;
        *reinterpret_cast<int4 *>(base + (((c & 7) ^ (row & 7)) << 4)) = s_val[lane];
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncwarp();
}

// Multi-token form of stage_current_token: the K/V rows of the query tokens that fall in
// the paged sub-block starting at position pos0 (k_new/v_new: [request][T][Hkv][D]) are
// copied asynchronously into `stage` (token i = position L - T + i at i * 4D bytes: its
// K row, then its V row), and the page id into *s_page.
template <int D>
__device__ __forceinline__ void stage_tokens(const AttnParams &p, int r, int kvh, int L, int pos0, int lane,
                                             uint8_t *stage, int *s_page) {
    constexpr int kChunks = D / 8;
    const int ntok = p.tokens;
    const int first = max(L - ntok, pos0), last = min(L, pos0 + kSubTokens);
    if (lane < 2 * kChunks) {
        const bool is_v = lane >= kChunks;
        const int c = is_v ? lane - kChunks : lane;
        const __nv_bfloat16 *src0 = (is_v ? p.v_new : p.k_new) + (int64_t)kvh * D + c * 8;
        for (int pos = first; pos < last; ++pos) {
            const int tok = pos - (L - ntok);
            const __nv_bfloat16 *src = src0 + ((int64_t)r * ntok + tok) * p.hkv * D;
            uint8_t *dst = stage + tok * (4 * D) + (is_v ? 2 * D : 0) + c * 16;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
        }
    }
    if (lane == 0) {
        const int32_t *src = p.page_table + (int64_t)r * p.max_pages + pos0 / kSubTokens;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(s_page)), "l"(src) : "memory");
    }
}

// Write the staged query tokens of the sub-block at pos0 into the paged cache (early in
// the stream, like store_current_token).
template <int D>
__device__ __forceinline__ void store_tokens(const AttnParams &p, int kvh, int L, int pos0, int lane,
                                             const uint8_t *stage, const int *s_page, int *s_bad) {
    constexpr int kChunks = D / 8;
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();
    const int ntok = p.tokens;
    const int first = max(L - ntok, pos0), last = min(L, pos0 + kSubTokens);
    const int page = *s_page;
    if (page < 0 || page >= p.num_pages) {
        if (lane == 0) {
            report(p.dev_status, SFI_DEV_BAD_PAGE);
            *s_bad = 1;  // the unit writes no output
        }
    } else if (lane < 2 * kChunks) {
        const bool is_v = lane >= kChunks;
        const int c = is_v ? lane - kChunks : lane;
        __nv_bfloat16 *dst0 = (is_v ? p.v_pool_w : p.k_pool_w) + ((int64_t)page * p.hkv + kvh) * kSubTokens * D + c * 8;
        for (int pos = first; pos < last; ++pos) {
            const int tok = pos - (L - ntok);
            *reinterpret_cast<int4 *>(dst0 + (int64_t)(pos - pos0) * D) =
                *reinterpret_cast<const int4 *>(stage + tok * (4 * D) + (is_v ? 2 * D : 0) + c * 16);
        }
    }
}

// The staged query tokens replace their rows of the swizzled K and V tiles at `tile`.
template <int D>
__device__ __forceinline__ void fuse_staged_tokens(uint8_t *tile, const AttnParams &p, int L, int pos0, int lane,
                                                   const uint8_t *stage) {
    using T = AttnTile<D>;
    constexpr int kChunks = D / 8;
    const int ntok = p.tokens;
    const int first = max(L - ntok, pos0), last = min(L, pos0 + kSubTokens);
    if (lane < 2 * kChunks) {
        const bool is_v = lane >= kChunks;
        const int c = is_v ? lane - kChunks : lane;
        uint8_t *base0 = tile + (is_v ? T::kSubBytes : 0) + (c >> 3) * (kSubTokens * 128);
        for (int pos = first; pos < last; ++pos) {
            const int tok = pos - (L - ntok), row = pos - pos0;
            *reinterpret_cast<int4 *>(base0 + row * 128 + (((c & 7) ^ (row & 7)) << 4)) =
                *reinterpret_cast<const int4 *>(stage + tok * (4 * D) + (is_v ? 2 * D : 0) + c * 16);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncwarp();
}

// Four consecutive output floats; the output is only 8-byte aligned (by contract), so two
// 8-byte stores.
__device__ __forceinline__ void store_out4(float *dst, float4 v) {
    *reinterpret_cast<float2 *>(dst) = make_float2(v.x, v.y);
    *reinterpret_cast<float2 *>(dst + 2) = make_float2(v.z, v.w);
}

// Floats of one pushed partial in the receive region: o [rows][D], m [rows], l [rows],
// padded to 16 bytes.
template <int D>
__host__ __device__ constexpr int cluster_slot_floats(int rows) {
    return (rows * (D + 2) + 3) & ~3;
}

// Whether the partials of `splits` CTAs with `rows` query rows fit rank 0's receive region.
template <int D>
__host__ __device__ constexpr bool cluster_push_fits(int splits, int rows, int recv_bytes = AttnTile<D>::kRecvBytes) {
    return (splits - 1) * cluster_slot_floats<D>(rows) * 4 <= recv_bytes;
}

// Whether the other CTAs' per-warp partials (one slot per consumer warp) fit rank 0's
// receive region: then those CTAs skip their own warp merge.
template <int D>
__host__ __device__ constexpr bool warp_push_fits(int splits, int rows, int recv_bytes = AttnTile<D>::kRecvBytes) {
    return (splits - 1) * kConsumerWarps * cluster_slot_floats<D>(rows) * 4 <= recv_bytes;
}

// Workspace merge of one unit's `nparts` partial states (this CTA's own already
// written): the CTA that arrives last merges them. A unit's partials are packed
// densely from the start of its region: (m, l) of split s, row `row` at float pair
// slot0 * kRows + s * rows + row of ws_ml, its output row at the same index (times D)
// of ws_part, so a batch of splits is one contiguous block of each. Run by the consumer
// threads (threadIdx.x < 128). `bar` is an mbarrier (count 1) for the bulk copies,
// `stage` (stage_bytes) and `scratch` shared memory this CTA no longer needs. A partial
// with l < 0 comes from a split that must not write: the merge then writes nothing for
// the unit.
template <int D, int kRows, typename OutRow>
__device__ __forceinline__ void workspace_merge(const AttnParams &p, uint64_t *bar, int *s_last, int rows, int nparts,
                                                int64_t unit, int64_t slot0, float *stage, int stage_bytes,
                                                float *scratch, OutRow out_row) {
    const int ctid = threadIdx.x;  // 0 .. 127
    // Every split arrives (a failed one with l = -1), so the counter always completes and
    // the last CTA leaves it zeroed for the next launch. One thread per CTA publishes
    // the CTA's partial and, in the last CTA, acquires the others' with one acquire-
    // release update of the counter after the CTA barrier.
    consumer_bar_sync();
    if (ctid == 0) {
        int prev;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(prev) : "l"(&p.ws_count[unit]) : "memory");
        *s_last = (prev == nparts - 1);
    }
    consumer_bar_sync();
    if (!*s_last) return;
    // The partials come into shared memory by two bulk copies per batch of splits (the
    // batch's (m, l) block and its output rows). Per batch, warps first derive each row's
    // maximum, normaliser and per-split weights (in `scratch`); each thread then sums its
    // 4-float output chunks with those weights and folds the batch into its running
    // state. (Copies issued one per split cost about 40 ns each to issue; loading the
    // partials with plain loads took longer to arrive.)
    const int warp = ctid >> 5, lane = ctid & 31;
    constexpr int kC = D / 4;  // 4-float chunks per row
    constexpr int kThreads = kConsumerWarps * 32;
    constexpr int kCpt = (kRows * kC + kThreads - 1) / kThreads;
    const int ml_split = rows * 2, o_split = rows * D;             // floats per split
    const int nfit = (stage_bytes / 4 / (ml_split + o_split)) & ~1;  // even: batches start 16-byte aligned
    const int ml_cap = nfit * ml_split + 4;                         // + the 16-byte rounding of the copy
    const int nbmax = min(nfit, (stage_bytes / 4 - ml_cap) / o_split & ~1);
    float *ml_st = stage;                                           // [nbmax][rows][2] (+ slack)
    float *o_st = stage + ml_cap;                                   // [nbmax][rows][D]
    float *w_st = scratch;                                          // [nbmax][rows] weights, 0 for l <= 0
    float *mb_st = scratch + nbmax * rows;                          // [rows] batch maximum
    float *lb_st = mb_st + kRows;                                   // [rows] batch normaliser, -1 if failed
    const float *ml_g = p.ws_ml + slot0 * kRows * 2;
    const float *o_g = p.ws_part + slot0 * kRows * D;
    // Each 4-float output chunk is summed by a group of tpc consecutive threads (more than
    // one when there are fewer chunks than threads), member i taking splits i, i + tpc, ...
    const int nchunk = rows * kC;
    int tpc = 1;
    while (tpc < 32 && 2 * tpc * nchunk <= kThreads) tpc *= 2;
    const int member = ctid & (tpc - 1), ngrp = kThreads / tpc;
    float4 acc[kCpt];
    float Mr[kCpt], Lr[kCpt];
    int crow[kCpt], cd[kCpt];
#pragma unroll
    for (int j = 0; j < kCpt; ++j) {
        const int c = ctid / tpc + j * ngrp;
        crow[j] = c < nchunk ? c / kC : -1;
        cd[j] = (c - (c / kC) * kC) * 4;
        acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        Mr[j] = -INFINITY;
        Lr[j] = 0.f;
    }
    bool fail = false;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // earlier generic use of the ring
    consumer_bar_sync();
    for (int b0 = 0, batch = 0; b0 < nparts; b0 += nbmax, ++batch) {
        const int nbt = min(nbmax, nparts - b0);
        if (ctid == 0) {
            // the (m, l) block rounded up to 16 bytes (the slack stays inside the unit's region)
            const uint32_t ml_bytes = ((uint32_t)(nbt * ml_split * 4) + 15u) & ~15u;
            const uint32_t o_bytes = (uint32_t)(nbt * o_split * 4);
            asm volatile("fence.proxy.async.global;" ::: "memory");  // the acquired partials, to the copies
            mbar_arrive_expect_tx(bar, ml_bytes + o_bytes);
            bulk_load_1d(ml_st, ml_g + (int64_t)b0 * ml_split, ml_bytes, bar);
            bulk_load_1d(o_st, o_g + (int64_t)b0 * o_split, o_bytes, bar);
        }
        const bool got = mbar_wait_warp(bar, batch & 1);
        if (!got && lane == 0) report(p.dev_status, SFI_DEV_TIMEOUT);
        if (got) {
            // per row of the batch: maximum, normaliser and weights (warp w: rows w, w + 4, ...)
            for (int row = warp; row < rows; row += kConsumerWarps) {
                float M = -INFINITY;
                bool f = false;
                for (int i = lane; i < nbt; i += 32) {
                    const float2 ml = *reinterpret_cast<const float2 *>(&ml_st[(i * rows + row) * 2]);
                    f |= ml.y < 0.f;
                    if (ml.y > 0.f) M = fmaxf(M, ml.x);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
                float Ls = 0.f;
                for (int i = lane; i < nbt; i += 32) {
                    const float2 ml = *reinterpret_cast<const float2 *>(&ml_st[(i * rows + row) * 2]);
                    const float wgt = ml.y > 0.f ? fast_exp2(ml.x - M) : 0.f;
                    w_st[i * rows + row] = wgt;
                    Ls += ml.y > 0.f ? ml.y * wgt : 0.f;
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, off);
                f = __any_sync(0xffffffffu, f);
                if (lane == 0) {
                    mb_st[row] = M;
                    lb_st[row] = f ? -1.f : Ls;
                }
            }
        }
        // a wait that ran out in any warp ends the merge for all of them
        if (consumer_bar_or(!got)) {
            fail = true;
            break;
        }
#pragma unroll
        for (int j = 0; j < kCpt; ++j) {
            const int row = crow[j];
            const float Lb = row >= 0 ? lb_st[row] : 0.f;
            fail |= Lb < 0.f;
            float4 ab = make_float4(0.f, 0.f, 0.f, 0.f);
            if (Lb > 0.f) {
                for (int i = member; i < nbt; i += tpc) {
                    const float wgt = w_st[i * rows + row];
                    const float4 o = *reinterpret_cast<const float4 *>(&o_st[(i * rows + row) * D + cd[j]]);
                    ab.x += o.x * wgt;
                    ab.y += o.y * wgt;
                    ab.z += o.z * wgt;
                    ab.w += o.w * wgt;
                }
            }
            for (int off = 1; off < tpc; off <<= 1) {  // the group's sum, in every member
                ab.x += __shfl_xor_sync(0xffffffffu, ab.x, off);
                ab.y += __shfl_xor_sync(0xffffffffu, ab.y, off);
                ab.z += __shfl_xor_sync(0xffffffffu, ab.z, off);
                ab.w += __shfl_xor_sync(0xffffffffu, ab.w, off);
            }
            if (Lb <= 0.f) continue;
            const float Mb = mb_st[row];
            const float Mn = fmaxf(Mr[j], Mb);
            const float a = Lr[j] > 0.f ? fast_exp2(Mr[j] - Mn) : 0.f;
            const float bb = fast_exp2(Mb - Mn);
            acc[j].x = acc[j].x * a + ab.x * bb;
            acc[j].y = acc[j].y * a + ab.y * bb;
            acc[j].z = acc[j].z * a + ab.z * bb;
            acc[j].w = acc[j].w * a + ab.w * bb;
            Lr[j] = Lr[j] * a + Lb * bb;
            Mr[j] = Mn;
        }
        // every thread is done with this batch (generic reads ordered before the next
        // batch's copies into the same shared memory)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        consumer_bar_sync();
    }
    // The counter goes back to zero for the next launch (after the last shared-memory
    // read: a global store would hold those up).
    if (ctid == 0) p.ws_count[unit] = 0;
    // A failed split fails every row of the unit; make the decision CTA-wide.
    if (consumer_bar_or(fail) || member != 0) return;
#pragma unroll
    for (int j = 0; j < kCpt; ++j) {
        if (crow[j] < 0) continue;
        const float lsum = Lr[j];
        float *dst = &p.out[out_row(crow[j]) * D + cd[j]];
        *reinterpret_cast<float2 *>(dst) = make_float2(acc[j].x / lsum, acc[j].y / lsum);
        *reinterpret_cast<float2 *>(dst + 2) = make_float2(acc[j].z / lsum, acc[j].w / lsum);
        if (cd[j] == 0 && p.lse) p.lse[out_row(crow[j])] = (Mr[j] + log2f(lsum)) * kLn2;
    }
}

// Cluster merge from per-warp partials (rank 0, when warp_push_fits): this CTA's warps
// have written theirs to sm_o [warps][kRows][MS], sm_m, sm_l; every warp of the other
// CTAs has pushed its (o [rows][D], m [rows], l [rows]) into slot (rank - 1) * warps +
// warp of `recv`, completing its bytes on `merge_bar`. One pass merges them all: one
// thread per row derives the maximum, normaliser and every partial's weight (own warps'
// weights over sm_m, the others' into `wrem` [partials][kRows]), then each thread sums
// 4-float chunks of the output rows. A partial with l < 0 (a failed split), `skip`
// (this CTA failed) or a wait that ran out writes nothing for the unit.
template <int D, int kRows, typename OutRow>
__device__ __forceinline__ void merge_cluster_warps(const AttnParams &p, uint64_t *merge_bar, const float *sm_o,
                                                    float *sm_m, const float *sm_l, const float *recv, float *wrem,
                                                    float *wsc, int rows, int splits, bool skip, OutRow out_row) {
    constexpr int MS = AttnTile<D>::kMergeStride;
    constexpr int kC = D / 4;  // 4-float chunks per row
    const int ctid = threadIdx.x;
    const int slot_f = cluster_slot_floats<D>(rows);
    const int nrem = (splits - 1) * kConsumerWarps;
    const bool got = mbar_wait_cluster_bounded(merge_bar, 0);  // every pushed byte has landed
    // The pushed partials are in this CTA's memory now: the other CTAs may exit.
    if (got && ctid >= 1 && ctid < splits) mbar_arrive_remote_relaxed(cluster_map(smem_u32(merge_bar), ctid));
    float *scale_row = wsc;        // [kRows]
    float *lse_row = wsc + kRows;  // [kRows]
    bool bad = skip || !got;
    if (!bad && ctid < rows) {
        const int row = ctid;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w)
            if (sm_l[w * kRows + row] > 0.f) M = fmaxf(M, sm_m[w * kRows + row]);
        for (int q = 0; q < nrem; ++q) {
            const float *ml = recv + q * slot_f + rows * D;
            const float l = ml[rows + row];
            bad |= l < 0.f;
            if (l > 0.f) M = fmaxf(M, ml[row]);
        }
        float lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float l = sm_l[w * kRows + row];
            const float f = l > 0.f ? fast_exp2(sm_m[w * kRows + row] - M) : 0.f;
            sm_m[w * kRows + row] = f;
            lsum += l > 0.f ? l * f : 0.f;
        }
        for (int q = 0; q < nrem; ++q) {
            const float *ml = recv + q * slot_f + rows * D;
            const float l = ml[rows + row];
            const float f = l > 0.f ? fast_exp2(ml[row] - M) : 0.f;
            wrem[q * kRows + row] = f;
            lsum += l > 0.f ? l * f : 0.f;
        }
        scale_row[row] = 1.f / lsum;
        lse_row[row] = (M + log2f(lsum)) * kLn2;
    }
    // A failed split fails every row of the unit; make the decision CTA-wide.
    const bool fail = consumer_bar_or(bad);
    if (!got && ctid == 0) report(p.dev_status, SFI_DEV_TIMEOUT);
    if (fail) return;
    // Every chunk of this thread is summed (all shared-memory reads) before any of the
    // stores is issued.
    constexpr int kIt = (kRows * kC + kConsumerWarps * 32 - 1) / (kConsumerWarps * 32);
    float4 acc[kIt];
    float lse_v[kIt];
#pragma unroll
    for (int i = 0; i < kIt; ++i) {
        const int c = ctid + i * kConsumerWarps * 32;
        acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        lse_v[i] = 0.f;
        if (c < rows * kC) {
            const int row = c / kC, d = (c - row * kC) * 4;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float f = sm_m[w * kRows + row];
                const float4 ow = *reinterpret_cast<const float4 *>(&sm_o[(w * kRows + row) * MS + d]);
                acc[i].x += ow.x * f;
                acc[i].y += ow.y * f;
                acc[i].z += ow.z * f;
                acc[i].w += ow.w * f;
            }
            for (int q = 0; q < nrem; ++q) {
                const float f = wrem[q * kRows + row];
                const float4 oq = *reinterpret_cast<const float4 *>(&recv[q * slot_f + row * D + d]);
                acc[i].x += oq.x * f;
                acc[i].y += oq.y * f;
                acc[i].z += oq.z * f;
                acc[i].w += oq.w * f;
            }
            const float sc = scale_row[row];
            acc[i] = make_float4(acc[i].x * sc, acc[i].y * sc, acc[i].z * sc, acc[i].w * sc);
            lse_v[i] = lse_row[row];
        }
    }
#pragma unroll
    for (int i = 0; i < kIt; ++i) {
        const int c = ctid + i * kConsumerWarps * 32;
        if (c >= rows * kC) break;
        const int row = c / kC, d = (c - row * kC) * 4;
        store_out4(&p.out[out_row(row) * D + d], acc[i]);
        if (d == 0 && p.lse) p.lse[out_row(row)] = lse_v[i];
    }
}

// Split merge of one unit's partial states (m, l, unnormalised o per query row), run by
// the consumer threads (threadIdx.x < 128) of each of the unit's CTAs once this CTA's
// partial is written. Without a cluster the partials are in the workspace (slots from
// slot0) and workspace_merge combines them. When the unit's splits form a thread-block
// cluster, the other CTAs either have pushed their partials into rank 0's receive region
// `recv` with asynchronous distributed shared-memory stores that complete their bytes on
// rank 0's `merge_bar` (`push`; each slot holds o [rows][D], m [rows], l [rows]) or keep
// them in their own cp_o [rows][D], cp_m, cp_l for rank 0 to
// pull, when they do not fit. Rank 0 merges in two passes: one thread per row derives
// the row's maximum, normaliser and the splits' weights (into `wsc`: [kMaxClusterSplits]
// [kRows] weights, then [kRows] output scales 1 / l and [kRows] natural-log LSEs), then
// each thread sums 4-float chunks of the output rows with those weights. A partial with
// l < 0 comes from a split that must not write (a bad page id or a timed-out wait): the
// merge then writes nothing for the unit. (Clusters of 8 whose partials then merge
// through the workspace were measured and dropped: batch-1 dense at 16K, 32 splits,
// 15.9 -> 22.9 us per layer against merging the 32 splits one by one.)
template <int D, int kRows, bool CLUSTER, typename OutRow>
__device__ __forceinline__ void merge_splits(const AttnParams &p, float *recv, bool push, uint64_t *merge_bar,
                                             int *s_last, float *cp_o, float *cp_m, float *cp_l, float *wsc,
                                             int rows, int splits, int split, int64_t unit, int64_t slot0,
                                             float *stage, int stage_bytes, OutRow out_row) {
    const int ctid = threadIdx.x;  // 0 .. 127
    if (!CLUSTER) {
        workspace_merge<D, kRows>(p, merge_bar, s_last, rows, splits, unit, slot0, stage, stage_bytes, recv, out_row);
        return;
    }
    const int csize = splits;
    if (split != 0) {
        if (push) {
            // This CTA's asynchronous stores complete on rank 0's barrier by themselves. Rank 0
            // signals once every push has landed; only then may this CTA exit.
            if (ctid == 0 && !mbar_wait_cluster_bounded(merge_bar, 0)) report(p.dev_status, SFI_DEV_TIMEOUT);
        } else {
            consumer_bar_sync();  // this CTA's partial is complete in its shared memory
            if (ctid == 0) {
                mbar_arrive_remote(cluster_map(smem_u32(merge_bar), 0));  // "my partial is ready"
                // Stay alive (shared memory readable) until rank 0 has read it.
                if (!mbar_wait_cluster_bounded(merge_bar, 0)) report(p.dev_status, SFI_DEV_TIMEOUT);
            }
        }
        return;
    }
    bool got;
    if (push) {
        got = mbar_wait_cluster_bounded(merge_bar, 0);  // every pushed byte has landed
        // The pushed partials are in this CTA's memory now: the peers may exit. The signal
        // orders nothing (a release here stalled the merge by about 1 us).
        if (got && ctid >= 1 && ctid < csize) mbar_arrive_remote_relaxed(cluster_map(smem_u32(merge_bar), ctid));
    } else {
        if (ctid == 0) *s_last = mbar_wait_cluster_bounded(merge_bar, 0) ? 1 : 0;
        consumer_bar_sync();
        got = *s_last != 0;
    }
    const int slot_f = cluster_slot_floats<D>(rows);
    float *w_row = wsc;                                   // [kMaxClusterSplits][kRows]
    float *scale_row = wsc + kMaxClusterSplits * kRows;   // [kRows]
    float *lse_row = scale_row + kRows;                   // [kRows]
    bool bad = !got;
    if (got && ctid < rows) {
        const int row = ctid;
        float ms[kMaxClusterSplits], ls[kMaxClusterSplits];
#pragma unroll
        for (int s = 0; s < kMaxClusterSplits; ++s) {
            if (s >= csize) break;
            if (s == 0) {
                ms[s] = cp_m[row];
                ls[s] = cp_l[row];
            } else if (push) {
                const float *src = recv + (s - 1) * slot_f + rows * D;
                ms[s] = src[row];
                ls[s] = src[rows + row];
            } else {
                ms[s] = ld_cluster_f32(cluster_map(smem_u32(&cp_m[row]), s));
                ls[s] = ld_cluster_f32(cluster_map(smem_u32(&cp_l[row]), s));
            }
        }
        float M = -INFINITY;
#pragma unroll
        for (int s = 0; s < kMaxClusterSplits; ++s) {
            if (s >= csize) break;
            if (ls[s] > 0.f) M = fmaxf(M, ms[s]);
            bad |= ls[s] < 0.f;
        }
        float lsum = 0.f;
#pragma unroll
        for (int s = 0; s < kMaxClusterSplits; ++s) {
            if (s >= csize) break;
            const float w = ls[s] > 0.f ? fast_exp2(ms[s] - M) : 0.f;
            w_row[s * kRows + row] = w;
            lsum += ls[s] > 0.f ? ls[s] * w : 0.f;
        }
        scale_row[row] = 1.f / lsum;
        lse_row[row] = (M + log2f(lsum)) * kLn2;
    }
    // A failed split fails every row of the unit; make the decision CTA-wide.
    const bool fail = consumer_bar_or(bad);
    if (!got && ctid == 0) report(p.dev_status, SFI_DEV_TIMEOUT);
    if (!fail) {
        constexpr int kC = D / 4;  // 4-float chunks per row
        // Every chunk of this thread is summed (the loads of all splits issued together, so
        // distributed shared-memory latencies overlap) before any of the stores is issued:
        // a shared-memory load after a global store waits for the store path.
        constexpr int kIt = (kRows * kC + kConsumerWarps * 32 - 1) / (kConsumerWarps * 32);
        float4 acc[kIt];
        float lse_v[kIt];
#pragma unroll
        for (int i = 0; i < kIt; ++i) {
            const int c = ctid + i * kConsumerWarps * 32;
            acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            lse_v[i] = 0.f;
            if (c < rows * kC) {
                const int row = c / kC, d = (c - row * kC) * 4;
#pragma unroll
                for (int s = 0; s < kMaxClusterSplits; ++s) {
                    if (s < csize) {
                        float4 o;
                        if (s == 0)
                            o = *reinterpret_cast<const float4 *>(&cp_o[row * D + d]);
                        else if (push)
                            o = *reinterpret_cast<const float4 *>(&recv[(s - 1) * slot_f + row * D + d]);
                        else
                            o = ld_cluster_f32x4(cluster_map(smem_u32(&cp_o[row * D + d]), s));
                        const float w = w_row[s * kRows + row];
                        acc[i].x += o.x * w;
                        acc[i].y += o.y * w;
                        acc[i].z += o.z * w;
                        acc[i].w += o.w * w;
                    }
                }
                const float sc = scale_row[row];
                acc[i] = make_float4(acc[i].x * sc, acc[i].y * sc, acc[i].z * sc, acc[i].w * sc);
                lse_v[i] = lse_row[row];
            }
        }
#pragma unroll
        for (int i = 0; i < kIt; ++i) {
            const int c = ctid + i * kConsumerWarps * 32;
            if (c >= rows * kC) break;
            const int row = c / kC, d = (c - row * kC) * 4;
            store_out4(&p.out[out_row(row) * D + d], acc[i]);
            if (d == 0 && p.lse) p.lse[out_row(row)] = lse_v[i];
        }
    }
    if (!push) {
        consumer_bar_sync();  // every read of the peers' shared memory is done
        if (got && ctid > 0 && ctid < csize) mbar_arrive_remote(cluster_map(smem_u32(merge_bar), ctid));
    }
}

// MQ: p.tokens query tokens per request (rows = tokens x G <= 16).
template <int D, int MODE, bool SCORES, bool CLUSTER, bool MQ>
__global__ void __launch_bounds__(kAttnThreads, kAttnCtasPerSm)
    attn_decode_kernel(const __grid_constant__ CUtensorMap tm_pool_k, const __grid_constant__ CUtensorMap tm_pool_v,
                       const __grid_constant__ CUtensorMap tm_comp_k, const __grid_constant__ CUtensorMap tm_comp_v,
                       const AttnParams p) {
    using T = AttnTile<D>;
    constexpr int kRows = MQ ? kMaxRows : kMaxGroup;  // query rows per unit in the merge buffers
    // bytes of the receive region open to the cluster push (the rest holds the query tile)
    constexpr int kPushBytes = MQ ? T::kRecvBytes - T::kQBytes : T::kRecvBytes;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned (the 128-byte swizzle pattern repeats every 1 KB). Offsetting the
    // array itself, rather than rounding an integer address, keeps every pointer derived
    // from it a shared-memory pointer to the compiler (shared loads and stores, and no
    // assumed aliasing with global stores in the merges).
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ __align__(8) uint64_t full_bar[T::kStages];
    __shared__ __align__(8) uint64_t empty_bar[T::kStages];
    __shared__ __align__(8) uint64_t merge_bar;  // cluster merge handshake, or the workspace merge's copies
    __shared__ int2 s_info[T::kStages][kConsumerWarps];
    __shared__ int s_last;
    __shared__ int s_timeout;
    __shared__ int s_bad;  // a page id of this unit is out of range: the unit writes no output
    __shared__ __align__(16) int4 s_app_val[32];  // the current token's K/V chunks (fused append)
    __shared__ int s_app_page;
    __shared__ int s_tok_page[kConsumerWarps];  // page ids of the staged query tokens (multi-token append)

    // ---- this CTA's work item: (request, KV head, split) and the unit's mode ----
    int split, kvh, b, splits;
    bool fast;
    int64_t unit, slot0;  // merge counter index; first partial slot of the unit
    const int *ids = p.req_ids;
    if (MODE == kModeMixed) {
        // 1-D grid: the slow units' splits first, then the fast units'
        int item = blockIdx.x;
        const int n_slow_items = p.n_slow * p.hkv * p.slow_splits;
        fast = item >= n_slow_items;
        splits = fast ? p.fast_splits : p.slow_splits;
        if (fast) item -= n_slow_items;
        split = item % splits;
        const int u_local = item / splits;
        kvh = u_local % p.hkv;
        b = u_local / p.hkv;
        ids = fast ? p.fast_ids : p.slow_ids;
        unit = fast ? (int64_t)p.n_slow * p.hkv + u_local : u_local;
        slot0 = fast ? (int64_t)p.n_slow * p.hkv * p.slow_splits + (int64_t)u_local * splits : (int64_t)u_local * splits;
    } else {
        split = blockIdx.x;
        kvh = blockIdx.y;
        b = blockIdx.z;
        splits = p.splits;
        fast = MODE == kModeFast;
        unit = (int64_t)b * p.hkv + kvh;
        slot0 = unit * splits;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tm_pool_k);
        tma_prefetch_desc(&tm_pool_v);
        if (MODE != kModeDense) {
            tma_prefetch_desc(&tm_comp_k);
            tma_prefetch_desc(&tm_comp_v);
        }
    }
    // Programmatic dependent launch: this CTA may have started while the previous
    // kernel in the stream was still running. By default it waits for that kernel
    // (and its memory) before touching any global data. With early_prefetch the
    // caller guarantees that kernel writes none of the KV state read below, so only
    // the consumer warps wait, right before they read q and write anything. The next
    // kernel is released only after this CTA's wait, so at most two kernels overlap.
    if (!p.early_prefetch) {
        grid_dependency_wait();
        grid_launch_dependents();
    }
    const int r = ids ? ids[b] : b;

    UnitStream u;
    if (!unit_stream(p, r, kvh, fast, split == 0, u)) return;  // uniform across the CTA and its cluster
    int per = (u.nb + splits - 1) / splits;
    if (MODE == kModeMixed) {
        const int chunk = fast ? p.fast_chunk_sb : p.slow_chunk_sb;
        if (chunk > 0) {
            // Fixed-size chunks (ragged batches): this unit uses ceil(nb / chunk) of the
            // grid's splits for its mode; the CTAs past them have nothing to do. A unit
            // longer than the host's bound takes bigger chunks, never more splits.
            per = max(chunk, (u.nb + splits - 1) / splits);
            splits = max(1, (u.nb + per - 1) / per);
            if (split >= splits) return;
        }
    }
    const int sb_begin = split * per;
    const int sb_end = min(u.nb, sb_begin + per);
    const int n_my = max(0, sb_end - sb_begin);
    // Stage st holds sub-blocks sb0 + 4 st + [0, 4) that lie in [sb_begin, sb_end). When
    // the split's count is not a multiple of 4 the partial stage comes first, where the
    // warps wait for the pipeline to fill anyway, so all four finish the last stage
    // together.
    const int pad = (kConsumerWarps - n_my % kConsumerWarps) % kConsumerWarps;
    const int sb0 = sb_begin - pad;
    const int n_stages = (n_my + pad) / kConsumerWarps;
    // Page id of sub-block sb (-1 for compact sub-blocks and past the split's range).
    const int32_t *ptab = p.page_table + (int64_t)r * p.max_pages;
    auto page_of = [&](int sb) -> int {
        if (sb >= sb_end || sb < sb_begin || sb < u.nb1) return -1;
        return ptab[u.page0 + (sb - u.nb1)];
    };
    // When the first stage holds paged sub-blocks (dense units), the producer warp issues
    // the loads of its first two chunks of page ids now: they travel while the barriers
    // are initialised.
    const bool ids_first = warp == kConsumerWarps && sb0 + kConsumerWarps > u.nb1;
    int ids_cur = -1, ids_nxt = -1;
    if (ids_first) {
        ids_cur = page_of(sb0 + lane);
        ids_nxt = page_of(sb0 + 32 + lane);
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < T::kStages; ++i) {
            mbar_init(&full_bar[i], kConsumerWarps);
            mbar_init(&empty_bar[i], kConsumerWarps);
        }
        // push merge: rank 0's barrier expects the bytes of the other CTAs' partials (their
        // asynchronous stores complete them); pull merge: one arrival per other CTA;
        // workspace merge: the last CTA's bulk copies of the unit's partials
        const int mrows = MQ ? p.rows : p.group;
        const bool wpush0 = CLUSTER && !MQ && warp_push_fits<D>(splits, mrows, kPushBytes);
        const bool push0 = CLUSTER && split == 0 && cluster_push_fits<D>(splits, mrows, kPushBytes);
        if (CLUSTER)
            mbar_init(&merge_bar, split != 0 || push0 ? 1u : (uint32_t)(splits - 1));
        else
            mbar_init(&merge_bar, 1u);
        if (push0)
            mbar_arrive_expect_tx(&merge_bar,
                                  (uint32_t)((splits - 1) * (wpush0 ? kConsumerWarps : 1) * mrows * (D + 2) * 4));
        s_timeout = 0;
        s_bad = 0;
        fence_barrier_init();
    }
    // Every CTA of a cluster reaches this point unconditionally (the only branch
    // before it depends on the unit's metadata, which all of them read alike) and
    // arrives on the cluster barrier; a thread waits on it only before its first access
    // to another CTA (after its stream), by when each CTA's merge barrier is
    // initialised for remote arrivals. (A relaxed cluster arrive instead of a release
    // one: drafts at batch 16, T = 1 / 4 / 8, 14.7 / 15.3 / 17.9 -> 14.5 / 15.2 / 17.3 us
    // per launch.)
    if (CLUSTER) cluster_arrive_after_init();
    else __syncthreads();

    if (warp == kConsumerWarps) {
        // ---------------- producer warp ----------------
        const uint64_t policy = l2_policy_evict_first();
        // Page ids of the current and the next chunk of 32 sub-blocks. When the first stage
        // is all compact rows they are loaded only after its copies are issued, so those
        // copies do not wait for the page table.
        int cur = ids_cur, nxt = ids_nxt;
        bool ids_loaded = ids_first;
        auto load_ids = [&]() {
            cur = page_of(sb0 + lane);
            nxt = page_of(sb0 + 32 + lane);
            ids_loaded = true;
        };
        // L2 prefetch of stage pst's sub-blocks (page ids of its chunk of 32 in page_src;
        // warp-collective). Dense units prefetch the rest of their first chunk right after
        // the ring's first fill, so the first refills read L2 without delaying the ring's
        // own copies. (Measured: it shortens the slow step; on short fast-step units it
        // costs more than it saves. A rolling prefetch 8 stages ahead for launches of at
        // most one CTA per SM made them slower: batch-1 dense at 16K, 21.2 -> 23.7 us.)
        auto prefetch_stage = [&](int pst, int page_src) {
            const int page = __shfl_sync(0xffffffffu, page_src, ((pst & 7) * kConsumerWarps) + (lane & (kConsumerWarps - 1)));
            const int sb = sb0 + pst * kConsumerWarps + lane;
            if (lane < kConsumerWarps && sb >= sb_begin && sb < sb_end) {
                if (sb < u.nb1) {  // compact rows
                    const int32_t y = static_cast<int32_t>(u.crow0 + (int64_t)sb * kSubTokens);
#pragma unroll
                    for (int bx = 0; bx < T::kBoxes; ++bx) {
                        tma_prefetch_l2_2d(&tm_comp_k, bx * 64, y);
                        tma_prefetch_l2_2d(&tm_comp_v, bx * 64, y);
                    }
                } else if (page >= 0 && page < p.num_pages) {
                    const int32_t y = (page * p.hkv + kvh) * kSubTokens;
#pragma unroll
                    for (int bx = 0; bx < T::kBoxes; ++bx) {
                        tma_prefetch_l2_2d(&tm_pool_k, bx * 64, y);
                        tma_prefetch_l2_2d(&tm_pool_v, bx * 64, y);
                    }
                }
            }
        };
        for (int st = 0; st < n_stages; ++st) {
            if (st > 0 && (st & 7) == 0) {  // 8 stages x 4 sub-blocks = 32 page ids per chunk
                cur = nxt;
                nxt = page_of(sb0 + (st / 8 + 1) * 32 + lane);
            }
            const int slot = st % T::kStages;
            if (st >= T::kStages) {
                if (!mbar_wait_warp(&empty_bar[slot], ((st / T::kStages) - 1) & 1)) {
                    if (lane == 0) report(p.dev_status, SFI_DEV_TIMEOUT);
                    break;
                }
            }
            if (p.withhold == st + 1) continue;  // diagnostic: this stage's copies never come
            // A stage of compact sub-blocks needs no page id; skipping the shuffle there keeps
            // the page-table loads off the path of the first TMA copies.
            const bool paged = sb0 + (st + 1) * kConsumerWarps > u.nb1;  // warp-uniform
            const int page =
                paged ? __shfl_sync(0xffffffffu, cur, ((st & 7) * kConsumerWarps) + (lane & (kConsumerWarps - 1))) : -1;
            if (lane < kConsumerWarps) {
                const int sb = sb0 + st * kConsumerWarps + lane;
                int lo = 0, hi = 0, pos0 = 0;
                const CUtensorMap *mk = &tm_pool_k;
                const CUtensorMap *mv = &tm_pool_v;
                int32_t y = 0;
                if (sb >= sb_begin && sb < sb_end) {
                    if (sb < u.nb1) {  // compact segment (fast mode only)
                        mk = &tm_comp_k;
                        mv = &tm_comp_v;
                        y = static_cast<int32_t>(u.crow0 + (int64_t)sb * kSubTokens);
                        hi = min(kSubTokens, u.n1 - sb * kSubTokens);
                        pos0 = -1;
                    } else {
                        const int pg = u.page0 + (sb - u.nb1);
                        if (page < 0 || page >= p.num_pages) {
                            report(p.dev_status, SFI_DEV_BAD_PAGE);
                            s_bad = 1;  // seen by the consumers through this stage's barrier
                        } else {
                            y = (page * p.hkv + kvh) * kSubTokens;
                            pos0 = pg * kSubTokens;
                            lo = max(0, u.lo_pos - pos0);
                            hi = min(kSubTokens, u.L - pos0);
                        }
                    }
                }
                s_info[slot][lane] = make_int2(lo | (hi << 16), pos0);
                if (hi > lo) {
                    uint8_t *kdst = smem + slot * T::kStageBytes + lane * 2 * T::kSubBytes;
                    uint8_t *vdst = kdst + T::kSubBytes;
                    mbar_arrive_expect_tx(&full_bar[slot], 2 * T::kSubBytes);
#pragma unroll
                    for (int bx = 0; bx < T::kBoxes; ++bx) {
                        tma_load_2d(kdst + bx * (kSubTokens * 128), mk, bx * 64, y, &full_bar[slot], policy);
                        tma_load_2d(vdst + bx * (kSubTokens * 128), mv, bx * 64, y, &full_bar[slot], policy);
                    }
                } else {
                    mbar_arrive(&full_bar[slot]);
                }
            }
            if (!ids_loaded) load_ids();
            if (!fast && st == T::kStages - 1)
                for (int pst = T::kStages; pst < 8 && pst < n_stages; ++pst) prefetch_stage(pst, cur);
        }
        if (CLUSTER) cluster_wait();
        return;  // the producer takes no part in the merges
    }

    // ---------------- consumer warps ----------------
    // Units that write scores first check every page id of the request; with
    // early_prefetch the page table is not written by the preceding kernel, so the first
    // loads of that check go out before the dependency wait.
    const bool check_pages = SCORES && p.scores && !fast && u.L <= p.score_stride;
    int pg_first[kPageCheckLoads];
    if (check_pages && p.early_prefetch) pages_first(p, r, u.L, pg_first);
    if (p.early_prefetch) {
        grid_dependency_wait();
        grid_launch_dependents();
    }
    if (check_pages && !p.early_prefetch) pages_first(p, r, u.L, pg_first);
    if (MQ && p.k_new != nullptr) {
        // The CTA that appends the query tokens' K/V (positions [L - T, L), in the last
        // one or two sub-blocks) brings their rows into L2 now; the append reads them
        // at the end of the stream.
        const int sb_first = u.sb_app - ((u.L - 1) / kSubTokens - (u.L0 - 1) / kSubTokens);
        if (sb_begin <= u.sb_app && sb_end > sb_first) {
            constexpr int kLines = D * 2 / 128;  // 128-byte lines per K (or V) row
            for (int i = threadIdx.x; i < p.tokens * 2 * kLines; i += kConsumerWarps * 32) {
                const int tok = i / (2 * kLines), rem = i - tok * 2 * kLines;
                const __nv_bfloat16 *src = (rem < kLines ? p.k_new : p.v_new) +
                                           (((int64_t)r * p.tokens + tok) * p.hkv + kvh) * D + (rem % kLines) * 64;
                asm volatile("prefetch.global.L2 [%0];" ::"l"(src));
            }
        }
    }
    const int g = lane >> 2, t = lane & 3;
    const int G = p.group;
    uint32_t qa[D / 16][2];
    const uint32_t qtile = smem_u32(smem + T::kRecvOffset + T::kRecvBytes - T::kQBytes);
    if constexpr (MQ) {
        // The 16-row query tile goes to shared memory (row rho is query token rho / G,
        // head rho % G of this KV head's group; rows past p.rows are zero), 16-byte
        // chunk c of row rho at chunk c ^ (rho & 7): the A fragments are read with
        // ldmatrix in each sub-block, which keeps 32 registers free. The rows come by
        // asynchronous copies in their own group, waited for right before the stream, so
        // their latency overlaps the rest of the set-up and the first stage's copies
        // (loading them through registers exposed one round trip per row a thread
        // loads: 1.1 us at T = 4, 2.0 us at T = 8, from the dependency wait to the loop).
        constexpr int kChunks = D / 8;
        uint8_t *qt = smem + T::kRecvOffset + T::kRecvBytes - T::kQBytes;
        for (int e = threadIdx.x; e < kMaxRows * kChunks; e += kConsumerWarps * 32) {
            const int rho = e / kChunks, c = e - rho * kChunks;
            uint8_t *dst = qt + rho * (D * 2) + ((c ^ (rho & 7)) << 4);
            if (rho < p.rows) {
                const int tok = rho / G;
                const __nv_bfloat16 *src =
                    p.q + (((int64_t)r * p.tokens + tok) * p.hq + (int64_t)kvh * G + (rho - tok * G)) * D + c * 8;
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
            } else {
                *reinterpret_cast<int4 *>(dst) = make_int4(0, 0, 0, 0);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    } else {
        const __nv_bfloat16 *qrow = p.q + ((int64_t)r * p.hq + (int64_t)kvh * G + g) * D;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            if (g < G) {
                qa[ks][0] = *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 2 * t);
                qa[ks][1] = *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 8 + 2 * t);
            } else {
                qa[ks][0] = 0u;
                qa[ks][1] = 0u;
            }
        }
    }
    // Per-row bounds (MQ): the length token rho / G sees and the start of its recent
    // window (0 in dense mode). Padding rows take the last token's.
    int row_len[2] = {u.L, u.L}, row_lo[2] = {0, 0};
    if constexpr (MQ) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int rho = min(g + 8 * half, p.rows - 1);
            row_len[half] = u.L0 + rho / G;
            row_lo[half] = fast ? max(p.sink, row_len[half] - p.recent) : 0;
        }
    }
    float o[D / 8][4];
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};  // rows g and g + 8 (MQ)
    float *score_row = nullptr;
    if (SCORES && p.scores && !fast) {
        if (check_pages) {
            // Scores are written as the stream goes; a unit with a bad page id anywhere in
            // [0, L) writes none of them (nor its output: the flag reaches the merge).
            if (!pages_bad(p, r, u.L, pg_first)) {
                score_row = p.scores + ((int64_t)r * p.hkv + kvh) * p.score_stride;
            } else if (threadIdx.x == 0) {
                s_bad = 1;
            }
        } else if (threadIdx.x == 0 && split == 0) {
            report(p.dev_status, SFI_DEV_BAD_LEN);  // score row too short: scores not written
        }
    }

    // the warp that owns the sub-block with the current token (single-token append)
    const bool app_mine = !MQ && p.k_new != nullptr && u.sb_app >= sb_begin && u.sb_app < sb_end &&
                          (u.sb_app - sb0) % kConsumerWarps == warp;
    if (app_mine) stage_current_token<D>(p, r, kvh, u, lane, s_app_val, &s_app_page);
    // Multi-token append: the first position of the paged sub-block with query tokens
    // that this warp owns (-1 if none). Their K/V are staged at the start of the receive
    // region, which nothing else uses during the stream unless this CTA is rank 0 of a
    // cluster (the push target): that CTA appends from global memory instead.
    int tok_pos0 = -1;
    uint8_t *tok_stage = smem + T::kRecvOffset;
    if (MQ && p.k_new != nullptr && !(CLUSTER && split == 0)) {
        const int pos_last = ((u.L - 1) / kSubTokens) * kSubTokens;
        for (int k = 0; k < 2; ++k) {  // T <= 16 tokens lie in at most two sub-blocks
            const int pos0 = pos_last - k * kSubTokens, sb = u.sb_app - k;
            // stop below the query tokens or outside the paged segment
            if (pos0 + kSubTokens <= u.L0 - 1 || u.lo_pos >= u.L || pos0 / kSubTokens < u.page0) break;
            if (sb >= sb_begin && sb < sb_end && (sb - sb0) % kConsumerWarps == warp) tok_pos0 = pos0;
        }
        if (tok_pos0 >= 0) stage_tokens<D>(p, r, kvh, u.L, tok_pos0, lane, tok_stage, &s_tok_page[warp]);
    }
    if constexpr (MQ) {
        // the query tile is complete (this thread's copies) and visible (every thread's)
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        consumer_bar_sync();
    }
    bool timed_out = false;
    const int store_st = min(2, n_stages - 1);
    for (int st = 0; st < n_stages; ++st) {
        const int slot = st % T::kStages;
        if (!mbar_wait_warp(&full_bar[slot], (st / T::kStages) & 1)) {
            timed_out = true;
            break;
        }
        const int2 in = s_info[slot][warp];
        const int lo = in.x & 0xffff, hi = in.x >> 16;
        const int sb_me = sb0 + st * kConsumerWarps + warp;  // this warp's sub-block in the stage
        // The appended tokens go to the pages at the third stage (the first ones wait on
        // the staged copies more often; at T = 8 drafts this was 0.3 us per launch faster
        // than the first stage).
        if (st == store_st && app_mine) store_current_token<D>(p, kvh, u, lane, s_app_val, &s_app_page, &s_bad);
        if (st == store_st && tok_pos0 >= 0)
            store_tokens<D>(p, kvh, u.L, tok_pos0, lane, tok_stage, &s_tok_page[warp], &s_bad);
        if (app_mine && sb_me == u.sb_app) {
            // Fused append: the current token's K/V replace row L - 1 of this tile (the
            // attention sees the cache after the append). Only the split that owns that
            // sub-block does it (a stage's padding slots past sb_end may carry the same
            // index).
            fuse_current_token<D>(smem + slot * T::kStageBytes + warp * 2 * T::kSubBytes, u, lane, s_app_val);
        }
        if (MQ && p.k_new != nullptr && in.y >= 0 && sb_me >= sb_begin && sb_me < sb_end &&
            in.y + kSubTokens > u.L0 - 1 && in.y < u.L) {
            // Fused append of the query tokens (positions [L - T, L)) in this paged sub-block.
            if (in.y == tok_pos0)
                fuse_staged_tokens<D>(smem + slot * T::kStageBytes + warp * 2 * T::kSubBytes, p, u.L, in.y, lane,
                                      tok_stage);
            else
                fuse_tokens<D>(smem + slot * T::kStageBytes + warp * 2 * T::kSubBytes, p, r, kvh, u.L, in.y, lane,
                               &s_bad);
        }
        if (hi > lo) {
            const uint32_t kaddr = smem_u32(smem + slot * T::kStageBytes + warp * 2 * T::kSubBytes);
            if constexpr (MQ) {
                RowSpan ra, rb;
                if (in.y >= 0) {  // paged positions pos0 + i
                    ra = RowSpan{max(lo, row_lo[0] - in.y), min(hi, row_len[0] - in.y)};
                    rb = RowSpan{max(lo, row_lo[1] - in.y), min(hi, row_len[1] - in.y)};
                } else {  // compact rows: without a selection they are the sink positions
                    const int c0 = sb_me * kSubTokens;
                    ra = RowSpan{lo, u.cnt > 0 ? hi : min(hi, row_len[0] - c0)};
                    rb = RowSpan{lo, u.cnt > 0 ? hi : min(hi, row_len[1] - c0)};
                }
                const bool full = __all_sync(0xffffffffu, ra.lo == 0 && ra.hi == kSubTokens && rb.lo == 0 &&
                                                              rb.hi == kSubTokens);
                consume_sub_block_mq<D, SCORES>(kaddr, kaddr + T::kSubBytes, lo, hi, full, ra, rb, in.y, qtile,
                                                o, m_run, l_run, p, score_row, u.L, lane);
            } else {
                consume_sub_block<D, SCORES>(kaddr, kaddr + T::kSubBytes, lo, hi, in.y, qa, o, m_run[0], l_run[0],
                                             p, score_row, u.L, lane);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[slot]);
    }
    // staged copies still in flight after a timed-out wait land before shared memory is reused
    if (app_mine || tok_pos0 >= 0) asm volatile("cp.async.wait_all;" ::: "memory");
    if (timed_out && lane == 0) {
        report(p.dev_status, SFI_DEV_TIMEOUT);
        s_timeout = 1;
    }
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        l_run[half] += __shfl_xor_sync(0xffffffffu, l_run[half], 1);
        l_run[half] += __shfl_xor_sync(0xffffffffu, l_run[half], 2);
    }
    if (CLUSTER) cluster_wait();  // the other CTAs' mbarriers are initialised
    // up to 8 query rows: rows g + 8 hold the P_lo V half of row g
    const bool packed = !MQ || p.rows <= kMaxGroup;
    const int rows = MQ ? p.rows : G;
    float *recv = reinterpret_cast<float *>(smem + T::kRecvOffset);
    // Small partials: every warp of a CTA other than cluster rank 0 sends its own partial
    // straight into its slot of rank 0's receive region as soon as its stream ends, and
    // rank 0 merges all the cluster's warps in one pass (no warp merge in those CTAs).
    // Single-token kernels only: in the multi-token one the partials rarely fit, and the
    // extra path alone cost its drafts 0.2 us per launch.
    const bool wpush = CLUSTER && !MQ && splits > 1 && warp_push_fits<D>(splits, rows, kPushBytes);
    if (wpush && split != 0) {
        const bool bad_w = timed_out || s_bad != 0;  // l = -1: rank 0 writes nothing for the unit
        const uint32_t cbar = cluster_map(smem_u32(&merge_bar), 0);
        const uint32_t slot = cluster_map(smem_u32(recv), 0) +
                              (uint32_t)(((split - 1) * kConsumerWarps + warp) * cluster_slot_floats<D>(rows)) * 4u;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int row = g + 8 * half;
            if ((half == 1 && packed) || row >= rows) continue;
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt) {
                float2 v = packed ? make_float2(o[nt][0] + o[nt][2], o[nt][1] + o[nt][3])
                                  : make_float2(o[nt][2 * half], o[nt][2 * half + 1]);
                if (bad_w) v = make_float2(0.f, 0.f);
                st_async_f32x2(slot + (uint32_t)(row * D + nt * 8 + 2 * t) * 4u, v, cbar);
            }
            if (t == 0) {
                st_async_f32(slot + (uint32_t)(rows * D + row) * 4u, m_run[half], cbar);
                st_async_f32(slot + (uint32_t)(rows * D + rows + row) * 4u, bad_w ? -1.f : l_run[half], cbar);
            }
        }
        // Rank 0 signals once every push has landed; only then may this CTA exit.
        if (threadIdx.x == 0 && !mbar_wait_cluster_bounded(&merge_bar, 0)) report(p.dev_status, SFI_DEV_TIMEOUT);
        return;
    }

    // ---- merge the consumer warps through shared memory (stage buffers are free now) ----
    consumer_bar_sync();
    const bool ok = s_timeout == 0;
    constexpr int MS = T::kMergeStride;
    constexpr int kC = D / 4;                                       // 4-float chunks per row
    float *sm_o = reinterpret_cast<float *>(smem);                  // [warps][kRows][MS]
    float *sm_m = sm_o + kConsumerWarps * kRows * MS;               // [warps][kRows] maxima, then weights
    float *sm_l = sm_m + kConsumerWarps * kRows;                    // [warps][kRows]
    float *cp_o = sm_l + kConsumerWarps * kRows;                    // [kRows][D]  this CTA's partial (cluster merge)
    float *cp_m = cp_o + kRows * D;                                 // [kRows]
    float *cp_l = cp_m + kRows;                                     // [kRows]
    float *wsc = cp_l + kRows;                                      // [kMaxClusterSplits + 2][kRows] merge scratch
    if (ok) {
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) {
            float2 v = packed ? make_float2(o[nt][0] + o[nt][2], o[nt][1] + o[nt][3]) : make_float2(o[nt][0], o[nt][1]);
            *reinterpret_cast<float2 *>(&sm_o[(warp * kRows + g) * MS + nt * 8 + 2 * t]) = v;
            if (!packed) {
                float2 w = make_float2(o[nt][2], o[nt][3]);
                *reinterpret_cast<float2 *>(&sm_o[(warp * kRows + g + 8) * MS + nt * 8 + 2 * t]) = w;
            }
        }
        if (t == 0) {
            sm_m[warp * kRows + g] = m_run[0];
            sm_l[warp * kRows + g] = l_run[0];
            if (!packed) {
                sm_m[warp * kRows + g + 8] = m_run[1];
                sm_l[warp * kRows + g + 8] = l_run[1];
            }
        }
    }
    consumer_bar_sync();

    const int ctid = threadIdx.x;  // 0 .. 127
    // output row of tile row `row`: (request, token row / G, head kvh * G + row % G)
    const int64_t head0 = (int64_t)r * p.hq + (int64_t)kvh * G;
    auto out_row = [&](int row) -> int64_t {
        if (!MQ) return head0 + row;
        const int tok = row / G;
        return ((int64_t)r * p.tokens + tok) * p.hq + (int64_t)kvh * G + (row - tok * G);
    };
    // A partial that must not reach the output (a bad page id in the unit, or a timed-out
    // wait) carries l = -1: every merge that sees it skips the unit's writes.
    const bool skip = !ok || s_bad != 0;
    if (wpush) {  // cluster rank 0 with per-warp partials from the other CTAs
        merge_cluster_warps<D, kRows>(p, &merge_bar, sm_o, sm_m, sm_l, recv, cp_o, wsc, rows, splits, skip, out_row);
        return;
    }
    // Where this CTA's partial goes: the output (one split), rank 0's receive region
    // (cluster push from another rank), cp_* (cluster rank 0, or pull), or the workspace.
    const bool push = CLUSTER && cluster_push_fits<D>(splits, rows, kPushBytes);
    const bool remote = push && split != 0;
    const uint32_t rdst =
        remote ? cluster_map(smem_u32(recv), 0) + (uint32_t)((split - 1) * cluster_slot_floats<D>(rows)) * 4u : 0u;
    const uint32_t rbar = remote ? cluster_map(smem_u32(&merge_bar), 0) : 0u;  // completes the pushed bytes
    const int64_t wslot = slot0 * kRows + (int64_t)split * rows;  // workspace slot of row 0 (packed per unit)
    // Two passes: one thread per row takes the row's maximum over the warps, turns each
    // warp's maximum into its weight 2^(m_w - M) and sums the normaliser; then each
    // thread sums 4-float chunks of the rows with those weights.
    if (ctid < rows) {
        const int row = ctid;
        float M = -INFINITY, lsum = -1.f;
        if (ok) {
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm_m[w * kRows + row]);
            lsum = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float mw = sm_m[w * kRows + row];
                const float f = mw != -INFINITY ? fast_exp2(mw - M) : 0.f;
                sm_m[w * kRows + row] = f;
                lsum += sm_l[w * kRows + row] * f;
            }
            if (skip) lsum = -1.f;
        }
        // Row results for the second pass go to shared memory: global stores here would
        // hold up this thread's shared-memory loads behind them (the store path is long
        // while the other CTAs stream).
        if (splits == 1) {
            wsc[row] = 1.f / lsum;
            wsc[kRows + row] = (M + log2f(lsum)) * kLn2;
        } else if (remote) {
            st_async_f32(rdst + (rows * D + row) * 4, M, rbar);
            st_async_f32(rdst + (rows * D + rows + row) * 4, lsum, rbar);
        } else if (CLUSTER) {
            cp_m[row] = M;
            cp_l[row] = lsum;
        } else if (ok) {
            wsc[row] = M;
            wsc[kRows + row] = lsum;
        } else {  // no second pass
            p.ws_ml[(wslot + row) * 2 + 0] = M;
            p.ws_ml[(wslot + row) * 2 + 1] = lsum;
        }
    }
    if (ok && !(splits == 1 && skip)) {
        consumer_bar_sync();
        // Every chunk of this thread is summed (all shared-memory reads) before any of the
        // stores is issued.
        constexpr int kIt = (kRows * kC + kConsumerWarps * 32 - 1) / (kConsumerWarps * 32);
        float4 acc[kIt];
        float2 rowv[kIt];  // the row's (scale, lse) or (m, l), read by its first chunk's thread
#pragma unroll
        for (int i = 0; i < kIt; ++i) {
            const int c = ctid + i * kConsumerWarps * 32;
            acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            rowv[i] = make_float2(0.f, 0.f);
            if (c < rows * kC) {
                const int row = c / kC;
                const int d = (c - row * kC) * 4;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) {
                    const float f = sm_m[w * kRows + row];  // 0 for a warp that saw no token (its o is 0)
                    const float4 ow = *reinterpret_cast<const float4 *>(&sm_o[(w * kRows + row) * MS + d]);
                    acc[i].x += ow.x * f;
                    acc[i].y += ow.y * f;
                    acc[i].z += ow.z * f;
                    acc[i].w += ow.w * f;
                }
                if (splits == 1 || d == 0) rowv[i] = make_float2(wsc[row], wsc[kRows + row]);
            }
        }
#pragma unroll
        for (int i = 0; i < kIt; ++i) {
            const int c = ctid + i * kConsumerWarps * 32;
            if (c >= rows * kC) break;
            const int row = c / kC, d = (c - row * kC) * 4;
            if (splits == 1) {
                const float sc = rowv[i].x;
                store_out4(&p.out[out_row(row) * D + d],
                           make_float4(acc[i].x * sc, acc[i].y * sc, acc[i].z * sc, acc[i].w * sc));
                if (d == 0 && p.lse) p.lse[out_row(row)] = rowv[i].y;
            } else if (remote) {
                st_async_f32x4(rdst + (row * D + d) * 4, acc[i], rbar);
            } else if (CLUSTER) {
                *reinterpret_cast<float4 *>(&cp_o[row * D + d]) = acc[i];
            } else {
                *reinterpret_cast<float4 *>(&p.ws_part[(wslot + row) * D + d]) = acc[i];
                if (d == 0) *reinterpret_cast<float2 *>(&p.ws_ml[(wslot + row) * 2]) = rowv[i];
            }
        }
    }
    if (remote && !ok) {
        // a failed split still delivers every byte rank 0 expects (its l = -1 marks it)
        for (int c = ctid; c < rows * kC; c += kConsumerWarps * 32)
            st_async_f32x4(rdst + (uint32_t)c * 16u, make_float4(0.f, 0.f, 0.f, 0.f), rbar);
    }
    if (splits == 1) return;
    merge_splits<D, kRows, CLUSTER>(p, recv, push, &merge_bar, &s_last, cp_o, cp_m, cp_l, wsc, rows, splits, split,
                                     unit, slot0, reinterpret_cast<float *>(smem), T::kRingBytes, out_row);
}

template <int D, int MODE, bool SCORES, bool CLUSTER, bool MQ>
static cudaError_t launch_one(const AttnMaps &maps, const AttnParams &p, int batch, cudaStream_t stream) {
    using T = AttnTile<D>;
    auto kern = attn_decode_kernel<D, MODE, SCORES, CLUSTER, MQ>;
    // The shared-memory opt-in is a per-device function attribute: set it once per device.
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
    if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    cudaLaunchConfig_t cfg = {};
    if (MODE == kModeMixed)
        cfg.gridDim = dim3((unsigned)(p.n_slow * p.hkv * p.slow_splits + p.n_fast * p.hkv * p.fast_splits));
    else
        cfg.gridDim = dim3(p.splits, p.hkv, batch);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = T::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    int n_attr = 1;
    if (CLUSTER) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = p.splits;  // the splits of one unit form one cluster
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        n_attr = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n_attr;
    e = cudaLaunchKernelEx(&cfg, kern, maps.pool_k, maps.pool_v, maps.comp_k, maps.comp_v, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace sfi
