// Selector of the SFI slow step: per (request, KV head) top-k over the masked
// candidate logits, ties to the lower position, result in ascending position order.
//
// Method: Slow-Fast Inference (Xie et al., 2026), Figure 2 caption (the Selector
// refreshes the selected memory from the masked logits collected by the slow step).
//
// Design: one CTA of 1024 threads per (request, KV head).
//  * Scores are mapped to order-preserving uint32 keys (-0 -> +0, NaN -> 0, below
//    -inf).
//  * The candidates are walked in rounds of 16384 positions; in a round, warp w owns
//    the contiguous positions [512 w, 512 w + 512) and lane l holds positions
//    512 w + 32 j + l, j < 16. Rounds reach shared memory through TMA bulk copies
//    (many small loads per thread would be limited by the SM's outstanding misses):
//    with one round the keys then stay in registers for the whole selection, with two
//    both rounds stay in shared memory, with more they stream through two buffers.
//  * Radix select, 4 passes of 8 bits from the top: a 256-bin shared histogram of the
//    keys that share the current prefix (warp-aggregated atomics via match.any),
//    then one warp scans the bins from the top to find the bin holding the k-th key.
//    The result is the exact k-th largest key tau and the number of keys equal to
//    tau that must be taken (the lowest positions among them).
//  * Output in ascending position order without sorting: per (round, warp) counts of
//    keys above / equal to tau, an exclusive scan over (round, warp) in position
//    order, then each warp writes its taken positions with ballot/popc ranks.
#include <atomic>

#include "sfi_device.cuh"
#include "sfi_internal.h"

namespace sfi {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkPerThread = 16;                               // keys per thread and round
constexpr int kTopkRound = kTopkThreads * kTopkPerThread;        // 16384 positions per round
constexpr int kTopkMaxRounds = 16;                               // |C| up to 262144
constexpr uint32_t kNoKey = 0xffffffffu;                         // marks positions past |C| (never counted)

__device__ __forceinline__ uint32_t order_key(float x) {
    uint32_t u = __float_as_uint(x);
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;  // NaN ranks below everything
    if (u == 0x80000000u) u = 0u;                    // -0 == +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Add this thread's keys that share `prefix` under `mask` to the histogram of bits [shift, shift+8).
__device__ __forceinline__ void histogram_round(const uint32_t (&key)[kTopkPerThread], uint32_t prefix, uint32_t mask,
                                                int shift, int lane, uint32_t *hist) {
#pragma unroll
    for (int j = 0; j < kTopkPerThread; ++j) {
        const bool in = key[j] != kNoKey && (key[j] & mask) == prefix;
        const uint32_t bin = (key[j] >> shift) & 255u;
        const uint32_t active = __ballot_sync(0xffffffffu, in);
        if (in) {
            const uint32_t same = __match_any_sync(active, bin);
            if ((same & ((1u << lane) - 1u)) == 0u) atomicAdd(&hist[bin], (uint32_t)__popc(same));
        }
    }
}

// Dynamic shared memory: two round buffers of scores, then the lane-replicated histogram.
constexpr int kTopkSmemBytes = 2 * kTopkRound * 4 + 256 * 32 * 4;

// The same histogram with one counter per (bin, lane): hrep[bin * 32 + lane]. One
// shared atomic per key and no warp aggregation; a warp's 32 atomics go to 32 banks.
// Cheaper than histogram_round when most keys are in play (the first two passes).
__device__ __forceinline__ void histogram_lanes(const uint32_t (&key)[kTopkPerThread], uint32_t prefix, uint32_t mask,
                                                int shift, int lane, uint32_t *hrep) {
#pragma unroll
    for (int j = 0; j < kTopkPerThread; ++j) {
        if (key[j] != kNoKey && (key[j] & mask) == prefix) atomicAdd(&hrep[((key[j] >> shift) & 255u) * 32 + lane], 1u);
    }
}

__device__ __forceinline__ int4 ld_nc_v4_sel(const void *ptr) {
    int4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr));
    return v;
}

__global__ void __launch_bounds__(kTopkThreads) select_topk_kernel(const TopkParams p) {
    extern __shared__ __align__(16) float s_keys[];
    __shared__ __align__(8) uint64_t s_bar[2];
    __shared__ uint32_t hist[2][256];  // pass p uses hist[p & 1]
    __shared__ uint32_t s_bin[2], s_rem[2];
    __shared__ int32_t s_gt[kTopkMaxRounds * kTopkWarps], s_eq[kTopkMaxRounds * kTopkWarps];

    const int kvh = blockIdx.x, b = blockIdx.y;
    const int r = p.req_ids ? p.req_ids[b] : b;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float *row = p.scores + ((int64_t)r * p.hkv + kvh) * p.score_stride + p.sink;
    // The row's first round (at most 16384 candidates) is requested before the length is
    // known, from the row's capacity (score_stride - S) rather than its length: the copy
    // then overlaps the metadata round trip. Every exit below waits for it first.
    const int64_t room = p.score_stride - p.sink;
    const int cap0 = room <= 0 ? 0 : room < kTopkRound ? (int)room : kTopkRound;
    float *const sbuf = s_keys;  // [2][kTopkRound]
    auto copy_span = [&](int base, int len, uintptr_t &a0, uintptr_t &a1) {  // 16-byte-aligned interior
        const uintptr_t a = reinterpret_cast<uintptr_t>(row + base);
        a0 = (a + 15) & ~uintptr_t(15);
        a1 = (a + 4 * (uintptr_t)len) & ~uintptr_t(15);
    };
    if (tid == 0) {
        mbar_init(&s_bar[0], 1);
        mbar_init(&s_bar[1], 1);
        fence_barrier_init();
        uintptr_t a0, a1;
        copy_span(0, cap0, a0, a1);
        if (a1 > a0) {
            mbar_arrive_expect_tx(&s_bar[0], (uint32_t)(a1 - a0));
            bulk_load_1d(sbuf, reinterpret_cast<const void *>(a0), (uint32_t)(a1 - a0), &s_bar[0]);
        } else {
            mbar_arrive(&s_bar[0]);
        }
    }
    __syncthreads();
    auto drain = [&]() { mbar_wait_warp(&s_bar[0], 0); };  // the first copy has landed (bounded)
    const int L = p.seq_lens[r];
    if (L < 0 || L > p.score_stride) {
        if (tid == 0 && kvh == 0) report(p.dev_status, SFI_DEV_BAD_LEN);
        drain();
        return;
    }
    const int n = max(0, L - p.recent - p.sink);  // |C|, C = [S, L - W)
    const int k = p.k_per_req[r];
    const int rounds = (n + kTopkRound - 1) / kTopkRound;
    if (k < 0 || k > p.k_cap || rounds > kTopkMaxRounds) {
        if (tid == 0 && kvh == 0) report(p.dev_status, SFI_DEV_K_OVERFLOW);
        drain();
        return;
    }
    const int keff = min(k, n);
    if (kvh == 0 && tid == 0) p.count_out[r] = keff;
    int32_t *out = p.idx_out + ((int64_t)r * p.hkv + kvh) * p.k_cap;
    if (keff == n) {  // everything is selected
        for (int i = tid; i < n; i += kTopkThreads) out[i] = p.sink + i;
    }
    if (keff == 0 || keff == n) {
        drain();
        return;
    }

    // Rounds of 16384 candidates come into shared memory by TMA bulk copies (each
    // copy covers the round's 16-byte-aligned interior and never leaves the row; the
    // few floats outside are read directly). One round: its keys stay in registers for
    // the whole selection. Two rounds: both stay in the two buffers. More: every use of
    // a round (4 radix passes, the counts, the output) streams through the two buffers,
    // the next copy in flight while the current round is read.
    uint32_t *hrep = reinterpret_cast<uint32_t *>(s_keys + 2 * kTopkRound);  // [256][32] lane counters
    const int total_uses = 6 * rounds;
    auto issue = [&](int b, int rd) {  // thread 0: copy round rd into buffer b
        const int base = rd * kTopkRound, len = min(kTopkRound, n - base);
        uintptr_t a0, a1;
        copy_span(base, len, a0, a1);
        if (a1 > a0) {
            mbar_arrive_expect_tx(&s_bar[b], (uint32_t)(a1 - a0));
            bulk_load_1d(sbuf + b * kTopkRound, reinterpret_cast<const void *>(a0), (uint32_t)(a1 - a0), &s_bar[b]);
        } else {
            mbar_arrive(&s_bar[b]);
        }
    };
    uint32_t key[kTopkPerThread];
    auto fetch = [&](int u) -> bool {  // this thread's keys of use u: round u % rounds, buffer u & 1
        const int rd = u % rounds, b = u & 1, base = rd * kTopkRound, len = min(kTopkRound, n - base);
        if ((rounds != 2 || u < 2) && !mbar_wait_warp(&s_bar[b], (u >> 1) & 1)) return false;
        const uintptr_t a = reinterpret_cast<uintptr_t>(row + base);
        uintptr_t a0, a1;
        copy_span(base, len, a0, a1);  // (the early copy of round 0 covers at least this span)
        const int lo_i = (int)((a0 - a) >> 2);  // row[base + i], lo_i <= i < hi_i, is sbuf[b][i - lo_i]
        const int hi_i = a1 > a0 ? (int)((a1 - a) >> 2) : lo_i;
        const float *bb = sbuf + b * kTopkRound;
#pragma unroll
        for (int j = 0; j < kTopkPerThread; ++j) {
            const int i = warp * (32 * kTopkPerThread) + 32 * j + lane;
            key[j] = i < len ? order_key(i >= lo_i && i < hi_i ? bb[i - lo_i] : __ldg(row + base + i)) : kNoKey;
        }
        return true;
    };
    auto release = [&](int u) {  // every thread has read use u: refill its buffer with use u + 2
        if (rounds >= 3 && u + 2 < total_uses) {
            __syncthreads();
            if (tid == 0) issue(u & 1, (u + 2) % rounds);
        }
    };
    if (tid == 0 && rounds > 1) issue(1, 1);  // round 0 is already on its way
    int use = 0;
    if (rounds == 1) {  // resident in registers for the whole selection
        if (!fetch(use++)) {
            if (lane == 0) report(p.dev_status, SFI_DEV_TIMEOUT);
            return;
        }
    }

    // ---- radix select of the keff-th largest key ----
    // Double-buffered bins and results: pass p clears hist[(p + 1) & 1] for the next pass
    // (its last reader, pass p - 1's scan, is behind every thread) and the lane counters
    // are cleared as they are summed, so each pass needs no barrier of its own for that.
    uint32_t prefix = 0u, mask = 0u;
    uint32_t rem = (uint32_t)keff;  // how many still to take inside the current prefix
    for (int i = tid; i < 256 * 32; i += kTopkThreads) hrep[i] = 0u;
    __syncthreads();
    int pass = 0;
    for (int shift = 24; shift >= 0; shift -= 8, ++pass) {
        const bool lanes = shift >= 16;
        uint32_t *const hcur = hist[pass & 1];
        if (tid < 256) hist[(pass + 1) & 1][tid] = 0u;
        if (rounds == 1) {
            if (lanes) histogram_lanes(key, prefix, mask, shift, lane, hrep);
            else histogram_round(key, prefix, mask, shift, lane, hcur);
        } else {
            for (int rd = 0; rd < rounds; ++rd) {
                if (!fetch(use)) {
                    if (lane == 0) report(p.dev_status, SFI_DEV_TIMEOUT);
                    return;
                }
                if (lanes) histogram_lanes(key, prefix, mask, shift, lane, hrep);
                else histogram_round(key, prefix, mask, shift, lane, hcur);
                release(use++);
            }
        }
        __syncthreads();
        if (lanes) {  // bin b = sum of its 32 lane counters (rotated: a warp's reads hit 32 banks), cleared
            if (tid < 256) {
                uint32_t sum = 0u;
#pragma unroll 8
                for (int l = 0; l < 32; ++l) {
                    const int i = tid * 32 + ((l + tid) & 31);
                    sum += hrep[i];
                    hrep[i] = 0u;
                }
                hcur[tid] = sum;
            }
            __syncthreads();
        }
        if (warp == 0) {
            // lane l owns bins 255-8l .. 248-8l (from the top)
            uint32_t c[8];
            uint32_t sum = 0u;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = hcur[255 - 8 * lane - j];
                sum += c[j];
            }
            uint32_t incl = sum;  // inclusive prefix over lanes (from the top bins)
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            const uint32_t excl = incl - sum;
            const bool here = excl < rem && rem <= incl;
            const uint32_t who = __ballot_sync(0xffffffffu, here);
            if (lane == __ffs(who) - 1) {
                uint32_t above = excl;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (above + c[j] >= rem) {
                        s_bin[pass & 1] = 255u - 8u * lane - j;
                        s_rem[pass & 1] = rem - above;
                        break;
                    }
                    above += c[j];
                }
            }
        }
        __syncthreads();
        prefix |= s_bin[pass & 1] << shift;
        mask |= 255u << shift;
        rem = s_rem[pass & 1];
    }
    const uint32_t tau = prefix;
    const int take_eq = (int)rem;  // keys equal to tau to take, lowest positions first

    // ---- ascending output: counts per (round, warp), scan, then ranked writes ----
    for (int rd = 0; rd < rounds; ++rd) {
        if (rounds > 1 && !fetch(use)) {
            if (lane == 0) report(p.dev_status, SFI_DEV_TIMEOUT);
            return;
        }
        unsigned gt_l = 0, eq_l = 0;  // this lane's counts, then summed over the warp
#pragma unroll
        for (int j = 0; j < kTopkPerThread; ++j) {
            gt_l += (key[j] != kNoKey && key[j] > tau) ? 1u : 0u;
            eq_l += key[j] == tau ? 1u : 0u;
        }
        const int gt = (int)__reduce_add_sync(0xffffffffu, gt_l);
        const int eq = (int)__reduce_add_sync(0xffffffffu, eq_l);
        if (lane == 0) {
            s_gt[rd * kTopkWarps + warp] = gt;
            s_eq[rd * kTopkWarps + warp] = eq;
        }
        if (rounds > 1) release(use++);
    }
    __syncthreads();
    if (warp == 0) {  // exclusive scan over (round, warp) in position order
        int carry_gt = 0, carry_eq = 0;
        const int entries = rounds * kTopkWarps;
        for (int base = 0; base < entries; base += 32) {
            const bool have = base + lane < entries;
            const int a0 = have ? s_gt[base + lane] : 0, e0 = have ? s_eq[base + lane] : 0;
            int a = a0, e = e0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int va = __shfl_up_sync(0xffffffffu, a, off);
                const int ve = __shfl_up_sync(0xffffffffu, e, off);
                if (lane >= off) {
                    a += va;
                    e += ve;
                }
            }
            if (have) {
                s_gt[base + lane] = carry_gt + a - a0;
                s_eq[base + lane] = carry_eq + e - e0;
            }
            carry_gt += __shfl_sync(0xffffffffu, a, 31);
            carry_eq += __shfl_sync(0xffffffffu, e, 31);
        }
    }
    __syncthreads();
    const uint32_t lt_mask = (1u << lane) - 1u;
    // With one round the selection (keff < n <= 16384 positions) is assembled in shared
    // memory (s_keys is free by now) and written out with one coalesced pass.
    int32_t *dst = rounds == 1 ? reinterpret_cast<int32_t *>(s_keys) : out;
    for (int rd = 0; rd < rounds; ++rd) {
        if (rounds > 1 && !fetch(use)) {
            if (lane == 0) report(p.dev_status, SFI_DEV_TIMEOUT);
            return;
        }
        int eq_before = s_eq[rd * kTopkWarps + warp];
        int out_pos = s_gt[rd * kTopkWarps + warp] + min(eq_before, take_eq);
        bool ties = false;  // does this warp hold keys equal to tau in this round?
#pragma unroll
        for (int j = 0; j < kTopkPerThread; ++j) ties |= key[j] == tau;
        if (!__any_sync(0xffffffffu, ties)) {  // common case: take exactly the keys above tau
#pragma unroll
            for (int j = 0; j < kTopkPerThread; ++j) {
                const bool take = key[j] != kNoKey && key[j] > tau;
                const uint32_t take_bal = __ballot_sync(0xffffffffu, take);
                if (take)
                    dst[out_pos + __popc(take_bal & lt_mask)] =
                        p.sink + rd * kTopkRound + warp * (32 * kTopkPerThread) + 32 * j + lane;
                out_pos += __popc(take_bal);
            }
        } else {
#pragma unroll
            for (int j = 0; j < kTopkPerThread; ++j) {
                const bool valid = key[j] != kNoKey;
                const bool is_eq = valid && key[j] == tau;
                const uint32_t eq_bal = __ballot_sync(0xffffffffu, is_eq);
                const int eq_rank = eq_before + __popc(eq_bal & lt_mask);
                const bool take = valid && (key[j] > tau || (is_eq && eq_rank < take_eq));
                const uint32_t take_bal = __ballot_sync(0xffffffffu, take);
                if (take)
                    dst[out_pos + __popc(take_bal & lt_mask)] =
                        p.sink + rd * kTopkRound + warp * (32 * kTopkPerThread) + 32 * j + lane;
                out_pos += __popc(take_bal);
                eq_before += __popc(eq_bal);
            }
        }
        if (rounds > 1) release(use++);
    }
    __syncthreads();  // the selection is complete (in shared memory, or in `out` for long rows)
    if (rounds == 1)
        for (int i = tid; i < keff; i += kTopkThreads) out[i] = dst[i];
}

cudaError_t launch_select_topk(const TopkParams &p, int batch, cudaStream_t stream) {
    // The shared-memory opt-in is a per-device function attribute: set it once per device.
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
    if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(select_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTopkSmemBytes);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    dim3 grid(p.hkv, batch);
    select_topk_kernel<<<grid, kTopkThreads, kTopkSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace sfi
