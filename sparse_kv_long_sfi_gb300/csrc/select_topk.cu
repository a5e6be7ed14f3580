// Selector of the SFI slow step: per (request, KV head) top-k over the masked
// candidate logits, ties to the lower position, result in ascending position order.
//
// Method: Slow-Fast Inference (Xie et al., 2026), Figure 2 caption (the Selector
// refreshes the selected memory from the masked logits collected by the slow step).
//
// Design: one CTA of 1024 threads per (request, KV head).
//  * Scores are mapped to order-preserving uint32 keys (-0 -> +0, NaN -> 0, below
//    -inf).
//  * Radix select, 4 passes of 8 bits from the top: a 256-bin shared histogram of the
//    keys that share the current prefix (warp-aggregated atomics via match.any),
//    then one warp scans the bins from the top to find the bin holding the k-th key.
//    The result is the exact k-th largest key tau and the number of keys equal to
//    tau that must be taken (the lowest positions among them).
//  * Output in ascending position order without sorting: each warp owns a
//    contiguous range of candidates; a counting pass gives per-warp (above tau,
//    equal tau) totals, a scan gives each warp's output offset and tie rank, and a
//    second pass writes positions with ballot/popc prefix counts.
// The candidates of a slow step are a few K to 128K floats, read from L2 for every
// pass after the first.
#include "sfi_device.cuh"
#include "sfi_internal.h"

namespace sfi {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;

__device__ __forceinline__ uint32_t order_key(float x) {
    uint32_t u = __float_as_uint(x);
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;  // NaN ranks below everything
    if (u == 0x80000000u) u = 0u;                    // -0 == +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kTopkThreads) select_topk_kernel(const TopkParams p) {
    __shared__ uint32_t hist[256];
    __shared__ uint32_t s_bin, s_rem;
    __shared__ int32_t w_gt[kTopkWarps], w_eq[kTopkWarps];

    const int kvh = blockIdx.x, b = blockIdx.y;
    const int r = p.req_ids ? p.req_ids[b] : b;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int L = p.seq_lens[r];
    if (L < 0 || L > p.score_stride) {
        if (tid == 0 && kvh == 0) report(p.dev_status, SFI_DEV_BAD_LEN);
        return;
    }
    const int n = max(0, L - p.recent - p.sink);  // |C|, C = [S, L - W)
    const int k = p.k_per_req[r];
    if (k < 0 || k > p.k_cap) {
        if (tid == 0 && kvh == 0) report(p.dev_status, SFI_DEV_K_OVERFLOW);
        return;
    }
    const int keff = min(k, n);
    if (kvh == 0 && tid == 0) p.count_out[r] = keff;
    if (keff == 0) return;
    int32_t *out = p.idx_out + ((int64_t)r * p.hkv + kvh) * p.k_cap;
    const float *row = p.scores + ((int64_t)r * p.hkv + kvh) * p.score_stride + p.sink;
    if (keff == n) {  // everything is selected
        for (int i = tid; i < n; i += kTopkThreads) out[i] = p.sink + i;
        return;
    }

    // ---- radix select of the keff-th largest key ----
    uint32_t prefix = 0u, mask = 0u;
    uint32_t rem = (uint32_t)keff;  // how many still to take inside the current prefix
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0u;
        __syncthreads();
        const int n_round = (n + 31) & ~31;  // whole warps iterate together for match.any
        for (int i = tid; i < n_round; i += kTopkThreads) {
            bool in = false;
            uint32_t bin = 0u;
            if (i < n) {
                const uint32_t key = order_key(__ldg(row + i));
                in = (key & mask) == prefix;
                bin = (key >> shift) & 255u;
            }
            const uint32_t active = __ballot_sync(0xffffffffu, in);
            if (in) {
                const uint32_t same = __match_any_sync(active, bin);
                if ((same & ((1u << lane) - 1u)) == 0u) atomicAdd(&hist[bin], (uint32_t)__popc(same));
            }
        }
        __syncthreads();
        if (warp == 0) {
            // lane l owns bins 255-8l .. 248-8l (from the top)
            uint32_t c[8];
            uint32_t sum = 0u;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = hist[255 - 8 * lane - j];
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
                        s_bin = 255u - 8u * lane - j;
                        s_rem = rem - above;
                        break;
                    }
                    above += c[j];
                }
            }
        }
        __syncthreads();
        prefix |= s_bin << shift;
        mask |= 255u << shift;
        rem = s_rem;
        __syncthreads();
    }
    const uint32_t tau = prefix;
    const int take_eq = (int)rem;  // keys equal to tau to take, lowest positions first

    // ---- ascending output ----
    const int per_warp = (((n + kTopkWarps - 1) / kTopkWarps) + 31) & ~31;
    const int w_lo = warp * per_warp;
    const int w_hi = min(n, w_lo + per_warp);
    int gt = 0, eq = 0;
    for (int base = w_lo; base < w_hi; base += 32) {
        const int i = base + lane;
        uint32_t key = 0u;
        if (i < w_hi) key = order_key(__ldg(row + i));
        const bool valid = i < w_hi;
        gt += __popc(__ballot_sync(0xffffffffu, valid && key > tau));
        eq += __popc(__ballot_sync(0xffffffffu, valid && key == tau));
    }
    if (lane == 0) {
        w_gt[warp] = gt;
        w_eq[warp] = eq;
    }
    __syncthreads();
    if (warp == 0) {
        int a = w_gt[lane], e = w_eq[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int va = __shfl_up_sync(0xffffffffu, a, off);
            const int ve = __shfl_up_sync(0xffffffffu, e, off);
            if (lane >= off) {
                a += va;
                e += ve;
            }
        }
        w_gt[lane] = a - w_gt[lane];  // exclusive
        w_eq[lane] = e - w_eq[lane];
    }
    __syncthreads();
    int eq_before = w_eq[warp];
    int out_pos = w_gt[warp] + min(eq_before, take_eq);
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int base = w_lo; base < w_hi; base += 32) {
        const int i = base + lane;
        const bool valid = i < w_hi;
        const uint32_t key = valid ? order_key(__ldg(row + i)) : 0u;
        const bool is_eq = valid && key == tau;
        const uint32_t eq_bal = __ballot_sync(0xffffffffu, is_eq);
        const int eq_rank = eq_before + __popc(eq_bal & lt_mask);
        const bool take = valid && (key > tau || (is_eq && eq_rank < take_eq));
        const uint32_t take_bal = __ballot_sync(0xffffffffu, take);
        if (take) out[out_pos + __popc(take_bal & lt_mask)] = p.sink + i;
        out_pos += __popc(take_bal);
        eq_before += __popc(eq_bal);
    }
}

cudaError_t launch_select_topk(const TopkParams &p, int batch, cudaStream_t stream) {
    dim3 grid(p.hkv, batch);
    select_topk_kernel<<<grid, kTopkThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace sfi
