// Byte-exact KV copies of the SFI path: the paged append of the newest token(s) and
// the compaction gather that packs sink + selected rows into the compact buffer.
//
// Method: Slow-Fast Inference (Xie et al., 2026), Figure 3 caption: the dense KV is
// kept in pages (recent tokens are read from it in place) and, at a slow step, the
// cache reorganisation packs sink and selected tokens into a contiguous compact
// buffer.
//
// Both kernels are pure HBM copies of 16-byte chunks. The compaction reads rows
// scattered over the page pool (each row D*2 bytes, i.e. whole 32-byte sectors) and
// writes them contiguously; every thread keeps kIters independent loads in flight
// before its stores.
#include "sfi_device.cuh"
#include "sfi_internal.h"

namespace sfi {

constexpr int kCopyThreads = 256;
constexpr int kCompactRowsPerCta = 64;
// Requests handled by one compaction launch (the chunk prefix lives in shared memory).
constexpr int kCompactMaxBatch = 512;

__device__ __forceinline__ int4 ld_nc_v4(const void *p) {
    int4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(void *p, int4 v) {
    asm volatile("st.global.v4.s32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Append of the p.tokens newest tokens of each request: token t goes to position
// L - tokens + t (L counts them); k_new/v_new are [request][tokens][Hkv][D].
template <int D>
__global__ void __launch_bounds__(kCopyThreads) paged_append_kernel(const CopyParams p) {
    constexpr int kChunks = D / 8;  // 16-byte chunks per row
    const int b = blockIdx.x;
    const int r = p.req_ids ? p.req_ids[b] : b;
    const int L = p.seq_lens[r];
    const int T = p.tokens;
    if (L < T || L > p.max_pages * kSubTokens) {
        if (threadIdx.x == 0) report(p.dev_status, SFI_DEV_BAD_LEN);
        return;
    }
    const int per_token = 2 * p.hkv * kChunks;
    for (int e = threadIdx.x; e < T * per_token; e += kCopyThreads) {
        const int tt = e / per_token, f0 = e - tt * per_token;
        const bool is_v = f0 >= p.hkv * kChunks;
        const int f = is_v ? f0 - p.hkv * kChunks : f0;
        const int kv = f / kChunks, c = f - (f / kChunks) * kChunks;
        const int pos = L - T + tt;
        const int page = p.page_table[(int64_t)r * p.max_pages + pos / kSubTokens];
        if (page < 0 || page >= p.num_pages) {
            report(p.dev_status, SFI_DEV_BAD_PAGE);
            continue;
        }
        const __nv_bfloat16 *src = (is_v ? p.v_new : p.k_new) + (((int64_t)r * T + tt) * p.hkv + kv) * D + c * 8;
        __nv_bfloat16 *dst = (is_v ? p.v_pool_dst : p.k_pool_dst) +
                             (((int64_t)page * p.hkv + kv) * kSubTokens + pos % kSubTokens) * D + c * 8;
        st_v4(dst, *reinterpret_cast<const int4 *>(src));
    }
}

// Rows a request's compaction writes per KV head: the sink [0, min(S, L)) and, when
// L >= S, the selection [S, S + count). -1 marks a request with invalid arguments
// (the reason is ORed into *err).
__device__ __forceinline__ int compact_rows(const CopyParams &p, int r, uint32_t *err) {
    const int L = p.seq_lens[r];
    if (L < 1 || L > p.max_pages * kSubTokens) {
        *err |= SFI_DEV_BAD_LEN;
        return -1;
    }
    const int cnt = p.count[r];
    const int cap = p.c_capacity[r];
    const int64_t off = p.c_row_offset[r];
    if (cnt < 0 || cnt > p.k_cap || p.sink + cnt > cap || (cnt > 0 && L < p.sink)) {
        *err |= SFI_DEV_K_OVERFLOW;
        return -1;
    }
    if (off < 0 || off + (int64_t)p.hkv * cap > p.c_total_rows) {
        *err |= SFI_DEV_BAD_COMPACT;
        return -1;
    }
    return L < p.sink ? L : p.sink + cnt;
}

// Persistent grid: every CTA derives the same list of 64-row chunks from the device
// counts (an exclusive prefix over the launch's requests, in shared memory) and walks
// it with a grid stride, so the work follows the rows actually selected, not k_cap.
template <int D>
__global__ void __launch_bounds__(kCopyThreads, 3) compact_gather_kernel(const CopyParams p, int b_begin, int nb) {
    constexpr int kChunks = D / 8;
    constexpr int kThreadsPerRow = 2 * kChunks;  // K chunks then V chunks
    constexpr int kRowsPerIter = kCopyThreads / kThreadsPerRow;
    constexpr int kIters = kCompactRowsPerCta / kRowsPerIter;
    constexpr int kWarps = kCopyThreads / 32;
    __shared__ int s_prefix[kCompactMaxBatch];  // first chunk of each request entry
    __shared__ int s_rows[kCompactMaxBatch];    // rows per KV head of each request entry
    __shared__ int s_len[kCompactMaxBatch];     // L, selected count and capacity of each entry
    __shared__ int s_cnt[kCompactMaxBatch];
    __shared__ int s_cap[kCompactMaxBatch];
    __shared__ long long s_off[kCompactMaxBatch];
    __shared__ int s_warp[kWarps];
    __shared__ int s_total;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t err = 0;
    int carry = 0;
    for (int base = 0; base < nb; base += kCopyThreads) {
        const int b = base + tid;
        int c = 0, rows = -1;
        if (b < nb) {
            const int r = p.req_ids ? p.req_ids[b_begin + b] : b_begin + b;
            rows = compact_rows(p, r, &err);
            c = rows > 0 ? p.hkv * ((rows + kCompactRowsPerCta - 1) / kCompactRowsPerCta) : 0;
        }
        int incl = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        if (lane == 31) s_warp[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int w = lane < kWarps ? s_warp[lane] : 0;
            int wi = w;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, wi, off);
                if (lane >= off) wi += v;
            }
            if (lane < kWarps) s_warp[lane] = wi - w;
            if (lane == 31) s_total = wi;
        }
        __syncthreads();
        if (b < nb) {
            s_prefix[b] = carry + s_warp[warp] + incl - c;
            s_rows[b] = rows;
            if (rows > 0) {  // compact_rows has validated these
                const int r = p.req_ids ? p.req_ids[b_begin + b] : b_begin + b;
                s_len[b] = p.seq_lens[r];
                s_cnt[b] = p.count[r];
                s_cap[b] = p.c_capacity[r];
                s_off[b] = p.c_row_offset[r];
            }
        }
        carry += s_total;
        __syncthreads();
    }
    if (err && blockIdx.x == 0) report(p.dev_status, err);
    const int total = carry;

    const int sub = tid / kThreadsPerRow;
    const int cc = tid - sub * kThreadsPerRow;
    const bool is_v = cc >= kChunks;
    const int chunk = is_v ? cc - kChunks : cc;
    const __nv_bfloat16 *pool = is_v ? p.v_pool_src : p.k_pool_src;
    uint32_t werr = 0;
    for (int work = blockIdx.x; work < total; work += gridDim.x) {
        // request entry owning this chunk: the last b with s_prefix[b] <= work (an entry
        // without chunks shares its prefix with the next entry, so it is never the last)
        int lo = 0, hi = nb - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_prefix[mid] <= work) lo = mid; else hi = mid - 1;
        }
        const int b = lo;
        const int r = p.req_ids ? p.req_ids[b_begin + b] : b_begin + b;
        const int rows = s_rows[b];
        const int per_head = (rows + kCompactRowsPerCta - 1) / kCompactRowsPerCta;
        const int within = work - s_prefix[b];
        const int kvh = within / per_head;
        const int row0 = (within - kvh * per_head) * kCompactRowsPerCta;
        const int L = s_len[b];
        const int ns = min(p.sink, L);
        const int cnt = s_cnt[b];
        const int cap = s_cap[b];
        const int64_t off = s_off[b];
        __nv_bfloat16 *dst_base = (is_v ? p.cv : p.ck) + (off + (int64_t)kvh * cap) * D + chunk * 8;
        const int32_t *sel = p.idx + ((int64_t)r * p.hkv + kvh) * p.k_cap;
        const int32_t *ptab = p.page_table + (int64_t)r * p.max_pages;

        // Three batched phases (all indices, then all page ids, then all rows), so the
        // kIters rows' dependent loads overlap instead of running one row after another;
        // errors are collected in a register and reported once.
        int pos[kIters];
        uint32_t take = 0;  // bit it: row it of this thread is copied
#pragma unroll
        for (int it = 0; it < kIters; ++it) {
            const int i = row0 + it * kRowsPerIter + sub;
            const bool t = i < ns || (i >= p.sink && i < p.sink + cnt);
            take |= (t ? 1u : 0u) << it;
            pos[it] = i < ns ? i : (t ? __ldg(&sel[i - p.sink]) : 0);
        }
        int page[kIters];
#pragma unroll
        for (int it = 0; it < kIters; ++it) {
            if (((take >> it) & 1u) && (pos[it] < 0 || pos[it] >= L)) {
                werr |= SFI_DEV_BAD_INDEX;
                take &= ~(1u << it);
            }
            page[it] = ((take >> it) & 1u) ? __ldg(&ptab[pos[it] / kSubTokens]) : 0;
        }
        int4 vals[kIters];
#pragma unroll
        for (int it = 0; it < kIters; ++it) {
            if (((take >> it) & 1u) && (page[it] < 0 || page[it] >= p.num_pages)) {
                werr |= SFI_DEV_BAD_PAGE;
                take &= ~(1u << it);
            }
            if ((take >> it) & 1u)
                vals[it] = ld_nc_v4(pool + (((int64_t)page[it] * p.hkv + kvh) * kSubTokens + pos[it] % kSubTokens) * D +
                                    chunk * 8);
        }
#pragma unroll
        for (int it = 0; it < kIters; ++it)
            if ((take >> it) & 1u) st_v4(dst_base + (int64_t)(row0 + it * kRowsPerIter + sub) * D, vals[it]);
    }
    if (werr) report(p.dev_status, werr);
}

cudaError_t launch_paged_append(const CopyParams &p, int batch, cudaStream_t stream) {
    if (p.head_dim == 128)
        paged_append_kernel<128><<<batch, kCopyThreads, 0, stream>>>(p);
    else
        paged_append_kernel<64><<<batch, kCopyThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_compact_gather(const CopyParams &p, int batch, int max_rows, cudaStream_t stream) {
    (void)max_rows;  // the grid follows the device counts
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = p.head_dim == 128
                ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, compact_gather_kernel<128>, kCopyThreads, 0)
                : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, compact_gather_kernel<64>, kCopyThreads, 0);
    if (e != cudaSuccess) return e;
    const int grid = sms * (per_sm > 0 ? per_sm : 1);  // one resident wave of persistent CTAs
    for (int b0 = 0; b0 < batch; b0 += kCompactMaxBatch) {
        const int nb = batch - b0 < kCompactMaxBatch ? batch - b0 : kCompactMaxBatch;
        if (p.head_dim == 128)
            compact_gather_kernel<128><<<grid, kCopyThreads, 0, stream>>>(p, b0, nb);
        else
            compact_gather_kernel<64><<<grid, kCopyThreads, 0, stream>>>(p, b0, nb);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace sfi
