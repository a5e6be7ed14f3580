// Byte-exact KV copies of the SFI path: the paged append of the current token and
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

template <int D>
__global__ void __launch_bounds__(kCopyThreads) paged_append_kernel(const CopyParams p) {
    constexpr int kChunks = D / 8;  // 16-byte chunks per row
    const int b = blockIdx.x;
    const int r = p.req_ids ? p.req_ids[b] : b;
    const int L = p.seq_lens[r];
    if (L < 1 || L > p.max_pages * kSubTokens) {
        if (threadIdx.x == 0) report(p.dev_status, SFI_DEV_BAD_LEN);
        return;
    }
    const int pos = L - 1;
    const int page = p.page_table[(int64_t)r * p.max_pages + pos / kSubTokens];
    if (page < 0 || page >= p.num_pages) {
        if (threadIdx.x == 0) report(p.dev_status, SFI_DEV_BAD_PAGE);
        return;
    }
    const int total = 2 * p.hkv * kChunks;
    for (int e = threadIdx.x; e < total; e += kCopyThreads) {
        const bool is_v = e >= p.hkv * kChunks;
        const int f = is_v ? e - p.hkv * kChunks : e;
        const int kv = f / kChunks, c = f - (f / kChunks) * kChunks;
        const __nv_bfloat16 *src = (is_v ? p.v_new : p.k_new) + ((int64_t)r * p.hkv + kv) * D + c * 8;
        __nv_bfloat16 *dst = (is_v ? p.v_pool_dst : p.k_pool_dst) +
                             (((int64_t)page * p.hkv + kv) * kSubTokens + pos % kSubTokens) * D + c * 8;
        st_v4(dst, *reinterpret_cast<const int4 *>(src));
    }
}

template <int D>
__global__ void __launch_bounds__(kCopyThreads) compact_gather_kernel(const CopyParams p) {
    constexpr int kChunks = D / 8;
    constexpr int kThreadsPerRow = 2 * kChunks;  // K chunks then V chunks
    constexpr int kRowsPerIter = kCopyThreads / kThreadsPerRow;
    constexpr int kIters = kCompactRowsPerCta / kRowsPerIter;
    const int kvh = blockIdx.y, b = blockIdx.z;
    const int r = p.req_ids ? p.req_ids[b] : b;
    const int L = p.seq_lens[r];
    const bool lead = threadIdx.x == 0 && blockIdx.x == 0 && kvh == 0;
    if (L < 1 || L > p.max_pages * kSubTokens) {
        if (lead) report(p.dev_status, SFI_DEV_BAD_LEN);
        return;
    }
    const int cnt = p.count[r];
    const int cap = p.c_capacity[r];
    const int64_t off = p.c_row_offset[r];
    if (cnt < 0 || cnt > p.k_cap || p.sink + cnt > cap || (cnt > 0 && L < p.sink)) {
        if (lead) report(p.dev_status, SFI_DEV_K_OVERFLOW);
        return;
    }
    if (off < 0 || off + (int64_t)p.hkv * cap > p.c_total_rows) {
        if (lead) report(p.dev_status, SFI_DEV_BAD_COMPACT);
        return;
    }
    const int ns = min(p.sink, L);
    const int sub = threadIdx.x / kThreadsPerRow;
    const int c = threadIdx.x - sub * kThreadsPerRow;
    const bool is_v = c >= kChunks;
    const int chunk = is_v ? c - kChunks : c;
    const __nv_bfloat16 *pool = is_v ? p.v_pool_src : p.k_pool_src;
    __nv_bfloat16 *dst_base = (is_v ? p.cv : p.ck) + (off + (int64_t)kvh * cap) * D + chunk * 8;
    const int32_t *sel = p.idx + ((int64_t)r * p.hkv + kvh) * p.k_cap;
    const int32_t *ptab = p.page_table + (int64_t)r * p.max_pages;

    int4 vals[kIters];
    int rows[kIters];
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
        const int i = blockIdx.x * kCompactRowsPerCta + it * kRowsPerIter + sub;
        int pos = -1;
        if (i < ns) {
            pos = i;
        } else if (i >= p.sink && i < p.sink + cnt) {
            pos = sel[i - p.sink];
            if (pos < 0 || pos >= L) {
                report(p.dev_status, SFI_DEV_BAD_INDEX);
                pos = -1;
            }
        }
        rows[it] = -1;
        if (pos >= 0) {
            const int page = ptab[pos / kSubTokens];
            if (page < 0 || page >= p.num_pages) {
                report(p.dev_status, SFI_DEV_BAD_PAGE);
            } else {
                vals[it] = ld_nc_v4(pool + (((int64_t)page * p.hkv + kvh) * kSubTokens + pos % kSubTokens) * D +
                                    chunk * 8);
                rows[it] = i;
            }
        }
    }
#pragma unroll
    for (int it = 0; it < kIters; ++it)
        if (rows[it] >= 0) st_v4(dst_base + (int64_t)rows[it] * D, vals[it]);
}

cudaError_t launch_paged_append(const CopyParams &p, int batch, cudaStream_t stream) {
    if (p.head_dim == 128)
        paged_append_kernel<128><<<batch, kCopyThreads, 0, stream>>>(p);
    else
        paged_append_kernel<64><<<batch, kCopyThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_compact_gather(const CopyParams &p, int batch, int max_rows, cudaStream_t stream) {
    dim3 grid((max_rows + kCompactRowsPerCta - 1) / kCompactRowsPerCta, p.hkv, batch);
    if (p.head_dim == 128)
        compact_gather_kernel<128><<<grid, kCopyThreads, 0, stream>>>(p);
    else
        compact_gather_kernel<64><<<grid, kCopyThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace sfi
