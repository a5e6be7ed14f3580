// Fast-step attention for callers that cannot allocate device memory.
//
// sfi_fast_decode_attn needs a caller-provided workspace for its split-KV partial
// results. Some callers have no way to provide one: a plugin running inside a host
// application that owns every device allocation, or a latency-critical path that
// must not call cudaMalloc (which can synchronise the whole device). This entry
// point keeps that scratch in a fixed-size array in the library's own device
// memory instead, so it allocates nothing at any time.
#include <atomic>
#include <mutex>

#include "sfi_internal.h"

namespace {

constexpr size_t kScratchBytes = SFI_NOALLOC_SCRATCH_BYTES;

// The scratch itself. Every GPU that loads the library holds these bytes until the
// process exits; all calls on a device share them.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_addr[kMaxDevices];
std::mutex g_setup_mutex;

// Device address of g_noalloc_scratch on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once per
// device with that device current.
sfi_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SFI_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SFI_ERR_UNSUPPORTED;
    void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        p = g_scratch_addr[dev].load(std::memory_order_acquire);
        if (!p) {
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SFI_ERR_CUDA;
            g_scratch_addr[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return SFI_OK;
}

}  // namespace

extern "C" sfi_status sfi_fast_decode_attn_noalloc(const sfi_attn_shape *shape, const sfi_paged_kv *kv,
                                                   const sfi_compact_kv *compact, int32_t sink, int32_t recent,
                                                   const void *q, const void *k_new, const void *v_new, float *out,
                                                   float *lse, const int32_t *req_ids,
                                                   int32_t batch, int32_t max_tokens, int32_t num_splits,
                                                   uint32_t flags, int32_t *dev_status, void *stream) {
    if (!shape || batch < 0 || num_splits < 0) return SFI_ERR_INVALID_ARG;
    // The scratch the inner call will use: the chunked plan's under SFI_ATTN_RAGGED,
    // the regular split plan's otherwise (0 when the splits merge inside a cluster).
    const bool ragged = (flags & SFI_ATTN_RAGGED) != 0;
    const size_t need = ragged ? sfi_mixed_workspace_size(shape, batch, 0, max_tokens, 0)
                               : sfi_workspace_size(shape, batch, max_tokens, num_splits);
    if (need > kScratchBytes) return SFI_ERR_WORKSPACE;  // the plan needs more than the fixed scratch
    void *scratch = nullptr;
    sfi_status st = scratch_address(&scratch);
    if (st != SFI_OK) return st;
    if (need > 0) {
        // Both plans start the scratch with one split counter per (request, KV head),
        // which must be zero; the array keeps whatever the last call (on any stream)
        // left in it.
        const sfi::WorkspaceLayout l = sfi::workspace_layout_slots((int64_t)batch * shape->num_kv_heads, 0,
                                                                   shape->head_dim);
        if (cudaMemsetAsync(static_cast<char *>(scratch) + l.count_off, 0, l.ml_off - l.count_off,
                            static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return SFI_ERR_CUDA;
    }
    return sfi_fast_decode_attn(shape, kv, compact, sink, recent, q, k_new, v_new, out, lse, req_ids, batch,
                                max_tokens, num_splits, flags, scratch, kScratchBytes, dev_status, stream);
}
