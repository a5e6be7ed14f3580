// Single-token attention launches (one query token per request): the fast step, the
// slow step's dense attention with scores, the dense baseline and the mixed launch.
// The kernel template is in attn_kernel.cuh.
#include "attn_kernel.cuh"

namespace sfi {

WorkspaceLayout workspace_layout_slots(int64_t units, int64_t slots, int head_dim, int rows, size_t bytes) {
    WorkspaceLayout w;
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t cnt = up(sizeof(int32_t) * (size_t)units);  // one split counter per unit
    const size_t ml = up(sizeof(float) * 2 * (size_t)rows * (size_t)slots);
    const size_t part = up(sizeof(float) * (size_t)head_dim * (size_t)rows * (size_t)slots);
    w.count_off = 0;
    w.data_bytes = ml + part;
    w.total = cnt + w.data_bytes;
    // The partial states sit at the end of the caller's buffer (right after the counters
    // when it is exactly `total` bytes), so the counters of every call sharing a buffer
    // stay clear of every other call's partial states, whatever their batch sizes.
    const size_t end = bytes >= w.total ? (bytes & ~size_t(255)) : w.total;
    w.part_off = end - part;
    w.ml_off = w.part_off - ml;
    return w;
}

WorkspaceLayout workspace_layout(int64_t units, int splits, int head_dim, int rows, size_t bytes) {
    return workspace_layout_slots(units, units * splits, head_dim, rows, bytes);
}

int attn_cluster_capacity(int size) {
    static std::atomic<int> cache[64][kMaxClusterSplits + 1];
    int dev = 0;
    if (size < 1 || size > kMaxClusterSplits || cudaGetDevice(&dev) != cudaSuccess) return 0;
    const bool cacheable = dev >= 0 && dev < 64;
    if (cacheable) {
        const int v = cache[dev][size].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    using T = AttnTile<128>;
    auto kern = attn_decode_kernel<128, kModeFast, false, true, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmemBytes) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)size);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = T::kSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = (unsigned)size;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();  // leave no error behind for the next launch's check
        return 0;
    }
    if (cacheable && n > 0) cache[dev][size].store(n, std::memory_order_relaxed);
    return n;
}

template <int D, bool CLUSTER>
static cudaError_t launch_mode(int mode, bool with_scores, const AttnMaps &maps, const AttnParams &p, int batch,
                               cudaStream_t stream) {
    if (mode == kModeMixed) return launch_one<D, kModeMixed, true, false, false>(maps, p, batch, stream);
    if (mode == kModeFast) return launch_one<D, kModeFast, false, CLUSTER, false>(maps, p, batch, stream);
    if (with_scores) return launch_one<D, kModeDense, true, CLUSTER, false>(maps, p, batch, stream);
    return launch_one<D, kModeDense, false, CLUSTER, false>(maps, p, batch, stream);
}

cudaError_t launch_attention(int head_dim, int mode, bool with_scores, const AttnMaps &maps, const AttnParams &p,
                             int batch, cudaStream_t stream) {
    const bool cluster = mode != kModeMixed && p.splits > 1 && p.splits <= kMaxClusterSplits;
    if (head_dim == 128)
        return cluster ? launch_mode<128, true>(mode, with_scores, maps, p, batch, stream)
                       : launch_mode<128, false>(mode, with_scores, maps, p, batch, stream);
    return cluster ? launch_mode<64, true>(mode, with_scores, maps, p, batch, stream)
                   : launch_mode<64, false>(mode, with_scores, maps, p, batch, stream);
}

}  // namespace sfi
