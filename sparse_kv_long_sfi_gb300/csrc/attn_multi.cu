// Multi-token attention launches ("A Sparse Glimpse of the Whole: Train-Free
// Self-Speculative Decoding", abstract): p.tokens query tokens per request over the
// sparse state (drafting) or over the whole context with the recycled statistics
// (verification). The kernel template is in attn_kernel.cuh; rows = tokens x G <= 16.
#include "attn_kernel.cuh"

namespace sfi {

template <int D, bool CLUSTER>
static cudaError_t launch_multi_mode(int mode, const AttnMaps &maps, const AttnParams &p, int batch,
                                     cudaStream_t stream) {
    if (mode == kModeFast) return launch_one<D, kModeFast, false, CLUSTER, true>(maps, p, batch, stream);
    return launch_one<D, kModeDense, true, CLUSTER, true>(maps, p, batch, stream);  // scores may be null
}

cudaError_t launch_attention_multi(int head_dim, int mode, const AttnMaps &maps, const AttnParams &p, int batch,
                                   cudaStream_t stream) {
    const bool cluster = p.splits > 1 && p.splits <= kMaxClusterSplits;
    if (head_dim == 128)
        return cluster ? launch_multi_mode<128, true>(mode, maps, p, batch, stream)
                       : launch_multi_mode<128, false>(mode, maps, p, batch, stream);
    return cluster ? launch_multi_mode<64, true>(mode, maps, p, batch, stream)
                   : launch_multi_mode<64, false>(mode, maps, p, batch, stream);
}

}  // namespace sfi
