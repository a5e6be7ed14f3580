// Internal interface between the C ABI layer (sfi_api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sfi.h"

namespace sfi {

// Tokens per sub-block: one page of the paged pool, one unit of TMA work, one
// mma.sync n-extent pair for a consumer warp.
constexpr int kSubTokens = 16;
// Consumer warps per attention CTA (each owns one sub-block of every stage).
constexpr int kConsumerWarps = 4;
// Rows of the query tile handled per (request, KV head): G <= 8 query heads share a KV head.
constexpr int kMaxGroup = 8;
// Query rows of one (request, KV head) unit in the multi-token kernels: tokens x G <= 16
// fill the whole M = 16 tile.
constexpr int kMaxRows = 16;
// Attention CTAs resident per SM (shared memory sized for this).
constexpr int kAttnCtasPerSm = 2;
// Splits of one unit that merge inside a thread-block cluster (portable cluster size);
// more splits merge through the global workspace.
constexpr int kMaxClusterSplits = 8;

// kModeMixed: one launch where each request is either fast (fast_ids) or slow
// (slow_ids: dense attention with scores); 1-D grid of work items.
enum AttnMode : int { kModeFast = 0, kModeDense = 1, kModeMixed = 2 };

struct AttnParams {
    const __nv_bfloat16 *q;  // [B][tokens][Hq][D]
    float *out;              // [B][tokens][Hq][D]
    float *lse;              // [B][tokens][Hq] or null
    float *scores;           // [B][Hkv][score_stride] or null
    int64_t score_stride;
    const int32_t *page_table;
    int32_t max_pages;
    int32_t num_pages;
    const int32_t *seq_lens;
    const int64_t *c_row_offset;
    const int32_t *c_capacity;
    const int32_t *c_count;
    int64_t c_total_rows;
    const int32_t *req_ids;
    int32_t hq, hkv, group;
    int32_t sink, recent;
    float scale;       // softmax scale
    float scale_log2;  // scale * log2(e)
    int32_t splits;
    // query tokens per request (positions L - tokens .. L - 1) and tile rows tokens x group
    int32_t tokens, rows;
    // mixed mode: request lists and per-mode split counts
    const int32_t *fast_ids;
    const int32_t *slow_ids;
    int32_t n_fast, n_slow, fast_splits, slow_splits;
    // sub-blocks per split in mixed mode (0: the mode's units split evenly into *_splits)
    int32_t fast_chunk_sb, slow_chunk_sb;
    int32_t early_prefetch;  // SFI_ATTN_EARLY_KV_PREFETCH: stream KV before the dependency wait
    int32_t withhold;        // SFI_ATTN_TEST_WITHHOLD: 1 + the stage whose copies are never issued (0 = none)
    // fused append of the current token (position L - 1), or null
    const __nv_bfloat16 *k_new;  // [B][Hkv][D]
    const __nv_bfloat16 *v_new;
    __nv_bfloat16 *k_pool_w;     // the paged pools, for the append's writes
    __nv_bfloat16 *v_pool_w;
    int32_t *ws_count;  // [units]
    float *ws_ml;       // [units][splits][rows per slot][2]
    float *ws_part;     // [units][splits][rows per slot][D]
    int32_t *dev_status;
};

struct AttnMaps {
    CUtensorMap pool_k, pool_v;  // rows = (page * Hkv + kv) * P + slot
    CUtensorMap comp_k, comp_v;  // rows = compact buffer rows (dummy copies of pool maps in dense mode)
};

// Workspace layout for `units` (request, KV head) pairs and `splits` splits: the split
// counters at the start, the partial states (data_bytes) at the end of a buffer of
// `bytes` bytes (0: exactly `total`).
struct WorkspaceLayout {
    size_t count_off, ml_off, part_off, data_bytes, total;
};
// Single-token launches keep kMaxGroup rows per partial slot, multi-token ones kMaxRows.
WorkspaceLayout workspace_layout(int64_t units, int splits, int head_dim, int rows = kMaxGroup, size_t bytes = 0);
WorkspaceLayout workspace_layout_slots(int64_t units, int64_t slots, int head_dim, int rows = kMaxGroup,
                                       size_t bytes = 0);

// Clusters of `size` attention CTAs (1..kMaxClusterSplits) the current device holds at
// once (the occupancy query of the head-dim-128 kernel, cached per device); 0 when the
// query fails or there is no device.
int attn_cluster_capacity(int size);

cudaError_t launch_attention(int head_dim, int mode, bool with_scores, const AttnMaps &maps, const AttnParams &p,
                             int batch, cudaStream_t stream);
// Multi-token launch: mode kModeFast (draft over the sparse state) or kModeDense
// (verification; scores written when p.scores is set).
cudaError_t launch_attention_multi(int head_dim, int mode, const AttnMaps &maps, const AttnParams &p, int batch,
                                   cudaStream_t stream);

struct TopkParams {
    const float *scores;
    int64_t score_stride;
    int32_t hkv;
    const int32_t *seq_lens;
    int32_t sink, recent;
    const int32_t *k_per_req;
    int32_t k_cap;
    int32_t *idx_out;
    int32_t *count_out;
    const int32_t *req_ids;
    int32_t *dev_status;
};
cudaError_t launch_select_topk(const TopkParams &p, int batch, cudaStream_t stream);

struct CopyParams {
    const __nv_bfloat16 *k_pool_src;
    const __nv_bfloat16 *v_pool_src;
    __nv_bfloat16 *k_pool_dst;
    __nv_bfloat16 *v_pool_dst;
    int32_t num_pages, max_pages;
    const int32_t *page_table;
    const int32_t *seq_lens;
    int32_t hkv, head_dim;
    const int32_t *req_ids;
    int32_t *dev_status;
    // append of the `tokens` newest tokens
    int32_t tokens;
    const __nv_bfloat16 *k_new;
    const __nv_bfloat16 *v_new;
    // compaction
    const int32_t *idx;
    const int32_t *count;
    int32_t k_cap, sink;
    __nv_bfloat16 *ck;
    __nv_bfloat16 *cv;
    int64_t c_total_rows;
    const int64_t *c_row_offset;
    const int32_t *c_capacity;
};
cudaError_t launch_paged_append(const CopyParams &p, int batch, cudaStream_t stream);
cudaError_t launch_compact_gather(const CopyParams &p, int batch, int max_rows, cudaStream_t stream);

}  // namespace sfi
