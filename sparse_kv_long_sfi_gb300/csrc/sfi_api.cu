// C ABI of libsfi (declared in include/sfi.h): argument validation, TMA descriptor
// encoding, split-KV planning and kernel dispatch. Stateless apart from per-device
// caches of the SM count and of kernel attributes; allocates nothing.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>

#include "sfi_internal.h"

namespace {

using sfi::AttnMaps;
using sfi::AttnParams;

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn tensor_map_encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D view [rows][D] of a bf16 buffer, boxes of [16 rows][64 elements] with the
// 128-byte swizzle (one box row = one 128-byte line).
bool encode_rows(CUtensorMap *map, void *base, int64_t rows, int head_dim) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)head_dim * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)sfi::kSubTokens};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count_current_device() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) {
        int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned8(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

sfi_status check_shape(const sfi_attn_shape *s) {
    if (!s) return SFI_ERR_INVALID_ARG;
    if (s->num_q_heads <= 0 || s->num_kv_heads <= 0 || s->num_q_heads % s->num_kv_heads != 0)
        return SFI_ERR_INVALID_ARG;
    const int g = s->num_q_heads / s->num_kv_heads;
    if (g != 1 && g != 2 && g != 4 && g != 8) return SFI_ERR_UNSUPPORTED;
    if (s->head_dim != 64 && s->head_dim != 128) return SFI_ERR_UNSUPPORTED;
    if (s->page_size != sfi::kSubTokens) return SFI_ERR_UNSUPPORTED;
    return SFI_OK;
}

sfi_status check_paged(const sfi_attn_shape *s, const sfi_paged_kv *kv) {
    if (!kv || !kv->k_pool || !kv->v_pool || !kv->page_table || !kv->seq_lens) return SFI_ERR_INVALID_ARG;
    if (kv->num_pages <= 0 || kv->max_pages_per_req <= 0) return SFI_ERR_INVALID_ARG;
    if (!aligned16(kv->k_pool) || !aligned16(kv->v_pool)) return SFI_ERR_INVALID_ARG;
    // TMA row coordinates are int32
    if ((int64_t)kv->num_pages * s->num_kv_heads * s->page_size >= (int64_t(1) << 31)) return SFI_ERR_UNSUPPORTED;
    if ((int64_t)kv->max_pages_per_req * s->page_size >= (int64_t(1) << 31)) return SFI_ERR_UNSUPPORTED;
    return SFI_OK;
}

// Split-KV plan of one attention launch. Automatic plans fill about 85% of one wave of
// resident CTAs (two per SM); an explicit request is honoured down to two stages per
// split. Leaving a sixth of the slots free lets the next launch's CTAs become resident
// and start streaming while this one drains (batch 1 at 16K, dense: 32 splits, 256 CTAs,
// 15.9 us per layer against 20.6 us for 38 splits, 304 CTAs). Plans of up to
// kMaxClusterSplits merge inside a thread-block cluster (no workspace); between 8 and 16
// splits the plan stays at 8; from 16 on the last CTA of a unit merges the splits from
// the workspace. How short a split may get depends on its merge: inside a cluster three
// stages (12 sub-blocks) per split pay for the CTA's start-up (batch 1, a bound of 1056
// tokens: 6 splits of 11 sub-blocks, 5.05 us per layer against 6.22 us for 4 splits of
// 16); a workspace merge publishes through a global release and wants four stages per
// split.
// The free slots are counted in whole clusters (one cluster of 8 needs 8 free slots of
// one GPC). On a GPU that holds 36 clusters of 8, 38 of 7, 46 of 6 and 58 of 5 (two
// CTAs per SM, 152 SMs): batch 4 at a bound of 2080 tokens, 32 clusters of 8 (32 slots
// free) take 10.3 us per layer against 8.1 us for 32 clusters of 7 (42 free), and at 16K
// dense 53.0 against 47.1 us; batch 5 at 1056 tokens, 40 clusters of 6 (36 free) take
// 5.1 us against 5.5 us for 40 clusters of 5.
int plan_splits(int64_t units, int32_t max_tokens, int32_t requested, int sm_count) {
    constexpr int kMaxSplits = 256;
    if (units <= 0) return 1;
    const int nb = max_tokens > 0 ? (max_tokens + sfi::kSubTokens - 1) / sfi::kSubTokens + 1 : 0;
    int s;
    if (requested > 0) {
        s = requested;
        if (nb > 0) s = std::min(s, std::max(1, nb / (2 * sfi::kConsumerWarps)));
    } else if (nb == 0) {
        s = 1;
    } else {
        s = (int)std::max<int64_t>(1, (int64_t)sm_count * sfi::kAttnCtasPerSm * 17 / 20 / units);
        if (s > sfi::kMaxClusterSplits && s < 2 * sfi::kMaxClusterSplits) s = sfi::kMaxClusterSplits;
        const int in_cluster = std::min(sfi::kMaxClusterSplits, (nb + 3 * sfi::kConsumerWarps - 1) / (3 * sfi::kConsumerWarps));
        s = std::min(s, std::max({1, nb / (4 * sfi::kConsumerWarps), in_cluster}));
        // A cluster is placed whole, so the slots the next launch's early start finds free
        // count in whole clusters: keep a ninth of the SM slots free in those terms.
        const int64_t reserve = (int64_t)sm_count * sfi::kAttnCtasPerSm / 9;
        while (s > 1 && s <= sfi::kMaxClusterSplits) {
            const int cap = sfi::attn_cluster_capacity(s);
            if (cap <= 0 || ((int64_t)cap - units) * s >= reserve) break;
            --s;
        }
    }
    return std::max(1, std::min(s, kMaxSplits));
}

bool needs_workspace(int splits) { return splits > sfi::kMaxClusterSplits; }


// Plan of a mixed launch. The host knows only upper bounds of the units' lengths, so
// each mode is cut into fixed-size chunks of sub-blocks: one wave of two CTAs per SM
// over the upper-bound work, at most 256 sub-blocks (4096 tokens) per chunk. The grid
// covers every unit at its upper bound; each CTA finds its unit's real chunk count on
// the device and exits when it has no chunk (ragged batches stay balanced).
struct MixedPlan {
    int fast_splits, slow_splits;
    int fast_chunk_sb, slow_chunk_sb;
    int64_t units, slots;
};

MixedPlan plan_mixed(int64_t fast_units, int64_t slow_units, int32_t max_fast_tokens, int32_t max_dense_tokens,
                     int sm_count) {
    MixedPlan m{1, 1, 0, 0, fast_units + slow_units, 0};
    const double total = (double)fast_units * std::max(1, max_fast_tokens) +
                         (double)slow_units * std::max(1, max_dense_tokens);
    const double per_cta = std::max(1.0, total / std::max(1, sm_count * sfi::kAttnCtasPerSm));
    const int chunk = (int)std::min(256.0, std::max(4.0 * sfi::kConsumerWarps, std::ceil(per_cta / sfi::kSubTokens)));
    auto splits_for = [&](int32_t tokens) {
        const int nb = (std::max(1, tokens) + sfi::kSubTokens - 1) / sfi::kSubTokens + 1;
        return std::max(1, std::min((nb + chunk - 1) / chunk, 4096));
    };
    if (fast_units > 0) {
        m.fast_splits = splits_for(max_fast_tokens);
        m.fast_chunk_sb = chunk;
    }
    if (slow_units > 0) {
        m.slow_splits = splits_for(max_dense_tokens);
        m.slow_chunk_sb = chunk;
    }
    m.slots = fast_units * m.fast_splits + slow_units * m.slow_splits;
    return m;
}

float resolve_scale(const sfi_attn_shape *s) {
    return s->softmax_scale > 0.f ? s->softmax_scale : 1.0f / std::sqrt((float)s->head_dim);
}

void fill_common(AttnParams &p, const sfi_attn_shape *s, const sfi_paged_kv *kv, const void *q, float *out,
                 float *lse, const int32_t *req_ids, int32_t sink, int32_t recent, int32_t *dev_status) {
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.out = out;
    p.lse = lse;
    p.scores = nullptr;
    p.score_stride = 0;
    p.page_table = kv->page_table;
    p.max_pages = kv->max_pages_per_req;
    p.num_pages = kv->num_pages;
    p.seq_lens = kv->seq_lens;
    p.c_row_offset = nullptr;
    p.c_capacity = nullptr;
    p.c_count = nullptr;
    p.c_total_rows = 0;
    p.req_ids = req_ids;
    p.hq = s->num_q_heads;
    p.hkv = s->num_kv_heads;
    p.group = s->num_q_heads / s->num_kv_heads;
    p.sink = sink;
    p.recent = recent;
    p.scale = resolve_scale(s);
    p.scale_log2 = p.scale * 1.4426950408889634f;
    p.tokens = 1;
    p.rows = p.group;
    p.dev_status = dev_status;
    p.k_new = nullptr;
    p.v_new = nullptr;
    p.k_pool_w = static_cast<__nv_bfloat16 *>(kv->k_pool);
    p.v_pool_w = static_cast<__nv_bfloat16 *>(kv->v_pool);
}

sfi_status bind_workspace(AttnParams &p, int64_t units, int head_dim, void *ws, size_t ws_bytes,
                          int rows = sfi::kMaxGroup) {
    p.ws_count = nullptr;
    p.ws_ml = nullptr;
    p.ws_part = nullptr;
    if (!needs_workspace(p.splits)) return SFI_OK;
    const sfi::WorkspaceLayout l = sfi::workspace_layout(units, p.splits, head_dim, rows, ws_bytes);
    if (!ws || ws_bytes < l.total || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return SFI_ERR_WORKSPACE;
    char *base = static_cast<char *>(ws);
    p.ws_count = reinterpret_cast<int32_t *>(base + l.count_off);
    p.ws_ml = reinterpret_cast<float *>(base + l.ml_off);
    p.ws_part = reinterpret_cast<float *>(base + l.part_off);
    return SFI_OK;
}

// SFI_ATTN_RAGGED: one mode's launch planned in fixed-size chunks through the mixed
// kernel (the requests are all fast or all slow; req_ids may be null).
sfi_status launch_chunked(AttnParams &p, bool fast, const int32_t *req_ids, int32_t batch, int head_dim,
                          int32_t max_tokens, const AttnMaps &maps, void *workspace, size_t workspace_bytes,
                          void *stream) {
    const int64_t units = (int64_t)batch * p.hkv;
    const MixedPlan m = plan_mixed(fast ? units : 0, fast ? 0 : units, fast ? max_tokens : 0, fast ? 0 : max_tokens,
                                   sm_count_current_device());
    p.fast_ids = fast ? req_ids : nullptr;
    p.slow_ids = fast ? nullptr : req_ids;
    p.n_fast = fast ? batch : 0;
    p.n_slow = fast ? 0 : batch;
    p.fast_splits = m.fast_splits;
    p.slow_splits = m.slow_splits;
    p.fast_chunk_sb = m.fast_chunk_sb;
    p.slow_chunk_sb = m.slow_chunk_sb;
    p.splits = std::max(m.fast_splits, m.slow_splits);
    p.ws_count = nullptr;
    p.ws_ml = nullptr;
    p.ws_part = nullptr;
    if (p.splits > 1) {
        const sfi::WorkspaceLayout l = sfi::workspace_layout_slots(m.units, m.slots, head_dim, sfi::kMaxGroup,
                                                                   workspace_bytes);
        if (!workspace || workspace_bytes < l.total || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
            return SFI_ERR_WORKSPACE;
        char *base = static_cast<char *>(workspace);
        p.ws_count = reinterpret_cast<int32_t *>(base + l.count_off);
        p.ws_ml = reinterpret_cast<float *>(base + l.ml_off);
        p.ws_part = reinterpret_cast<float *>(base + l.part_off);
    }
    return sfi::launch_attention(head_dim, sfi::kModeMixed, true, maps, p, 0, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? SFI_OK
               : SFI_ERR_CUDA;
}

sfi_status append_tokens(const sfi_attn_shape *shape, const sfi_paged_kv *kv, const void *k_new, const void *v_new,
                         int32_t tokens, const int32_t *req_ids, int32_t batch, int32_t *dev_status, void *stream) {
    sfi_status st = check_shape(shape);
    if (st != SFI_OK) return st;
    if ((st = check_paged(shape, kv)) != SFI_OK) return st;
    if (batch < 0 || !k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return SFI_ERR_INVALID_ARG;
    if (batch == 0) return SFI_OK;
    sfi::CopyParams p{};
    p.k_pool_dst = static_cast<__nv_bfloat16 *>(kv->k_pool);
    p.v_pool_dst = static_cast<__nv_bfloat16 *>(kv->v_pool);
    p.num_pages = kv->num_pages;
    p.max_pages = kv->max_pages_per_req;
    p.page_table = kv->page_table;
    p.seq_lens = kv->seq_lens;
    p.hkv = shape->num_kv_heads;
    p.head_dim = shape->head_dim;
    p.req_ids = req_ids;
    p.dev_status = dev_status;
    p.tokens = tokens;
    p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    return sfi::launch_paged_append(p, batch, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SFI_OK
                                                                                                : SFI_ERR_CUDA;
}

}  // namespace

extern "C" {

int32_t sfi_version(void) { return SFI_VERSION; }

const char *sfi_status_string(sfi_status status) {
    switch (status) {
        case SFI_OK: return "SFI_OK";
        case SFI_ERR_INVALID_ARG: return "SFI_ERR_INVALID_ARG";
        case SFI_ERR_UNSUPPORTED: return "SFI_ERR_UNSUPPORTED";
        case SFI_ERR_WORKSPACE: return "SFI_ERR_WORKSPACE";
        case SFI_ERR_CUDA: return "SFI_ERR_CUDA";
    }
    return "SFI_ERR_UNKNOWN";
}

int32_t sfi_plan_splits(const sfi_attn_shape *shape, int32_t batch, int32_t max_tokens, int32_t num_splits) {
    if (check_shape(shape) != SFI_OK || batch < 0 || num_splits < 0) return 0;
    return plan_splits((int64_t)batch * shape->num_kv_heads, max_tokens, num_splits, sm_count_current_device());
}

int32_t sfi_attn_cluster_capacity(int32_t cluster_size) { return sfi::attn_cluster_capacity(cluster_size); }

// Bytes for the split plans of every batch size 1..batch sharing one buffer: the counters
// of `batch` requests plus the largest partial-state block of any of those plans (each
// call puts its partial states at the end of the buffer); 0 when no plan needs any.
size_t subset_workspace_size(const sfi_attn_shape *shape, int32_t batch, int32_t max_tokens, int32_t num_splits,
                             int rows) {
    if (check_shape(shape) != SFI_OK || batch < 0 || num_splits < 0) return 0;
    size_t data = 0;
    bool any = false;
    for (int32_t b = 1; b <= batch; ++b) {
        const int32_t s = sfi_plan_splits(shape, b, max_tokens, num_splits);
        if (!needs_workspace(s)) continue;
        any = true;
        data = std::max(data, sfi::workspace_layout((int64_t)b * shape->num_kv_heads, s, shape->head_dim, rows)
                                  .data_bytes);
    }
    if (!any) return 0;
    return sfi::workspace_layout((int64_t)batch * shape->num_kv_heads, 0, shape->head_dim, rows).total + data;
}

size_t sfi_workspace_size(const sfi_attn_shape *shape, int32_t batch, int32_t max_tokens, int32_t num_splits) {
    return subset_workspace_size(shape, batch, max_tokens, num_splits, sfi::kMaxGroup);
}

sfi_status sfi_paged_kv_append(const sfi_attn_shape *shape, const sfi_paged_kv *kv, const void *k_new,
                               const void *v_new, const int32_t *req_ids, int32_t batch, int32_t *dev_status,
                               void *stream) {
    return append_tokens(shape, kv, k_new, v_new, 1, req_ids, batch, dev_status, stream);
}

sfi_status sfi_paged_kv_append_tokens(const sfi_attn_shape *shape, const sfi_paged_kv *kv, const void *k_new,
                                      const void *v_new, int32_t num_tokens, const int32_t *req_ids, int32_t batch,
                                      int32_t *dev_status, void *stream) {
    if (num_tokens < 1 || num_tokens > SFI_MAX_QUERY_TOKENS) return SFI_ERR_INVALID_ARG;
    return append_tokens(shape, kv, k_new, v_new, num_tokens, req_ids, batch, dev_status, stream);
}

sfi_status sfi_fast_decode_attn(const sfi_attn_shape *shape, const sfi_paged_kv *kv, const sfi_compact_kv *compact,
                                int32_t sink, int32_t recent, const void *q, const void *k_new, const void *v_new,
                                float *out, float *lse,
                                const int32_t *req_ids, int32_t batch, int32_t max_tokens, int32_t num_splits, uint32_t flags,
                                void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream) {
    sfi_status st = check_shape(shape);
    if (st != SFI_OK) return st;
    if ((st = check_paged(shape, kv)) != SFI_OK) return st;
    if (batch < 0 || sink < 0 || recent < 0 || num_splits < 0 || !q || !out || !aligned8(out))
        return SFI_ERR_INVALID_ARG;
    if (!compact || !compact->k || !compact->v || !compact->row_offset || !compact->capacity || !compact->count)
        return SFI_ERR_INVALID_ARG;
    if (compact->total_rows <= 0 || !aligned16(compact->k) || !aligned16(compact->v) || !aligned16(q))
        return SFI_ERR_INVALID_ARG;
    if (compact->total_rows >= (int64_t(1) << 31)) return SFI_ERR_UNSUPPORTED;
    if (batch == 0) return SFI_OK;
    if ((k_new == nullptr) != (v_new == nullptr) || (k_new && (!aligned16(k_new) || !aligned16(v_new))))
        return SFI_ERR_INVALID_ARG;
    AttnParams p{};
    fill_common(p, shape, kv, q, out, lse, req_ids, sink, recent, dev_status);
    p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    p.early_prefetch = (flags & SFI_ATTN_EARLY_KV_PREFETCH) ? 1 : 0;
    p.withhold = (flags & SFI_ATTN_TEST_WITHHOLD) ? 2 : 0;  // the second stage
    p.c_row_offset = compact->row_offset;
    p.c_capacity = compact->capacity;
    p.c_count = compact->count;
    p.c_total_rows = compact->total_rows;
    AttnMaps maps;
    const int64_t pool_rows = (int64_t)kv->num_pages * shape->num_kv_heads * shape->page_size;
    if (!encode_rows(&maps.pool_k, kv->k_pool, pool_rows, shape->head_dim) ||
        !encode_rows(&maps.pool_v, kv->v_pool, pool_rows, shape->head_dim) ||
        !encode_rows(&maps.comp_k, compact->k, compact->total_rows, shape->head_dim) ||
        !encode_rows(&maps.comp_v, compact->v, compact->total_rows, shape->head_dim))
        return SFI_ERR_CUDA;
    if (flags & SFI_ATTN_RAGGED)
        return launch_chunked(p, true, req_ids, batch, shape->head_dim, max_tokens, maps, workspace, workspace_bytes,
                              stream);
    const int64_t units = (int64_t)batch * shape->num_kv_heads;
    p.splits = plan_splits(units, max_tokens, num_splits, sm_count_current_device());
    if ((st = bind_workspace(p, units, shape->head_dim, workspace, workspace_bytes)) != SFI_OK) return st;
    return sfi::launch_attention(shape->head_dim, sfi::kModeFast, false, maps, p, batch,
                                 static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SFI_OK
               : SFI_ERR_CUDA;
}

sfi_status sfi_slow_dense_attn_with_scores(const sfi_attn_shape *shape, const sfi_paged_kv *kv, int32_t sink,
                                           int32_t recent, const void *q, const void *k_new, const void *v_new,
                                           float *out, float *lse, float *scores,
                                           int64_t score_stride, const int32_t *req_ids, int32_t batch,
                                           int32_t max_tokens, int32_t num_splits, uint32_t flags, void *workspace,
                                           size_t workspace_bytes, int32_t *dev_status, void *stream) {
    sfi_status st = check_shape(shape);
    if (st != SFI_OK) return st;
    if ((st = check_paged(shape, kv)) != SFI_OK) return st;
    if (batch < 0 || sink < 0 || recent < 0 || num_splits < 0 || !q || !out || !aligned16(q) || !aligned8(out))
        return SFI_ERR_INVALID_ARG;
    if (scores && score_stride <= 0) return SFI_ERR_INVALID_ARG;
    if (batch == 0) return SFI_OK;
    if ((k_new == nullptr) != (v_new == nullptr) || (k_new && (!aligned16(k_new) || !aligned16(v_new))))
        return SFI_ERR_INVALID_ARG;
    AttnParams p{};
    fill_common(p, shape, kv, q, out, lse, req_ids, sink, recent, dev_status);
    p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    p.early_prefetch = (flags & SFI_ATTN_EARLY_KV_PREFETCH) ? 1 : 0;
    p.withhold = (flags & SFI_ATTN_TEST_WITHHOLD) ? 2 : 0;  // the second stage
    p.scores = scores;
    p.score_stride = score_stride;
    AttnMaps maps;
    const int64_t pool_rows = (int64_t)kv->num_pages * shape->num_kv_heads * shape->page_size;
    if (!encode_rows(&maps.pool_k, kv->k_pool, pool_rows, shape->head_dim) ||
        !encode_rows(&maps.pool_v, kv->v_pool, pool_rows, shape->head_dim))
        return SFI_ERR_CUDA;
    maps.comp_k = maps.pool_k;  // unused in dense mode
    maps.comp_v = maps.pool_v;
    if (flags & SFI_ATTN_RAGGED)
        return launch_chunked(p, false, req_ids, batch, shape->head_dim, max_tokens, maps, workspace,
                              workspace_bytes, stream);
    const int64_t units = (int64_t)batch * shape->num_kv_heads;
    p.splits = plan_splits(units, max_tokens, num_splits, sm_count_current_device());
    if ((st = bind_workspace(p, units, shape->head_dim, workspace, workspace_bytes)) != SFI_OK) return st;
    return sfi::launch_attention(shape->head_dim, sfi::kModeDense, scores != nullptr, maps, p, batch,
                                 static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SFI_OK
               : SFI_ERR_CUDA;
}

size_t sfi_mixed_workspace_size(const sfi_attn_shape *shape, int32_t n_fast, int32_t n_slow, int32_t max_fast_tokens,
                                int32_t max_dense_tokens) {
    if (check_shape(shape) != SFI_OK || n_fast < 0 || n_slow < 0) return 0;
    const int hkv = shape->num_kv_heads;
    const int sms = sm_count_current_device();
    // One mode only (the chunked plans of SFI_ATTN_RAGGED): valid for every batch size up
    // to n, like sfi_workspace_size. Both modes: this split of the requests.
    const int32_t n = n_fast + n_slow;
    const int32_t b_lo = (n_fast == 0 || n_slow == 0) ? 1 : n;
    size_t data = 0;
    bool any = false;
    for (int32_t b = std::max(1, b_lo); b <= n; ++b) {
        const int64_t f = n_slow == 0 ? b : n_fast, sl = n_fast == 0 ? b : n_slow;
        const MixedPlan m = plan_mixed(f * hkv, sl * hkv, max_fast_tokens, max_dense_tokens, sms);
        if (m.fast_splits == 1 && m.slow_splits == 1) continue;
        any = true;
        data = std::max(data, sfi::workspace_layout_slots(m.units, m.slots, shape->head_dim).data_bytes);
    }
    if (!any) return 0;
    return sfi::workspace_layout_slots((int64_t)n * hkv, 0, shape->head_dim).total + data;
}

sfi_status sfi_mixed_decode_attn(const sfi_attn_shape *shape, const sfi_paged_kv *kv, const sfi_compact_kv *compact,
                                 int32_t sink, int32_t recent, const void *q, const void *k_new, const void *v_new,
                                 float *out, float *lse, float *scores, int64_t score_stride, const int32_t *fast_ids,
                                 int32_t n_fast, const int32_t *slow_ids, int32_t n_slow, int32_t max_fast_tokens,
                                 int32_t max_dense_tokens, uint32_t flags, void *workspace, size_t workspace_bytes,
                                 int32_t *dev_status, void *stream) {
    sfi_status st = check_shape(shape);
    if (st != SFI_OK) return st;
    if ((st = check_paged(shape, kv)) != SFI_OK) return st;
    if (n_fast < 0 || n_slow < 0 || sink < 0 || recent < 0 || !q || !out || !aligned16(q) || !aligned8(out))
        return SFI_ERR_INVALID_ARG;
    if ((n_fast > 0 && !fast_ids) || (n_slow > 0 && !slow_ids)) return SFI_ERR_INVALID_ARG;
    if ((k_new == nullptr) != (v_new == nullptr) || (k_new && (!aligned16(k_new) || !aligned16(v_new))))
        return SFI_ERR_INVALID_ARG;
    if (scores && score_stride <= 0) return SFI_ERR_INVALID_ARG;
    if (n_fast > 0) {
        if (!compact || !compact->k || !compact->v || !compact->row_offset || !compact->capacity || !compact->count)
            return SFI_ERR_INVALID_ARG;
        if (compact->total_rows <= 0 || !aligned16(compact->k) || !aligned16(compact->v)) return SFI_ERR_INVALID_ARG;
        if (compact->total_rows >= (int64_t(1) << 31)) return SFI_ERR_UNSUPPORTED;
    }
    if (n_fast + n_slow == 0) return SFI_OK;
    AttnParams p{};
    fill_common(p, shape, kv, q, out, lse, nullptr, sink, recent, dev_status);
    p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    p.early_prefetch = (flags & SFI_ATTN_EARLY_KV_PREFETCH) ? 1 : 0;
    p.scores = scores;
    p.score_stride = score_stride;
    if (n_fast > 0) {
        p.c_row_offset = compact->row_offset;
        p.c_capacity = compact->capacity;
        p.c_count = compact->count;
        p.c_total_rows = compact->total_rows;
    }
    const MixedPlan m = plan_mixed((int64_t)n_fast * shape->num_kv_heads, (int64_t)n_slow * shape->num_kv_heads,
                                   max_fast_tokens, max_dense_tokens, sm_count_current_device());
    p.fast_ids = fast_ids;
    p.slow_ids = slow_ids;
    p.n_fast = n_fast;
    p.n_slow = n_slow;
    p.fast_splits = m.fast_splits;
    p.slow_splits = m.slow_splits;
    p.fast_chunk_sb = m.fast_chunk_sb;
    p.slow_chunk_sb = m.slow_chunk_sb;
    p.splits = std::max(m.fast_splits, m.slow_splits);  // > 1: partial states go through the workspace
    if (p.splits > 1) {
        const sfi::WorkspaceLayout l = sfi::workspace_layout_slots(m.units, m.slots, shape->head_dim,
                                                                   sfi::kMaxGroup, workspace_bytes);
        if (!workspace || workspace_bytes < l.total || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
            return SFI_ERR_WORKSPACE;
        char *base = static_cast<char *>(workspace);
        p.ws_count = reinterpret_cast<int32_t *>(base + l.count_off);
        p.ws_ml = reinterpret_cast<float *>(base + l.ml_off);
        p.ws_part = reinterpret_cast<float *>(base + l.part_off);
    }
    AttnMaps maps;
    const int64_t pool_rows = (int64_t)kv->num_pages * shape->num_kv_heads * shape->page_size;
    if (!encode_rows(&maps.pool_k, kv->k_pool, pool_rows, shape->head_dim) ||
        !encode_rows(&maps.pool_v, kv->v_pool, pool_rows, shape->head_dim))
        return SFI_ERR_CUDA;
    if (n_fast > 0) {
        if (!encode_rows(&maps.comp_k, compact->k, compact->total_rows, shape->head_dim) ||
            !encode_rows(&maps.comp_v, compact->v, compact->total_rows, shape->head_dim))
            return SFI_ERR_CUDA;
    } else {
        maps.comp_k = maps.pool_k;
        maps.comp_v = maps.pool_v;
    }
    return sfi::launch_attention(shape->head_dim, sfi::kModeMixed, true, maps, p, 0,
                                 static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SFI_OK
               : SFI_ERR_CUDA;
}

size_t sfi_multi_workspace_size(const sfi_attn_shape *shape, int32_t batch, int32_t num_tokens, int32_t max_tokens,
                                int32_t num_splits) {
    if (num_tokens < 1 || num_tokens > SFI_MAX_QUERY_TOKENS) return 0;
    return subset_workspace_size(shape, batch, max_tokens, num_splits, sfi::kMaxRows);
}

sfi_status sfi_dense_verify_attn(const sfi_attn_shape *shape, const sfi_paged_kv *kv, int32_t sink, int32_t recent,
                                 const void *q, int32_t num_tokens, const void *k_new, const void *v_new, float *out,
                                 float *lse, float *scores,
                                 int64_t score_stride, const int32_t *req_ids, int32_t batch, int32_t max_tokens,
                                 int32_t num_splits, uint32_t flags, void *workspace, size_t workspace_bytes,
                                 int32_t *dev_status, void *stream) {
    sfi_status st = check_shape(shape);
    if (st != SFI_OK) return st;
    if ((st = check_paged(shape, kv)) != SFI_OK) return st;
    if (batch < 0 || sink < 0 || recent < 0 || num_splits < 0 || !q || !out || !aligned16(q) || !aligned8(out))
        return SFI_ERR_INVALID_ARG;
    if (num_tokens < 1 || num_tokens > SFI_MAX_QUERY_TOKENS) return SFI_ERR_INVALID_ARG;
    if (num_tokens * (shape->num_q_heads / shape->num_kv_heads) > sfi::kMaxRows) return SFI_ERR_UNSUPPORTED;
    if ((k_new == nullptr) != (v_new == nullptr) || (k_new && (!aligned16(k_new) || !aligned16(v_new))))
        return SFI_ERR_INVALID_ARG;
    if (scores && score_stride <= 0) return SFI_ERR_INVALID_ARG;
    if (batch == 0) return SFI_OK;
    AttnParams p{};
    fill_common(p, shape, kv, q, out, lse, req_ids, sink, recent, dev_status);
    p.tokens = num_tokens;
    p.rows = num_tokens * p.group;
    p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    p.early_prefetch = (flags & SFI_ATTN_EARLY_KV_PREFETCH) ? 1 : 0;
    p.scores = scores;
    p.score_stride = score_stride;
    const int64_t units = (int64_t)batch * shape->num_kv_heads;
    p.splits = plan_splits(units, max_tokens, num_splits, sm_count_current_device());
    if ((st = bind_workspace(p, units, shape->head_dim, workspace, workspace_bytes, sfi::kMaxRows)) != SFI_OK)
        return st;
    AttnMaps maps;
    const int64_t pool_rows = (int64_t)kv->num_pages * shape->num_kv_heads * shape->page_size;
    if (!encode_rows(&maps.pool_k, kv->k_pool, pool_rows, shape->head_dim) ||
        !encode_rows(&maps.pool_v, kv->v_pool, pool_rows, shape->head_dim))
        return SFI_ERR_CUDA;
    maps.comp_k = maps.pool_k;  // unused in dense mode
    maps.comp_v = maps.pool_v;
    return sfi::launch_attention_multi(shape->head_dim, sfi::kModeDense, maps, p, batch,
                                       static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SFI_OK
               : SFI_ERR_CUDA;
}

sfi_status sfi_sparse_draft_attn(const sfi_attn_shape *shape, const sfi_paged_kv *kv, const sfi_compact_kv *compact,
                                 int32_t sink, int32_t recent, const void *q, int32_t num_tokens, const void *k_new,
                                 const void *v_new, float *out, float *lse, const int32_t *req_ids, int32_t batch, int32_t max_tokens,
                                 int32_t num_splits, uint32_t flags, void *workspace, size_t workspace_bytes,
                                 int32_t *dev_status, void *stream) {
    sfi_status st = check_shape(shape);
    if (st != SFI_OK) return st;
    if ((st = check_paged(shape, kv)) != SFI_OK) return st;
    if (batch < 0 || sink < 0 || recent < 0 || num_splits < 0 || !q || !out || !aligned16(q) || !aligned8(out))
        return SFI_ERR_INVALID_ARG;
    if (num_tokens < 1 || num_tokens > SFI_MAX_QUERY_TOKENS) return SFI_ERR_INVALID_ARG;
    if (num_tokens * (shape->num_q_heads / shape->num_kv_heads) > sfi::kMaxRows) return SFI_ERR_UNSUPPORTED;
    if ((k_new == nullptr) != (v_new == nullptr) || (k_new && (!aligned16(k_new) || !aligned16(v_new))))
        return SFI_ERR_INVALID_ARG;
    if (!compact || !compact->k || !compact->v || !compact->row_offset || !compact->capacity || !compact->count)
        return SFI_ERR_INVALID_ARG;
    if (compact->total_rows <= 0 || !aligned16(compact->k) || !aligned16(compact->v)) return SFI_ERR_INVALID_ARG;
    if (compact->total_rows >= (int64_t(1) << 31)) return SFI_ERR_UNSUPPORTED;
    if (batch == 0) return SFI_OK;
    // One draft token is one fast step (same streams, same fused append, same output
    // layout): the single-token kernel keeps the query in registers and skips the per-row
    // bookkeeping, 14.2 -> 13.1 us per launch at batch 16. Its workspace need (the same
    // split plan, fewer rows per slot) is within the multi-token size.
    if (num_tokens == 1)
        return sfi_fast_decode_attn(shape, kv, compact, sink, recent, q, k_new, v_new, out, lse, req_ids, batch,
                                    max_tokens, num_splits, flags & SFI_ATTN_EARLY_KV_PREFETCH, workspace,
                                    workspace_bytes, dev_status, stream);
    AttnParams p{};
    fill_common(p, shape, kv, q, out, lse, req_ids, sink, recent, dev_status);
    p.tokens = num_tokens;
    p.rows = num_tokens * p.group;
    p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    p.early_prefetch = (flags & SFI_ATTN_EARLY_KV_PREFETCH) ? 1 : 0;
    p.c_row_offset = compact->row_offset;
    p.c_capacity = compact->capacity;
    p.c_count = compact->count;
    p.c_total_rows = compact->total_rows;
    const int64_t units = (int64_t)batch * shape->num_kv_heads;
    p.splits = plan_splits(units, max_tokens, num_splits, sm_count_current_device());
    if ((st = bind_workspace(p, units, shape->head_dim, workspace, workspace_bytes, sfi::kMaxRows)) != SFI_OK)
        return st;
    AttnMaps maps;
    const int64_t pool_rows = (int64_t)kv->num_pages * shape->num_kv_heads * shape->page_size;
    if (!encode_rows(&maps.pool_k, kv->k_pool, pool_rows, shape->head_dim) ||
        !encode_rows(&maps.pool_v, kv->v_pool, pool_rows, shape->head_dim) ||
        !encode_rows(&maps.comp_k, compact->k, compact->total_rows, shape->head_dim) ||
        !encode_rows(&maps.comp_v, compact->v, compact->total_rows, shape->head_dim))
        return SFI_ERR_CUDA;
    return sfi::launch_attention_multi(shape->head_dim, sfi::kModeFast, maps, p, batch,
                                       static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SFI_OK
               : SFI_ERR_CUDA;
}

sfi_status sfi_select_topk(const float *scores, int64_t score_stride, int32_t num_kv_heads, const int32_t *seq_lens,
                           int32_t sink, int32_t recent, const int32_t *k_per_req, int32_t k_cap, int32_t *idx_out,
                           int32_t *count_out, const int32_t *req_ids, int32_t batch, int32_t *dev_status,
                           void *stream) {
    if (!scores || !seq_lens || !k_per_req || !idx_out || !count_out) return SFI_ERR_INVALID_ARG;
    if (score_stride <= 0 || num_kv_heads <= 0 || sink < 0 || recent < 0 || k_cap < 0 || batch < 0)
        return SFI_ERR_INVALID_ARG;
    if (batch == 0) return SFI_OK;
    sfi::TopkParams p{};
    p.scores = scores;
    p.score_stride = score_stride;
    p.hkv = num_kv_heads;
    p.seq_lens = seq_lens;
    p.sink = sink;
    p.recent = recent;
    p.k_per_req = k_per_req;
    p.k_cap = k_cap;
    p.idx_out = idx_out;
    p.count_out = count_out;
    p.req_ids = req_ids;
    p.dev_status = dev_status;
    return sfi::launch_select_topk(p, batch, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SFI_OK
                                                                                               : SFI_ERR_CUDA;
}

sfi_status sfi_compact_gather(const sfi_attn_shape *shape, const sfi_paged_kv *kv, const int32_t *idx,
                              const int32_t *count, int32_t k_cap, int32_t sink, const sfi_compact_kv *compact,
                              const int32_t *req_ids, int32_t batch, int32_t *dev_status, void *stream) {
    sfi_status st = check_shape(shape);
    if (st != SFI_OK) return st;
    if ((st = check_paged(shape, kv)) != SFI_OK) return st;
    if (!idx || !count || k_cap < 0 || sink < 0 || batch < 0) return SFI_ERR_INVALID_ARG;
    if (!compact || !compact->k || !compact->v || !compact->row_offset || !compact->capacity)
        return SFI_ERR_INVALID_ARG;
    if (compact->total_rows <= 0 || !aligned16(compact->k) || !aligned16(compact->v)) return SFI_ERR_INVALID_ARG;
    if (batch == 0 || (int64_t)sink + k_cap == 0) return SFI_OK;
    if ((int64_t)sink + k_cap >= (int64_t(1) << 31)) return SFI_ERR_INVALID_ARG;
    sfi::CopyParams p{};
    p.k_pool_src = static_cast<const __nv_bfloat16 *>(kv->k_pool);
    p.v_pool_src = static_cast<const __nv_bfloat16 *>(kv->v_pool);
    p.num_pages = kv->num_pages;
    p.max_pages = kv->max_pages_per_req;
    p.page_table = kv->page_table;
    p.seq_lens = kv->seq_lens;
    p.hkv = shape->num_kv_heads;
    p.head_dim = shape->head_dim;
    p.req_ids = req_ids;
    p.dev_status = dev_status;
    p.idx = idx;
    p.count = count;
    p.k_cap = k_cap;
    p.sink = sink;
    p.ck = static_cast<__nv_bfloat16 *>(compact->k);
    p.cv = static_cast<__nv_bfloat16 *>(compact->v);
    p.c_total_rows = compact->total_rows;
    p.c_row_offset = compact->row_offset;
    p.c_capacity = compact->capacity;
    return sfi::launch_compact_gather(p, batch, sink + k_cap, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SFI_OK
               : SFI_ERR_CUDA;
}

sfi_status sfi_select_compact(const sfi_attn_shape *shape, const sfi_paged_kv *kv, const float *scores,
                              int64_t score_stride, int32_t sink, int32_t recent, const int32_t *k_per_req,
                              int32_t k_cap, int32_t *idx_out, int32_t *count_out, const sfi_compact_kv *compact,
                              const int32_t *req_ids, int32_t batch, int32_t *dev_status, void *stream) {
    sfi_status st = check_shape(shape);
    if (st != SFI_OK) return st;
    if ((st = check_paged(shape, kv)) != SFI_OK) return st;
    if (!scores || !k_per_req || !idx_out || !count_out) return SFI_ERR_INVALID_ARG;
    if (score_stride <= 0 || sink < 0 || recent < 0 || k_cap < 0 || batch < 0) return SFI_ERR_INVALID_ARG;
    if (!compact || !compact->k || !compact->v || !compact->row_offset || !compact->capacity)
        return SFI_ERR_INVALID_ARG;
    if (compact->total_rows <= 0 || !aligned16(compact->k) || !aligned16(compact->v)) return SFI_ERR_INVALID_ARG;
    if ((int64_t)sink + k_cap >= (int64_t(1) << 31)) return SFI_ERR_INVALID_ARG;
    if (batch == 0) return SFI_OK;
    sfi::TopkParams p{};
    p.scores = scores;
    p.score_stride = score_stride;
    p.hkv = shape->num_kv_heads;
    p.seq_lens = kv->seq_lens;
    p.sink = sink;
    p.recent = recent;
    p.k_per_req = k_per_req;
    p.k_cap = k_cap;
    p.idx_out = idx_out;
    p.count_out = count_out;
    p.req_ids = req_ids;
    p.dev_status = dev_status;
    sfi::CopyParams c{};
    c.k_pool_src = static_cast<const __nv_bfloat16 *>(kv->k_pool);
    c.v_pool_src = static_cast<const __nv_bfloat16 *>(kv->v_pool);
    c.num_pages = kv->num_pages;
    c.max_pages = kv->max_pages_per_req;
    c.page_table = kv->page_table;
    c.seq_lens = kv->seq_lens;
    c.hkv = shape->num_kv_heads;
    c.head_dim = shape->head_dim;
    c.req_ids = req_ids;
    c.dev_status = dev_status;
    c.k_cap = k_cap;
    c.sink = sink;
    c.ck = static_cast<__nv_bfloat16 *>(compact->k);
    c.cv = static_cast<__nv_bfloat16 *>(compact->v);
    c.c_total_rows = compact->total_rows;
    c.c_row_offset = compact->row_offset;
    c.c_capacity = compact->capacity;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (sfi::launch_select_topk(p, batch, s) != cudaSuccess) return SFI_ERR_CUDA;
    if ((int64_t)sink + k_cap == 0) return SFI_OK;
    c.idx = idx_out;
    c.count = count_out;
    return sfi::launch_compact_gather(c, batch, sink + k_cap, s) == cudaSuccess ? SFI_OK : SFI_ERR_CUDA;
}

}  // extern "C"
