/*
 * sfi.h - C ABI of libsfi: Slow-Fast Inference (SFI) decode attention over a
 * sparse, recallable KV memory, for NVIDIA GB300 (sm_103a).
 *
 * Method: "Slow-Fast Inference: Training-Free Inference Acceleration via
 * Within-Sentence Support Stability" (Xie et al., 2026).
 *   Figure 2 caption: fast steps attend to a managed sparse state
 *     (sink + selected + recent); a slow step performs dense attention, collects
 *     masked attention logits over the allowed candidate set and invokes the
 *     Selector to refresh the selected memory for the next segment.
 *   Figure 3 caption: (A) the Selector and cache reorganisation of layer i run on
 *     an aux stream while the main stream computes layer i+1's attention;
 *     (B) sink and selected tokens are packed into a contiguous compact buffer and
 *     recent tokens are read in place from paged KV.
 *   Table 1: kernel-level sparse/dense speedup at KV length 16K, batch 16, bf16.
 * The same per-KV-head logit statistics are what "A Sparse Glimpse of the Whole:
 * Train-Free Self-Speculative Decoding" (SparseSpec-L, abstract) recycles as its
 * importance signal.
 *
 * Notation: B requests, Hq query heads, Hkv KV heads, G = Hq / Hkv, D head_dim,
 * P page size, L the current length of a request (the current token included),
 * S sink size, W recent-window size, k selected tokens per KV head.
 * Query head h reads KV head h / G. Softmax scale defaults to 1/sqrt(D).
 *
 * Sparse state of a request at length L (the fast step attends to exactly this):
 *   sink     positions [0, min(S, L))              compact rows [0, min(S, L))
 *   selected positions idx[0 .. count)             compact rows [S, S + count)
 *   recent   positions [max(S, L - W), L)          read in place from the pages
 * Candidates of a slow step at length L: C = [S, L - W) (empty when L <= S + W).
 *
 * Conventions for every entry point:
 *   - The caller owns every buffer. The library allocates nothing, frees nothing,
 *     never synchronises and never changes the current device. Device pointers
 *     must belong to the current device.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream)
 *     and runs asynchronously.
 *   - Host-side errors (a NULL pointer, an unsupported shape, a short workspace)
 *     are returned before anything is launched. A failed launch returns
 *     SFI_ERR_CUDA.
 *   - Device-side errors never trap: the kernel ORs an SFI_DEV_* bit into
 *     *dev_status (optional; may be NULL) and skips the offending unit's writes.
 *     In the attention calls the unit is a (request, KV head): when any of its
 *     page ids is out of range, or one of its waits runs out, none of its outputs,
 *     log-sum-exps or score entries is written (the caller's values stay), in every
 *     split plan; other units are unaffected.
 *   - Per-request arrays (q, out, lse, scores, seq_lens, page_table rows,
 *     k_per_req, counts, compact rows) are indexed by the request id r. An entry
 *     point processes `batch` requests: r = req_ids[b] when req_ids is non-NULL
 *     (a subset of a larger batch, e.g. the slow subset of a mixed step), else
 *     r = b. req_ids must not repeat an id within one call.
 *   - Supported: head_dim 64 or 128, page_size 16, G in {1, 2, 4, 8}. Q/K/V are
 *     bf16; outputs, LSE and scores are fp32; positions are int32.
 *   - LSE is the natural log of sum_j exp(scale * q . k_j) over the attended
 *     positions.
 */
#ifndef SFI_H
#define SFI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SFI_VERSION 1

#if defined(__GNUC__)
#define SFI_API __attribute__((visibility("default")))
#else
#define SFI_API
#endif

typedef enum {
    SFI_OK = 0,
    SFI_ERR_INVALID_ARG = 1, /* NULL pointer, negative size, inconsistent shape */
    SFI_ERR_UNSUPPORTED = 2, /* head_dim, page_size or group size not supported */
    SFI_ERR_WORKSPACE = 3,   /* workspace missing or smaller than sfi_workspace_size() */
    SFI_ERR_CUDA = 4         /* a CUDA call or launch failed */
} sfi_status;

/* Bits ORed into *dev_status by the kernels (0 = no error). */
#define SFI_DEV_BAD_PAGE 1u     /* a page-table entry outside [0, num_pages) */
#define SFI_DEV_BAD_LEN 2u      /* seq_len < 1 or beyond the page table */
#define SFI_DEV_K_OVERFLOW 4u   /* k_r < 0, k_r > k_cap, or sink + count > capacity */
#define SFI_DEV_BAD_INDEX 8u    /* a selected position outside [0, L) */
#define SFI_DEV_TIMEOUT 16u     /* an in-kernel pipeline wait ran past its bound */
#define SFI_DEV_BAD_COMPACT 32u /* compact rows of a request fall outside the buffer */

/* Launch flags of the attention entry points (bitwise OR). */
/* SFI_ATTN_EARLY_KV_PREFETCH: the kernel that precedes this call on the stream does
 * not write this call's paged KV pools, compact buffer, page table, lengths or
 * request ids, nor the compact counts and capacities. The
 * kernel may then start streaming them (programmatic dependent launch) before that
 * preceding kernel has finished; q, k_new and v_new are still read, and every output
 * written, only after it has finished. Without the flag nothing is read before then. */
#define SFI_ATTN_EARLY_KV_PREFETCH 1u
/* SFI_ATTN_RAGGED (sfi_fast_decode_attn and sfi_slow_dense_attn_with_scores): the
 * requests' lengths differ widely (a ragged batch). The launch is then planned in
 * fixed-size chunks, as sfi_mixed_decode_attn does (each (request, KV head) gets
 * splits in proportion to its real length, found on the device), instead of the same
 * number of splits for every request; num_splits is ignored and the workspace must
 * hold sfi_mixed_workspace_size(shape, batch, 0, max_tokens, 0) bytes for the fast
 * call and sfi_mixed_workspace_size(shape, 0, batch, 0, max_tokens) for the dense one. */
#define SFI_ATTN_RAGGED 2u
/* SFI_ATTN_TEST_WITHHOLD (the same two calls; diagnostic, for testing the bounded
 * in-kernel waits): the TMA producer of every CTA withholds the copies of its second
 * stage, so the consumers' wait for it runs out (after about 2 s) and the launch
 * reports SFI_DEV_TIMEOUT; the affected units write no output, the workspace is
 * left zeroed as after any launch, and the context stays usable. Units shorter than
 * two stages are unaffected. Not for production use. */
#define SFI_ATTN_TEST_WITHHOLD 4u

/* Most query tokens per request in the multi-token calls (tokens x G must also be
 * <= 16: G = 2 allows 8 tokens, G = 4 four, G = 8 two). */
#define SFI_MAX_QUERY_TOKENS 16

/* Attention geometry shared by all calls. */
typedef struct {
    int32_t num_q_heads;  /* Hq */
    int32_t num_kv_heads; /* Hkv */
    int32_t head_dim;     /* D: 64 or 128 */
    int32_t page_size;    /* P: 16 */
    float softmax_scale;  /* <= 0 selects 1/sqrt(D) */
} sfi_attn_shape;

/* Paged bf16 KV cache (Figure 3: the dense KV is kept in pages and never discarded). */
typedef struct {
    void *k_pool;               /* bf16 [num_pages][Hkv][P][D], 16-byte aligned */
    void *v_pool;               /* bf16 [num_pages][Hkv][P][D], 16-byte aligned */
    int32_t num_pages;          /* pages in each pool */
    int32_t max_pages_per_req;  /* row stride of page_table */
    const int32_t *page_table;  /* int32 [B][max_pages_per_req]: page of positions [16p, 16p+16) */
    const int32_t *seq_lens;    /* int32 [B]: L of each request, current token included */
} sfi_paged_kv;

/* Compact buffer (Figure 3B: sink + selected packed contiguously), one per layer.
 * Row i of KV head h of request r is buffer row  row_offset[r] + h * capacity[r] + i,
 * each row D bf16 values. Rows [0, min(S, L)) hold the sink, rows [S, S + count[r])
 * the selection in ascending position order. */
typedef struct {
    void *k;                   /* bf16 [total_rows][D], 16-byte aligned */
    void *v;                   /* bf16 [total_rows][D], 16-byte aligned */
    int64_t total_rows;        /* rows in each of k and v */
    const int64_t *row_offset; /* int64 [B] */
    const int32_t *capacity;   /* int32 [B] rows per KV head, >= S + k_r */
    const int32_t *count;      /* int32 [B] selected rows per KV head (written by sfi_select_topk) */
} sfi_compact_kv;

/*
 * sfi_paged_kv_append - write the current token's K and V into the paged cache.
 * Figure 3 caption (paged KV). For each request r, position L_r - 1 (L_r =
 * seq_lens[r], which already counts the new token) receives k_new[r] and v_new[r]:
 * slot (L_r - 1) % P of page page_table[r][(L_r - 1) / P].
 *   k_new, v_new : bf16 [B][Hkv][D], indexed by request id like q
 * Device errors: SFI_DEV_BAD_LEN, SFI_DEV_BAD_PAGE (that request is skipped).
 */
SFI_API sfi_status sfi_paged_kv_append(const sfi_attn_shape *shape, const sfi_paged_kv *kv, const void *k_new,
                               const void *v_new, const int32_t *req_ids, int32_t batch, int32_t *dev_status,
                               void *stream);

/*
 * sfi_fast_decode_attn - the fast step (Figure 2: attention over sink + selected +
 * recent; Figure 3B: the compact segment is streamed contiguously, the recent
 * segment is gathered page by page in place).
 * Each query head h of request r attends, with one softmax, to compact rows
 * [0, min(S, L) + count[r]) of KV head h / G followed by paged positions
 * [max(S, L - W), L). The compact buffer must have been filled by
 * sfi_compact_gather at a length >= min(S, L) (the sink is complete).
 *   q       : bf16 [B][Hq][D]
 *   k_new, v_new : bf16 [B][Hkv][D] or both NULL. When given, the call first does
 *                what sfi_paged_kv_append does (the current token goes to position
 *                L - 1 of the pages) and attends to the cache after that append;
 *                when L <= S the token is a sink row and is used in place of compact
 *                row L - 1 (the compact buffer itself is not written).
 *   out     : fp32 [B][Hq][D], 8-byte aligned
 *   lse     : fp32 [B][Hq] or NULL
 *   max_tokens : an upper bound on S + max count + W + P over the batch, used to
 *                plan split-KV; 0 lets the library assume the compact capacity
 *                is small. It affects speed only, never results.
 *   num_splits : 0 = automatic; otherwise the number of KV splits per
 *                (request, KV head) (clamped to the plan's maximum).
 *   flags      : 0, SFI_ATTN_EARLY_KV_PREFETCH and/or SFI_ATTN_RAGGED (and the diagnostic
 *                SFI_ATTN_TEST_WITHHOLD).
 *   workspace  : at least sfi_workspace_size(shape, batch, max_tokens, num_splits)
 *                bytes of device memory, zero-filled before its first use. The
 *                kernels leave its split counters zero-filled again when they
 *                finish, device errors and timed-out waits included (every split
 *                of a unit reaches the counter). Launches that share one
 *                workspace must not overlap in time.
 * Device errors: SFI_DEV_BAD_LEN, SFI_DEV_BAD_PAGE, SFI_DEV_K_OVERFLOW,
 * SFI_DEV_BAD_COMPACT, SFI_DEV_TIMEOUT.
 */
SFI_API sfi_status sfi_fast_decode_attn(const sfi_attn_shape *shape, const sfi_paged_kv *kv, const sfi_compact_kv *compact,
                                int32_t sink, int32_t recent, const void *q, const void *k_new, const void *v_new,
                                float *out, float *lse,
                                const int32_t *req_ids, int32_t batch, int32_t max_tokens, int32_t num_splits, uint32_t flags,
                                void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * sfi_slow_dense_attn_with_scores - the slow step (Figure 2 caption: dense
 * attention plus the masked attention logits over the candidate set).
 * Each query head attends to all positions [0, L) of its KV head through the page
 * table. When scores is non-NULL it also writes, for every KV head kv,
 *   scores[r][kv][j] = sum_{g < G} scale * q_{kv*G+g} . k_{kv,j}   for j in [S, L - W)
 *   scores[r][kv][j] = -inf                                        for other j < L
 * in fp32; entries j >= L are not written. With scores == NULL this is the dense
 * full-KV decode attention (the denominator of Table 1).
 *   k_new, v_new : bf16 [B][Hkv][D] or both NULL: the current token, appended at
 *                  position L - 1 before the attention (as sfi_paged_kv_append)
 *   scores       : fp32 [B][Hkv][score_stride], score_stride >= max L, or NULL
 *   max_tokens   : an upper bound on L + P over the batch (split planning only)
 *   num_splits, flags, workspace, workspace_bytes : as for sfi_fast_decode_attn
 * Device errors: SFI_DEV_BAD_LEN (also when L > score_stride: the scores of that
 * request are then not written), SFI_DEV_BAD_PAGE, SFI_DEV_TIMEOUT.
 */
SFI_API sfi_status sfi_slow_dense_attn_with_scores(const sfi_attn_shape *shape, const sfi_paged_kv *kv, int32_t sink,
                                           int32_t recent, const void *q, const void *k_new, const void *v_new,
                                           float *out, float *lse, float *scores,
                                           int64_t score_stride, const int32_t *req_ids, int32_t batch,
                                           int32_t max_tokens, int32_t num_splits, uint32_t flags, void *workspace,
                                           size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * sfi_mixed_decode_attn - one launch for a batch whose requests are at different
 * steps: the requests fast_ids[0 .. n_fast) do the fast step of
 * sfi_fast_decode_attn, the requests slow_ids[0 .. n_slow) the slow step of
 * sfi_slow_dense_attn_with_scores (dense attention, plus the masked scores when
 * scores is non-NULL). "ASPIRE: Asynchronous Batched Self-Speculative Decoding for
 * Long-Context LLM Inference" (abstract): drafting and verifying requests coexist in
 * the same batched forward pass; SFI (Figure 2 caption): each request takes fast steps
 * and, at its own boundaries, slow steps. A request id must appear in at most one of
 * the two lists.
 *   q, k_new, v_new, out, lse, scores, score_stride : as for the two calls above
 *   compact          : required when n_fast > 0
 *   max_fast_tokens  : an upper bound on S + max count + W + P over the fast requests
 *   max_dense_tokens : an upper bound on L + P over the slow requests
 *   flags            : 0 or SFI_ATTN_EARLY_KV_PREFETCH
 *   workspace        : at least sfi_mixed_workspace_size(...) bytes, zero-filled before
 *                      its first use (left zero-filled after each launch without
 *                      device error); launches sharing it must not overlap.
 * Device errors: those of sfi_fast_decode_attn and sfi_slow_dense_attn_with_scores.
 */
SFI_API sfi_status sfi_mixed_decode_attn(const sfi_attn_shape *shape, const sfi_paged_kv *kv,
                                         const sfi_compact_kv *compact, int32_t sink, int32_t recent, const void *q,
                                         const void *k_new, const void *v_new, float *out, float *lse, float *scores,
                                         int64_t score_stride, const int32_t *fast_ids, int32_t n_fast,
                                         const int32_t *slow_ids, int32_t n_slow, int32_t max_fast_tokens,
                                         int32_t max_dense_tokens, uint32_t flags, void *workspace,
                                         size_t workspace_bytes, int32_t *dev_status, void *stream);

/* Workspace bytes sfi_mixed_decode_attn needs for these arguments on the current
 * device (0 when it needs none). With one of n_fast, n_slow zero (the SFI_ATTN_RAGGED
 * plans of the single-mode calls) the size is valid for every batch size up to the
 * other, as for sfi_workspace_size. */
SFI_API size_t sfi_mixed_workspace_size(const sfi_attn_shape *shape, int32_t n_fast, int32_t n_slow,
                                        int32_t max_fast_tokens, int32_t max_dense_tokens);

/*
 * Multi-token calls. "A Sparse Glimpse of the Whole: Train-Free Self-Speculative
 * Decoding" (abstract): drafts come from the target model itself over the sparse,
 * recallable KV state; a full-context verification checks them and its per-head
 * attention statistics are recycled as the importance signal, with no extra forward.
 * Here a request carries T = num_tokens query tokens at positions L - T .. L - 1
 * (L = seq_lens[r] counts them). Query token t sees the context as it stands at length
 * L_t = L - T + t + 1 (causal).
 *   q   : bf16 [B][T][Hq][D], indexed by request id
 *   k_new, v_new : bf16 [B][T][Hkv][D] or both NULL. When given, the call first does
 *         what sfi_paged_kv_append_tokens does (the T tokens go to their page slots)
 *         and attends to the cache after that append; otherwise their K/V must already
 *         be in the pages. In the draft call the T positions must lie past the sink
 *         (L - T >= S): the compact buffer is not written.
 *   out : fp32 [B][T][Hq][D], 8-byte aligned;  lse : fp32 [B][T][Hq] or NULL
 * T x G > 16 returns SFI_ERR_UNSUPPORTED.
 */

/*
 * sfi_paged_kv_append_tokens - sfi_paged_kv_append for the T newest tokens: token t
 * of request r goes to position L_r - T + t.
 *   k_new, v_new : bf16 [B][T][Hkv][D], indexed by request id
 * Device errors: SFI_DEV_BAD_LEN (L < T), SFI_DEV_BAD_PAGE (that row is skipped).
 */
SFI_API sfi_status sfi_paged_kv_append_tokens(const sfi_attn_shape *shape, const sfi_paged_kv *kv, const void *k_new,
                                              const void *v_new, int32_t num_tokens, const int32_t *req_ids,
                                              int32_t batch, int32_t *dev_status, void *stream);

/*
 * sfi_dense_verify_attn - verification: token t of each request attends densely to
 * positions [0, L_t). When scores is non-NULL it writes the recycled statistic, for
 * every KV head kv:
 *   scores[r][kv][j] = sum over tokens t with j < L_t, sum_{g < G} of
 *                      scale * q_{t, kv*G+g} . k_{kv,j}          for j in [S, L - W)
 *   scores[r][kv][j] = -inf                                      for other j < L
 * (with T = 1 this is sfi_slow_dense_attn_with_scores). The Selector
 * (sfi_select_topk) then refreshes the selection from it; run it with the accepted
 * length, whose candidate set [S, L' - W) lies inside the scored one.
 *   scores, score_stride : as for sfi_slow_dense_attn_with_scores
 *   max_tokens : an upper bound on L + P over the batch (split planning only)
 *   num_splits, flags : as for sfi_fast_decode_attn (with k_new/v_new the append is
 *                part of the call, so SFI_ATTN_EARLY_KV_PREFETCH remains valid)
 *   workspace  : at least sfi_multi_workspace_size(shape, batch, T, max_tokens,
 *                num_splits) bytes, zero-filled before first use (kept so).
 * Device errors: SFI_DEV_BAD_LEN (also L < T, or L > score_stride), SFI_DEV_BAD_PAGE,
 * SFI_DEV_TIMEOUT.
 */
SFI_API sfi_status sfi_dense_verify_attn(const sfi_attn_shape *shape, const sfi_paged_kv *kv, int32_t sink,
                                         int32_t recent, const void *q, int32_t num_tokens, const void *k_new,
                                         const void *v_new, float *out, float *lse,
                                         float *scores, int64_t score_stride, const int32_t *req_ids, int32_t batch,
                                         int32_t max_tokens, int32_t num_splits, uint32_t flags, void *workspace,
                                         size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * sfi_sparse_draft_attn - T draft tokens over the sparse state in one pass: token t
 * sees exactly what sfi_fast_decode_attn at length L_t sees, compact rows
 * [0, min(S, L_t) + count[r]) and the recent window [max(S, L_t - W), L_t); so the
 * result equals T single-token fast steps. A non-empty selection (count[r] > 0)
 * needs L - T + 1 >= S (else SFI_DEV_K_OVERFLOW). With T = 1 the call is
 * sfi_fast_decode_attn (same kernel; flags other than SFI_ATTN_EARLY_KV_PREFETCH are
 * ignored, and the token may also lie in the sink).
 *   max_tokens : an upper bound on S + max count + W + T + P (split planning only)
 *   num_splits, flags, workspace : as for sfi_dense_verify_attn
 * Device errors: those of sfi_fast_decode_attn.
 */
SFI_API sfi_status sfi_sparse_draft_attn(const sfi_attn_shape *shape, const sfi_paged_kv *kv,
                                         const sfi_compact_kv *compact, int32_t sink, int32_t recent, const void *q,
                                         int32_t num_tokens, const void *k_new, const void *v_new, float *out,
                                         float *lse, const int32_t *req_ids,
                                         int32_t batch, int32_t max_tokens, int32_t num_splits, uint32_t flags,
                                         void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream);

/* Workspace bytes the two multi-token attention calls need on the current device,
 * valid for every batch size 1..batch as for sfi_workspace_size (0 when none; 0 also
 * on invalid input). */
SFI_API size_t sfi_multi_workspace_size(const sfi_attn_shape *shape, int32_t batch, int32_t num_tokens,
                                        int32_t max_tokens, int32_t num_splits);

/*
 * sfi_select_topk - the Selector (Figure 2 caption): for every (request r, KV
 * head kv) keep the k_eff = min(k_per_req[r], |C|) candidates of C = [S, L - W)
 * with the largest score; equal scores go to the lower position; -0 equals +0;
 * NaN ranks below every number. The result is written in ascending position
 * order, and k_eff to count_out[r].
 *   scores    : fp32 [B][Hkv][score_stride] (as written by the slow step)
 *   seq_lens  : int32 [B] (L at the slow step)
 *   k_per_req : int32 [B], 0 <= k_r <= k_cap
 *   idx_out   : int32 [B][Hkv][k_cap]; entries past k_eff are not written
 *   count_out : int32 [B]
 * Limits: |C| <= 262144 candidates per request.
 * Device errors: SFI_DEV_K_OVERFLOW (also when |C| is past the limit),
 * SFI_DEV_BAD_LEN (L > score_stride); that request's outputs are not written.
 */
SFI_API sfi_status sfi_select_topk(const float *scores, int64_t score_stride, int32_t num_kv_heads, const int32_t *seq_lens,
                           int32_t sink, int32_t recent, const int32_t *k_per_req, int32_t k_cap, int32_t *idx_out,
                           int32_t *count_out, const int32_t *req_ids, int32_t batch, int32_t *dev_status,
                           void *stream);

/*
 * sfi_compact_gather - cache reorganisation (Figure 3: sink and selected tokens
 * packed into the contiguous compact buffer). For every (request, KV head):
 *   compact row i          <- paged position i          for i < min(S, L)
 *   compact row S + t      <- paged position idx[t]     for t < count[r]
 * for both K and V, copied bit for bit. `count` is the Selector's count_out and
 * normally the same array as compact->count.
 *   idx   : int32 [B][Hkv][k_cap] ascending positions (from sfi_select_topk)
 *   count : int32 [B]
 * Device errors: SFI_DEV_BAD_LEN, SFI_DEV_BAD_PAGE, SFI_DEV_BAD_INDEX,
 * SFI_DEV_K_OVERFLOW, SFI_DEV_BAD_COMPACT (offending rows are skipped).
 */
SFI_API sfi_status sfi_compact_gather(const sfi_attn_shape *shape, const sfi_paged_kv *kv, const int32_t *idx,
                              const int32_t *count, int32_t k_cap, int32_t sink, const sfi_compact_kv *compact,
                              const int32_t *req_ids, int32_t batch, int32_t *dev_status, void *stream);

/*
 * sfi_select_compact - sfi_select_topk followed by sfi_compact_gather in one call
 * (Figure 2 caption: the Selector refreshes the selected memory; Figure 3: cache
 * reorganisation into the contiguous compact buffer): the two kernels are launched in
 * sequence on the stream, with count = count_out.
 *   scores, score_stride, k_per_req, k_cap, idx_out : as for sfi_select_topk
 *   count_out : int32 [B], normally the same array as compact->count
 *   kv->seq_lens gives L (as for both calls)
 * Device errors: those of the two calls (a request with an invalid compact layout
 * keeps its selection but is not packed).
 */
SFI_API sfi_status sfi_select_compact(const sfi_attn_shape *shape, const sfi_paged_kv *kv, const float *scores,
                                      int64_t score_stride, int32_t sink, int32_t recent, const int32_t *k_per_req,
                                      int32_t k_cap, int32_t *idx_out, int32_t *count_out,
                                      const sfi_compact_kv *compact, const int32_t *req_ids, int32_t batch,
                                      int32_t *dev_status, void *stream);

/*
 * sfi_fast_decode_attn_noalloc - the fast step of sfi_fast_decode_attn for callers
 * that cannot allocate device memory. The paper has no counterpart to this call; it
 * exists for users of this library.
 * Who needs it: sfi_fast_decode_attn wants a caller-provided device workspace for
 * its split-KV partial results. A plugin running inside a host application that owns
 * every device allocation, or a latency-critical path that must not call cudaMalloc
 * (which can synchronise the whole device), has no way to provide one. This call
 * takes the same inputs and outputs, minus the workspace, and uses instead a fixed
 * array of SFI_NOALLOC_SCRATCH_BYTES inside the library's device memory. Every GPU
 * that loads the library holds that array until the process exits.
 *   - It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - Its first call on a device looks up the array's device address on that device
 *     (cudaGetSymbolAddress, with that device current); make that first call before
 *     any stream capture.
 *   - The looked-up address is kept for the life of the process: a device reset
 *     (cudaDeviceReset) after the first call on a device is not supported.
 *   - Returns SFI_ERR_WORKSPACE when the split plan for these arguments needs more
 *     than SFI_NOALLOC_SCRATCH_BYTES (sfi_workspace_size tells the need, or
 *     sfi_mixed_workspace_size(shape, batch, 0, max_tokens, 0) with SFI_ATTN_RAGGED);
 *     reduce num_splits or the batch per call.
 *   - All calls on a device share the one array, which keeps what the last call left
 *     in it. A call whose plan uses the array (more than 8 splits, or any chunked
 *     plan of more than one chunk under SFI_ATTN_RAGGED) first zeroes its split
 *     counters with an async memset on `stream`; a plan that merges inside a
 *     thread-block cluster uses no scratch and issues no memset. Calls whose work can
 *     overlap on the GPU (for example on two streams) race on the array: order them
 *     on one stream.
 * Arguments, results and device errors are those of sfi_fast_decode_attn.
 */
#define SFI_NOALLOC_SCRATCH_BYTES (4u << 20)
SFI_API sfi_status sfi_fast_decode_attn_noalloc(const sfi_attn_shape *shape, const sfi_paged_kv *kv,
                                                const sfi_compact_kv *compact, int32_t sink, int32_t recent,
                                                const void *q, const void *k_new, const void *v_new, float *out,
                                                float *lse, const int32_t *req_ids,
                                                int32_t batch, int32_t max_tokens, int32_t num_splits, uint32_t flags,
                                                int32_t *dev_status, void *stream);

/*
 * sfi_workspace_size - bytes of workspace the attention entry points need for this
 * batch, token bound and split request on the current device, valid for every batch
 * size 1..batch (calls on a subset of the requests plan their splits for the subset):
 * one split counter per (request, KV head) at the start of the buffer, and the largest
 * block of split-KV partial states of those plans, which each call places at the end
 * of the buffer it is given. So calls with different batch sizes may share one buffer
 * (one at a time) when it holds the size for the largest of them. Returns 0 when no
 * plan needs any (at most 8 splits: the splits of a unit merge inside a thread-block
 * cluster) and on invalid input.
 */
SFI_API size_t sfi_workspace_size(const sfi_attn_shape *shape, int32_t batch, int32_t max_tokens, int32_t num_splits);

/*
 * sfi_plan_splits - the split count the attention entry points will use for these
 * arguments on the current device (for reports and tests). 0 on invalid input.
 * Automatic plans (num_splits = 0) give the (request, KV head) units about 85% of one
 * wave of two CTAs per SM; a count between 8 and 16 becomes 8. Every split keeps at
 * least four stages of 64 tokens, or three while the plan stays at most 8 splits (the
 * splits of a unit then merge inside a thread-block cluster). A plan of 2..8 splits
 * also leaves a ninth of the SM slots free in whole clusters, by the count of
 * sfi_attn_cluster_capacity, one split fewer at a time until it does. An explicit
 * num_splits is honoured down to two stages per split.
 */
SFI_API int32_t sfi_plan_splits(const sfi_attn_shape *shape, int32_t batch, int32_t max_tokens, int32_t num_splits);

/*
 * sfi_attn_cluster_capacity - how many thread-block clusters of cluster_size attention
 * CTAs (1..8) the current device holds at once (its occupancy query for the attention
 * kernel, cached per device). A cluster is placed whole on one GPC, so this can be
 * below the SM slots divided by cluster_size. 0 on invalid input, when there is no
 * device, or when the query fails.
 */
SFI_API int32_t sfi_attn_cluster_capacity(int32_t cluster_size);

/* Human-readable name of a status code (static string). */
SFI_API const char *sfi_status_string(sfi_status status);

/* SFI_VERSION of the built library. */
SFI_API int32_t sfi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SFI_H */
