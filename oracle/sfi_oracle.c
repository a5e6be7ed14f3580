/*
 * CPU oracle for Slow-Fast Inference (SFI) decode attention over a sparse,
 * recallable KV memory.
 *
 * TEST INFRASTRUCTURE. This file is the plain, slow reference that the CUDA path
 * is checked against. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load it. It shares no code, header or constant with the CUDA
 * library and never calls it. Every function is fp64, single-threaded, written
 * for readability, not speed.
 *
 * Source: "Slow-Fast Inference: Training-Free Inference Acceleration via
 * Within-Sentence Support Stability" (Xie et al., 2026):
 *   - Figure 2 caption: fast steps attend to a managed sparse state
 *     "sink + selected + recent"; a slow step performs dense attention, collects
 *     masked attention logits over the allowed candidate set and lets the Selector
 *     refresh the selected memory.
 *   - Figure 3 caption (B): sink and selected tokens are packed into a contiguous
 *     compact buffer; recent tokens are read in place from paged KV.
 *   - Table 1: at 100% retention the sparse kernel equals the dense one (1.00x).
 * Readings where the page is silent (each is listed in the design notes):
 *   softmax scale 1/sqrt(D); query head h uses KV head floor(h / G); the score
 *   of a KV head is the sum over its G query heads of the scaled logit; the
 *   candidate set of a slow step at length L is [S, L - W); ties in the Selector
 *   go to the lower position; NaN ranks below every number and -0 equals +0;
 *   the selection is returned in ascending position order; the recent window of
 *   a step at length L is [max(S, L - W), L); the compact buffer keeps the sink
 *   in rows [0, min(S, L)) and the selection from row S on.
 *
 * Data formats (bytes shared with the callers, no code):
 *   bf16 values are uint16 bit patterns; widened exactly to double here.
 *   paged pools: [num_pages][Hkv][P][D]; page_row: the request's page list.
 *   query of one request: [Hq][D]; outputs: double [Hq][D] and lse double [Hq].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_EXPORT __attribute__((visibility("default")))

static double widen_bf16(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Pointer to the D values of (position pos, KV head kv) in a paged pool. */
static const uint16_t *paged_row(const uint16_t *pool, const int32_t *page_row, int pos, int kv, int Hkv,
                                 int P, int D)
{
    int page = page_row[pos / P];
    size_t row = ((size_t)page * (size_t)Hkv + (size_t)kv) * (size_t)P + (size_t)(pos % P);
    return pool + row * (size_t)D;
}

/*
 * Softmax attention of one query over an explicit list of n key/value rows:
 *   s_j = scale * q . k_j,  m = max_j s_j,  p_j = exp(s_j - m) / sum_i exp(s_i - m),
 *   o = sum_j p_j v_j,      lse = m + ln sum_j exp(s_j - m).
 * n == 0 gives o = 0 and lse = -inf.
 */
static void attend_rows(const double *q, const uint16_t *const *krows, const uint16_t *const *vrows, int n,
                        int D, double scale, double *o, double *lse)
{
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (n == 0) {
        *lse = -INFINITY;
        return;
    }
    double *s = (double *)malloc((size_t)n * sizeof(double));
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += q[d] * widen_bf16(krows[j][d]);
        s[j] = scale * acc;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int j = 0; j < n; ++j) {
        double p = exp(s[j] - m);
        l += p;
        for (int d = 0; d < D; ++d) o[d] += p * widen_bf16(vrows[j][d]);
    }
    for (int d = 0; d < D; ++d) o[d] /= l;
    *lse = m + log(l);
    free(s);
}

static void widen_query(const uint16_t *q_head, int D, double *out)
{
    for (int d = 0; d < D; ++d) out[d] = widen_bf16(q_head[d]);
}

static double default_scale(double scale, int D) { return scale > 0.0 ? scale : 1.0 / sqrt((double)D); }

/*
 * Dense decode attention (the slow step's attention and the full-KV baseline):
 * every query head h attends to positions [0, L) of KV head floor(h / G).
 */
ORACLE_EXPORT void oracle_dense_attn(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                                     const int32_t *page_row, int L, int Hq, int Hkv, int D, int P, double scale,
                                     double *out, double *lse)
{
    int G = Hq / Hkv;
    scale = default_scale(scale, D);
    const uint16_t **kr = (const uint16_t **)malloc((size_t)(L > 0 ? L : 1) * sizeof(void *));
    const uint16_t **vr = (const uint16_t **)malloc((size_t)(L > 0 ? L : 1) * sizeof(void *));
    double *qd = (double *)malloc((size_t)D * sizeof(double));
    for (int h = 0; h < Hq; ++h) {
        int kv = h / G;
        for (int j = 0; j < L; ++j) {
            kr[j] = paged_row(k_pool, page_row, j, kv, Hkv, P, D);
            vr[j] = paged_row(v_pool, page_row, j, kv, Hkv, P, D);
        }
        widen_query(q + (size_t)h * D, D, qd);
        attend_rows(qd, kr, vr, L, D, scale, out + (size_t)h * D, lse + h);
    }
    free(kr);
    free(vr);
    free(qd);
}

/*
 * Dense attention restricted to an explicit position set per KV head
 * (positions [Hkv][n_per_head], each row n entries): "dense attention with all
 * other positions masked".
 */
ORACLE_EXPORT void oracle_index_attn(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                                     const int32_t *page_row, const int32_t *positions, int n, int Hq, int Hkv,
                                     int D, int P, double scale, double *out, double *lse)
{
    int G = Hq / Hkv;
    scale = default_scale(scale, D);
    const uint16_t **kr = (const uint16_t **)malloc((size_t)(n > 0 ? n : 1) * sizeof(void *));
    const uint16_t **vr = (const uint16_t **)malloc((size_t)(n > 0 ? n : 1) * sizeof(void *));
    double *qd = (double *)malloc((size_t)D * sizeof(double));
    for (int h = 0; h < Hq; ++h) {
        int kv = h / G;
        const int32_t *pos = positions + (size_t)kv * n;
        for (int j = 0; j < n; ++j) {
            kr[j] = paged_row(k_pool, page_row, pos[j], kv, Hkv, P, D);
            vr[j] = paged_row(v_pool, page_row, pos[j], kv, Hkv, P, D);
        }
        widen_query(q + (size_t)h * D, D, qd);
        attend_rows(qd, kr, vr, n, D, scale, out + (size_t)h * D, lse + h);
    }
    free(kr);
    free(vr);
    free(qd);
}

/*
 * Masked logits collected by the slow step, one row per KV head:
 *   score[kv][j] = fp32( sum_{g < G} scale * q_{kv*G+g} . k_{kv, j} )  for j in C = [S, L - W)
 *   score[kv][j] = -inf                                                for j in [0, L) outside C
 * The sum is formed in double and rounded once to float (nearest-even).
 * Rows have stride `stride` floats; entries at j >= L are left untouched.
 */
ORACLE_EXPORT void oracle_group_scores(const uint16_t *q, const uint16_t *k_pool, const int32_t *page_row, int L,
                                       int S, int W, int Hq, int Hkv, int D, int P, double scale, float *scores,
                                       long stride)
{
    int G = Hq / Hkv;
    scale = default_scale(scale, D);
    int c_lo = S, c_hi = L - W;
    double *qd = (double *)malloc((size_t)G * (size_t)D * sizeof(double));
    for (int kv = 0; kv < Hkv; ++kv) {
        for (int g = 0; g < G; ++g) widen_query(q + (size_t)(kv * G + g) * D, D, qd + (size_t)g * D);
        float *row = scores + (size_t)kv * (size_t)stride;
        for (int j = 0; j < L; ++j) {
            if (j < c_lo || j >= c_hi) {
                row[j] = -INFINITY;
                continue;
            }
            const uint16_t *k = paged_row(k_pool, page_row, j, kv, Hkv, P, D);
            double sigma = 0.0;
            for (int g = 0; g < G; ++g) {
                double acc = 0.0;
                for (int d = 0; d < D; ++d) acc += qd[(size_t)g * D + d] * widen_bf16(k[d]);
                sigma += scale * acc;
            }
            row[j] = (float)sigma;
        }
    }
    free(qd);
}

/* ---- Selector: top-k by (score descending, position ascending) ---------------- */

static const float *g_sort_scores; /* comparator context (single-threaded oracle) */

/* Total order on candidates: higher score first; NaN below every number;
 * -0 == +0 (C float comparison); equal scores -> lower position first. */
static int selector_order(const void *a, const void *b)
{
    int ia = *(const int32_t *)a, ib = *(const int32_t *)b;
    float sa = g_sort_scores[ia], sb = g_sort_scores[ib];
    int na = isnan(sa), nb = isnan(sb);
    if (na != nb) return na ? 1 : -1; /* the NaN one goes after */
    if (!na) {
        if (sa > sb) return -1;
        if (sa < sb) return 1;
    }
    return (ia > ib) - (ia < ib);
}

static int ascending_int(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/*
 * Selector for one (request, KV head): among candidates C = [S, L - W) keep the
 * k_eff = min(k, |C|) best under the order above, returned as positions in
 * ascending order. Brute force: sort all of C, take the head, sort it by position.
 * Returns k_eff.
 */
ORACLE_EXPORT int oracle_select_topk(const float *score_row, int L, int S, int W, int k, int32_t *idx_out)
{
    int n = L - W - S;
    if (n <= 0 || k <= 0) return 0;
    int32_t *cand = (int32_t *)malloc((size_t)n * sizeof(int32_t));
    for (int i = 0; i < n; ++i) cand[i] = S + i;
    g_sort_scores = score_row;
    qsort(cand, (size_t)n, sizeof(int32_t), selector_order);
    int keff = k < n ? k : n;
    memcpy(idx_out, cand, (size_t)keff * sizeof(int32_t));
    qsort(idx_out, (size_t)keff, sizeof(int32_t), ascending_int);
    free(cand);
    return keff;
}

/*
 * Cache reorganisation for one request: for every KV head, compact rows
 *   [0, min(S, L))      <- positions 0 .. min(S, L) - 1  (the sink)
 *   [S, S + k_eff)      <- positions idx[kv][0 .. k_eff)  (the selection)
 * copied bit for bit from the paged pools. ck, cv: [Hkv][cap][D].
 * idx: [Hkv][idx_stride].
 */
ORACLE_EXPORT void oracle_compact(const uint16_t *k_pool, const uint16_t *v_pool, const int32_t *page_row, int L,
                                  int S, const int32_t *idx, int idx_stride, int k_eff, int Hkv, int D, int P,
                                  uint16_t *ck, uint16_t *cv, int cap)
{
    int ns = S < L ? S : L;
    for (int kv = 0; kv < Hkv; ++kv) {
        uint16_t *kdst = ck + (size_t)kv * (size_t)cap * (size_t)D;
        uint16_t *vdst = cv + (size_t)kv * (size_t)cap * (size_t)D;
        for (int i = 0; i < ns; ++i) {
            memcpy(kdst + (size_t)i * D, paged_row(k_pool, page_row, i, kv, Hkv, P, D), (size_t)D * 2);
            memcpy(vdst + (size_t)i * D, paged_row(v_pool, page_row, i, kv, Hkv, P, D), (size_t)D * 2);
        }
        for (int t = 0; t < k_eff; ++t) {
            int pos = idx[(size_t)kv * idx_stride + t];
            memcpy(kdst + (size_t)(S + t) * D, paged_row(k_pool, page_row, pos, kv, Hkv, P, D), (size_t)D * 2);
            memcpy(vdst + (size_t)(S + t) * D, paged_row(v_pool, page_row, pos, kv, Hkv, P, D), (size_t)D * 2);
        }
    }
}

/*
 * Fast step for one request at length L: each query head attends to
 *   compact rows [0, min(S, L) + count)          (sink + selected, contiguous)
 *   followed by paged positions [max(S, L - W), L) (recent window, read in place)
 * of its KV head, with one softmax over the whole list. ck, cv: [Hkv][cap][D].
 */
ORACLE_EXPORT void oracle_fast_attn(const uint16_t *q, const uint16_t *ck, const uint16_t *cv, int cap, int count,
                                    const uint16_t *k_pool, const uint16_t *v_pool, const int32_t *page_row, int L,
                                    int S, int W, int Hq, int Hkv, int D, int P, double scale, double *out,
                                    double *lse)
{
    int G = Hq / Hkv;
    scale = default_scale(scale, D);
    int ns = S < L ? S : L;
    int n_compact = ns + count;
    int rs = (L - W) > S ? (L - W) : S;
    int n_recent = L > rs ? L - rs : 0;
    int n = n_compact + n_recent;
    const uint16_t **kr = (const uint16_t **)malloc((size_t)(n > 0 ? n : 1) * sizeof(void *));
    const uint16_t **vr = (const uint16_t **)malloc((size_t)(n > 0 ? n : 1) * sizeof(void *));
    double *qd = (double *)malloc((size_t)D * sizeof(double));
    for (int h = 0; h < Hq; ++h) {
        int kv = h / G;
        const uint16_t *kb = ck + (size_t)kv * (size_t)cap * (size_t)D;
        const uint16_t *vb = cv + (size_t)kv * (size_t)cap * (size_t)D;
        for (int i = 0; i < n_compact; ++i) {
            kr[i] = kb + (size_t)i * D;
            vr[i] = vb + (size_t)i * D;
        }
        for (int i = 0; i < n_recent; ++i) {
            kr[n_compact + i] = paged_row(k_pool, page_row, rs + i, kv, Hkv, P, D);
            vr[n_compact + i] = paged_row(v_pool, page_row, rs + i, kv, Hkv, P, D);
        }
        widen_query(q + (size_t)h * D, D, qd);
        attend_rows(qd, kr, vr, n, D, scale, out + (size_t)h * D, lse + h);
    }
    free(kr);
    free(vr);
    free(qd);
}

/*
 * Split-KV evaluation of dense attention for one query head (flash-decoding):
 * positions [0, L) are cut at bounds[0] = 0 < bounds[1] < ... < bounds[nchunks] = L;
 * each chunk c yields (m_c, l_c, o~_c) with m_c = max s, l_c = sum exp(s - m_c),
 * o~_c = sum exp(s - m_c) v; then m = max m_c, l = sum l_c exp(m_c - m),
 * o = sum o~_c exp(m_c - m) / l, lse = m + ln l. Empty chunks have m_c = -inf
 * and contribute nothing.
 */
ORACLE_EXPORT void oracle_split_merge_attn(const uint16_t *q_head, int kv, const uint16_t *k_pool,
                                           const uint16_t *v_pool, const int32_t *page_row, const int32_t *bounds,
                                           int nchunks, int Hkv, int D, int P, double scale, double *out,
                                           double *lse)
{
    scale = default_scale(scale, D);
    double *qd = (double *)malloc((size_t)D * sizeof(double));
    double *mc = (double *)malloc((size_t)nchunks * sizeof(double));
    double *lc = (double *)malloc((size_t)nchunks * sizeof(double));
    double *oc = (double *)calloc((size_t)nchunks * (size_t)D, sizeof(double));
    widen_query(q_head, D, qd);
    for (int c = 0; c < nchunks; ++c) {
        int lo = bounds[c], hi = bounds[c + 1];
        double m = -INFINITY;
        for (int j = lo; j < hi; ++j) {
            const uint16_t *k = paged_row(k_pool, page_row, j, kv, Hkv, P, D);
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += qd[d] * widen_bf16(k[d]);
            double s = scale * acc;
            if (s > m) m = s;
        }
        double l = 0.0;
        for (int j = lo; j < hi; ++j) {
            const uint16_t *k = paged_row(k_pool, page_row, j, kv, Hkv, P, D);
            const uint16_t *v = paged_row(v_pool, page_row, j, kv, Hkv, P, D);
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += qd[d] * widen_bf16(k[d]);
            double p = exp(scale * acc - m);
            l += p;
            for (int d = 0; d < D; ++d) oc[(size_t)c * D + d] += p * widen_bf16(v[d]);
        }
        mc[c] = m;
        lc[c] = l;
    }
    double m = -INFINITY;
    for (int c = 0; c < nchunks; ++c)
        if (mc[c] > m) m = mc[c];
    double l = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int c = 0; c < nchunks; ++c) {
        if (lc[c] == 0.0) continue;
        double w = exp(mc[c] - m);
        l += lc[c] * w;
        for (int d = 0; d < D; ++d) out[d] += oc[(size_t)c * D + d] * w;
    }
    for (int d = 0; d < D; ++d) out[d] /= l;
    *lse = m + log(l);
    free(qd);
    free(mc);
    free(lc);
    free(oc);
}

/*
 * Paged append: the current token of a request (length L after the append) goes
 * to position L - 1, i.e. slot (L - 1) % P of page page_row[(L - 1) / P].
 * k_new, v_new: [Hkv][D].
 */
ORACLE_EXPORT void oracle_paged_append(uint16_t *k_pool, uint16_t *v_pool, const int32_t *page_row, int L,
                                       const uint16_t *k_new, const uint16_t *v_new, int Hkv, int D, int P)
{
    int pos = L - 1;
    for (int kv = 0; kv < Hkv; ++kv) {
        uint16_t *kd = (uint16_t *)paged_row(k_pool, page_row, pos, kv, Hkv, P, D);
        uint16_t *vd = (uint16_t *)paged_row(v_pool, page_row, pos, kv, Hkv, P, D);
        memcpy(kd, k_new + (size_t)kv * D, (size_t)D * 2);
        memcpy(vd, v_new + (size_t)kv * D, (size_t)D * 2);
    }
}

/*
 * Verification of T drafted tokens ("A Sparse Glimpse of the Whole: Train-Free
 * Self-Speculative Decoding", abstract: drafts come from the sparse, recallable KV
 * state; full-context verification produces the per-head attention statistics that
 * are recycled as the importance signal). The T tokens occupy positions
 * L - T .. L - 1 (L counts them); query token t attends causally to positions
 * [0, L - T + t]. q: [T][Hq][D]; out: [T][Hq][D]; lse: [T][Hq].
 */
ORACLE_EXPORT void oracle_verify_attn(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                                      const int32_t *page_row, int L, int T, int Hq, int Hkv, int D, int P,
                                      double scale, double *out, double *lse)
{
    for (int t = 0; t < T; ++t)
        oracle_dense_attn(q + (size_t)t * Hq * D, k_pool, v_pool, page_row, L - T + t + 1, Hq, Hkv, D, P, scale,
                          out + (size_t)t * Hq * D, lse + (size_t)t * Hq);
}

/*
 * T query tokens over the sparse state (drafting several tokens in one pass): token
 * t sees what a fast step at length L_t = L - T + t + 1 sees, the compact rows and
 * the recent window [max(S, L_t - W), L_t). q: [T][Hq][D]; out: [T][Hq][D];
 * lse: [T][Hq]. A non-empty selection needs L - T + 1 >= S.
 */
ORACLE_EXPORT void oracle_fast_multi_attn(const uint16_t *q, const uint16_t *ck, const uint16_t *cv, int cap,
                                          int count, const uint16_t *k_pool, const uint16_t *v_pool,
                                          const int32_t *page_row, int L, int T, int S, int W, int Hq, int Hkv,
                                          int D, int P, double scale, double *out, double *lse)
{
    for (int t = 0; t < T; ++t)
        oracle_fast_attn(q + (size_t)t * Hq * D, ck, cv, cap, count, k_pool, v_pool, page_row, L - T + t + 1, S, W,
                         Hq, Hkv, D, P, scale, out + (size_t)t * Hq * D, lse + (size_t)t * Hq);
}

/*
 * Statistics of a verification: for every KV head kv and candidate j in
 * C = [S, L - W), the scaled logit summed over the G query heads of the group and
 * over the query tokens t that see j (j <= L - T + t); -inf at the other positions
 * below L. Formed in double, rounded once to float. Rows have stride `stride`.
 */
ORACLE_EXPORT void oracle_verify_scores(const uint16_t *q, const uint16_t *k_pool, const int32_t *page_row, int L,
                                        int T, int S, int W, int Hq, int Hkv, int D, int P, double scale,
                                        float *scores, long stride)
{
    int G = Hq / Hkv;
    scale = default_scale(scale, D);
    double *qd = (double *)malloc((size_t)T * G * D * sizeof(double));
    for (int kv = 0; kv < Hkv; ++kv) {
        for (int t = 0; t < T; ++t)
            for (int g = 0; g < G; ++g)
                widen_query(q + ((size_t)t * Hq + (size_t)(kv * G + g)) * D, D, qd + ((size_t)t * G + g) * D);
        float *row = scores + (size_t)kv * (size_t)stride;
        for (int j = 0; j < L; ++j) {
            if (j < S || j >= L - W) {
                row[j] = -INFINITY;
                continue;
            }
            const uint16_t *k = paged_row(k_pool, page_row, j, kv, Hkv, P, D);
            double sigma = 0.0;
            for (int t = 0; t < T; ++t) {
                if (j > L - T + t) continue; /* not visible to query token t */
                for (int g = 0; g < G; ++g) {
                    double acc = 0.0;
                    for (int d = 0; d < D; ++d) acc += qd[((size_t)t * G + g) * D + d] * widen_bf16(k[d]);
                    sigma += scale * acc;
                }
            }
            row[j] = (float)sigma;
        }
    }
    free(qd);
}

/*
 * Append of T tokens: request positions L - T .. L - 1 (L counts them) receive
 * k_new[t], v_new[t] ([T][Hkv][D]).
 */
ORACLE_EXPORT void oracle_paged_append_tokens(uint16_t *k_pool, uint16_t *v_pool, const int32_t *page_row, int L,
                                              int T, const uint16_t *k_new, const uint16_t *v_new, int Hkv, int D,
                                              int P)
{
    for (int t = 0; t < T; ++t)
        oracle_paged_append(k_pool, v_pool, page_row, L - T + t + 1, k_new + (size_t)t * Hkv * D,
                            v_new + (size_t)t * Hkv * D, Hkv, D, P);
}

/*
 * Slow/fast schedule (Figure 2 caption: a slow step fires on a boundary token or
 * when a fixed refresh interval is reached). For each request, step t is slow if
 * it is the request's first step, if boundary[t][b] is set, or if `interval`
 * steps have passed since the last slow step; otherwise fast.
 * modes_out[t][b]: 1 = slow, 0 = fast.
 */
ORACLE_EXPORT void oracle_schedule(const uint8_t *boundary, int steps, int batch, int interval, uint8_t *modes_out)
{
    for (int b = 0; b < batch; ++b) {
        int last_slow = 0;
        for (int t = 0; t < steps; ++t) {
            int slow = (t == 0) || boundary[(size_t)t * batch + b] || (t - last_slow >= interval);
            modes_out[(size_t)t * batch + b] = (uint8_t)slow;
            if (slow) last_slow = t;
        }
    }
}
