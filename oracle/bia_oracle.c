/*
 * CPU oracle for batch-invariant paged-KV grouped-query attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library; the two meet only through the seeded input generators.
 *
 * What it computes is the plain definition of the attention that the pages
 * describe as a paged-KV prefill / decode wrapper over page tables and
 * qo/kv indptr arrays ("sglang PR #43612", Summary: BatchPrefillWithPagedKVCacheWrapper
 * with a fixed split-KV tile; "sglang PR #10417 [POC] Support deterministic
 * inference", Modifications: paged prefill wrapper for every prefill, fixed
 * split-KV of 2048 for decode and 4096 for prefill).  The pages print no
 * formula, so the readings below are the plainest ones the rest supports:
 *
 *   - request b owns q tokens qo_indptr[b] .. qo_indptr[b+1]-1 and
 *     kv_len = (kv_indptr[b+1]-kv_indptr[b]-1)*page_size + last_page_len[b]
 *     keys (0 when it owns no page);
 *   - key j of request b lives at page kv_indices[kv_indptr[b] + j/page_size],
 *     slot j % page_size; the caches are [num_pages, page_size, Hkv, D] bf16;
 *   - q head h reads kv head h / (Hq/Hkv) (consecutive GQA grouping);
 *   - the q tokens are the last q_len positions of the sequence, so in-call
 *     token t sits at absolute position p = kv_len - q_len + t; a causal row
 *     sees keys 0..p, a non-causal row sees all kv_len keys;
 *   - s_j = sm_scale * <q, k_j>, out = sum_j e^{s_j-m} v_j / sum_j e^{s_j-m},
 *     lse = m + ln sum_j e^{s_j-m} (natural log), m = max_j s_j;
 *   - a row that sees no key has out = 0 and lse = -inf;
 *   - an optional custom mask (the pages name none; it follows the bit-packed
 *     per-request [q_len, kv_len] mask of paged prefill wrappers) removes
 *     further keys: key j is visible to in-call token t of request b only if
 *     bit mask_indptr[b] + t*kv_len + j of the little-endian bit string is 1.
 *
 * An optional key window [key_lo, key_hi) restricts the visible keys further;
 * with the window set to one split-KV tile it yields that split's partial
 * (o_s, lse_s), which the merge below combines.  Arithmetic is fp64 on the
 * exactly decoded bf16 inputs.  Everything is a direct loop: no blocking, no
 * online softmax, no reordering beyond the definition.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_NO_MEM (-2)

/* bf16 is the upper half of an IEEE binary32: widen bit-exactly. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    int32_t num_qo_heads, num_kv_heads, head_dim, page_size;
    double sm_scale;
    int32_t causal;
    const uint16_t *q, *k_cache, *v_cache;
    const int32_t *qo_indptr, *kv_indptr, *kv_indices, *kv_last_page_len;
    int32_t batch;
    int64_t key_lo, key_hi;
    const int64_t *rows; /* pairs (global q token, q head); NULL = every row */
    int64_t n_rows;
    double *out, *lse;
    /* optional custom mask: bit (mask_indptr[b] + t*kv_len + j) of the
     * little-endian bit string `mask` says whether in-call token t of
     * request b may see key j (on top of the causal rule when causal) */
    const uint8_t *mask;
    const int64_t *mask_indptr;
} oracle_problem;

/* Whether row (request b, in-call token tl) may see key j by the custom mask. */
static int mask_allows(const oracle_problem *pb, int b, int64_t tl, int64_t kv_len, int64_t j)
{
    if (!pb->mask)
        return 1;
    int64_t bit = pb->mask_indptr[b] + tl * kv_len + j;
    return (pb->mask[bit >> 3] >> (bit & 7)) & 1;
}

static int64_t request_kv_len(const oracle_problem *pb, int b)
{
    int64_t pages = (int64_t)pb->kv_indptr[b + 1] - pb->kv_indptr[b];
    if (pages <= 0)
        return 0;
    return (pages - 1) * pb->page_size + pb->kv_last_page_len[b];
}

/* Row n of k_cache / v_cache that holds key j, kv head g, of request b. */
static const uint16_t *paged_row(const oracle_problem *pb, const uint16_t *cache, int b,
                                 int64_t j, int g)
{
    int64_t page = pb->kv_indices[pb->kv_indptr[b] + j / pb->page_size];
    int64_t slot = j % pb->page_size;
    return cache + ((page * pb->page_size + slot) * pb->num_kv_heads + g) * pb->head_dim;
}

/* The request that owns global q token t (qo_indptr is non-decreasing). */
static int owner_of_token(const oracle_problem *pb, int64_t t)
{
    int lo = 0, hi = pb->batch - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (pb->qo_indptr[mid] <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    /* skip requests with no q token that share the same start */
    while (lo + 1 < pb->batch && pb->qo_indptr[lo + 1] <= t)
        lo++;
    return lo;
}

/* One output row: global q token t, q head h.  scores is scratch of kv_len. */
static void attend_row(const oracle_problem *pb, int64_t t, int h, double *scores, double *out,
                       double *lse)
{
    const int D = pb->head_dim;
    const int G = pb->num_qo_heads / pb->num_kv_heads;
    const int g = h / G;
    const int b = owner_of_token(pb, t);
    const int64_t q_len = (int64_t)pb->qo_indptr[b + 1] - pb->qo_indptr[b];
    const int64_t kv_len = request_kv_len(pb, b);
    const int64_t p = kv_len - q_len + (t - pb->qo_indptr[b]);

    int64_t last = pb->causal ? p : kv_len - 1; /* last visible key */
    if (last > kv_len - 1)
        last = kv_len - 1;
    int64_t first = pb->key_lo > 0 ? pb->key_lo : 0;
    if (pb->key_hi - 1 < last)
        last = pb->key_hi - 1;

    const uint16_t *qrow = pb->q + (t * pb->num_qo_heads + h) * D;
    for (int d = 0; d < D; d++)
        out[d] = 0.0;
    if (last < first) {
        *lse = -INFINITY;
        return;
    }

    const int64_t tl = t - pb->qo_indptr[b];
    double m = -INFINITY;
    int any = 0;
    for (int64_t j = first; j <= last; j++) {
        if (!mask_allows(pb, b, tl, kv_len, j)) {
            scores[j - first] = -INFINITY;
            continue;
        }
        any = 1;
        const uint16_t *krow = paged_row(pb, pb->k_cache, b, j, g);
        double dot = 0.0;
        for (int d = 0; d < D; d++)
            dot += bf16_value(qrow[d]) * bf16_value(krow[d]);
        double s = pb->sm_scale * dot;
        scores[j - first] = s;
        if (s > m)
            m = s;
    }
    if (!any) {
        *lse = -INFINITY;
        return;
    }
    double denom = 0.0;
    for (int64_t j = first; j <= last; j++) {
        if (scores[j - first] == -INFINITY) {
            scores[j - first] = 0.0;
            continue;
        }
        double w = exp(scores[j - first] - m);
        scores[j - first] = w;
        denom += w;
    }
    for (int64_t j = first; j <= last; j++) {
        if (scores[j - first] == 0.0)
            continue;
        const uint16_t *vrow = paged_row(pb, pb->v_cache, b, j, g);
        double w = scores[j - first] / denom;
        for (int d = 0; d < D; d++)
            out[d] += w * bf16_value(vrow[d]);
    }
    *lse = m + log(denom);
}

typedef struct {
    const oracle_problem *pb;
    int64_t begin, end, max_kv;
    int status;
} oracle_slice;

static void *run_slice(void *arg)
{
    oracle_slice *sl = (oracle_slice *)arg;
    const oracle_problem *pb = sl->pb;
    double *scores = (double *)malloc((size_t)(sl->max_kv > 0 ? sl->max_kv : 1) * sizeof(double));
    if (!scores) {
        sl->status = ORACLE_NO_MEM;
        return NULL;
    }
    for (int64_t i = sl->begin; i < sl->end; i++) {
        int64_t t;
        int h;
        if (pb->rows) {
            t = pb->rows[2 * i];
            h = (int)pb->rows[2 * i + 1];
        } else {
            t = i / pb->num_qo_heads;
            h = (int)(i % pb->num_qo_heads);
        }
        attend_row(pb, t, h, scores, pb->out + i * pb->head_dim, pb->lse + i);
    }
    free(scores);
    sl->status = ORACLE_OK;
    return NULL;
}

/*
 * Paged GQA attention for the listed rows (or all rows when rows == NULL).
 * out: [n, D] fp64, lse: [n] fp64, n = n_rows or total_q * Hq (row-major
 * over (token, head)).  key_lo/key_hi bound the visible keys (pass 0 and
 * INT64_MAX for the plain attention).  Returns 0 or a negative code.
 */
int oracle_attention_rows_masked(int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t page_size, double sm_scale, int32_t causal,
                                 const uint16_t *q, const uint16_t *k_cache,
                                 const uint16_t *v_cache, const int32_t *qo_indptr,
                                 const int32_t *kv_indptr, const int32_t *kv_indices,
                                 const int32_t *kv_last_page_len, int32_t batch, int64_t key_lo,
                                 int64_t key_hi, const uint8_t *mask, const int64_t *mask_indptr,
                                 const int64_t *rows, int64_t n_rows, double *out, double *lse,
                                 int32_t n_threads)
{
    if (num_qo_heads <= 0 || num_kv_heads <= 0 || num_qo_heads % num_kv_heads != 0 ||
        head_dim <= 0 || page_size <= 0 || batch <= 0 || !q || !k_cache || !v_cache ||
        !qo_indptr || !kv_indptr || !kv_indices || !kv_last_page_len || !out || !lse ||
        (mask && !mask_indptr))
        return ORACLE_BAD_ARG;
    oracle_problem pb = {num_qo_heads, num_kv_heads, head_dim, page_size, sm_scale, causal,
                         q, k_cache, v_cache, qo_indptr, kv_indptr, kv_indices,
                         kv_last_page_len, batch, key_lo, key_hi, rows, n_rows, out, lse,
                         mask, mask_indptr};
    int64_t total = rows ? n_rows : (int64_t)qo_indptr[batch] * num_qo_heads;
    int64_t max_kv = 0;
    for (int b = 0; b < batch; b++) {
        int64_t kv = request_kv_len(&pb, b);
        if (kv > max_kv)
            max_kv = kv;
    }
    if (n_threads < 1)
        n_threads = 1;
    if (n_threads > 256)
        n_threads = 256;
    if (total < n_threads)
        n_threads = total > 0 ? (int32_t)total : 1;

    pthread_t th[256];
    oracle_slice sl[256];
    int started[256];
    for (int i = 0; i < n_threads; i++) {
        sl[i].pb = &pb;
        sl[i].begin = total * i / n_threads;
        sl[i].end = total * (i + 1) / n_threads;
        sl[i].max_kv = max_kv;
        sl[i].status = ORACLE_NO_MEM;
        started[i] = (n_threads > 1) && pthread_create(&th[i], NULL, run_slice, &sl[i]) == 0;
        if (!started[i])
            run_slice(&sl[i]);
    }
    int status = ORACLE_OK;
    for (int i = 0; i < n_threads; i++) {
        if (started[i])
            pthread_join(th[i], NULL);
        if (sl[i].status != ORACLE_OK)
            status = sl[i].status;
    }
    return status;
}

/* oracle_attention_rows_masked without a custom mask. */
int oracle_attention_rows(int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t page_size, double sm_scale, int32_t causal, const uint16_t *q,
                          const uint16_t *k_cache, const uint16_t *v_cache,
                          const int32_t *qo_indptr, const int32_t *kv_indptr,
                          const int32_t *kv_indices, const int32_t *kv_last_page_len,
                          int32_t batch, int64_t key_lo, int64_t key_hi, const int64_t *rows,
                          int64_t n_rows, double *out, double *lse, int32_t n_threads)
{
    return oracle_attention_rows_masked(num_qo_heads, num_kv_heads, head_dim, page_size,
                                        sm_scale, causal, q, k_cache, v_cache, qo_indptr,
                                        kv_indptr, kv_indices, kv_last_page_len, batch, key_lo,
                                        key_hi, NULL, NULL, rows, n_rows, out, lse, n_threads);
}

/*
 * The attention weights of one row: probs[j] for j in 0..kv_len-1 (0 for keys
 * the row cannot see).  Global q token t, q head h.  Used to check that the
 * weights form a distribution and respect the causal mask.
 */
int oracle_row_probs(int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                     int32_t page_size, double sm_scale, int32_t causal, const uint16_t *q,
                     const uint16_t *k_cache, const uint16_t *v_cache, const int32_t *qo_indptr,
                     const int32_t *kv_indptr, const int32_t *kv_indices,
                     const int32_t *kv_last_page_len, int32_t batch, int64_t t, int32_t h,
                     double *probs, int64_t probs_len)
{
    if (num_qo_heads <= 0 || num_kv_heads <= 0 || num_qo_heads % num_kv_heads != 0 ||
        batch <= 0 || !probs || t < 0 || t >= qo_indptr[batch] || h < 0 || h >= num_qo_heads)
        return ORACLE_BAD_ARG;
    oracle_problem pb = {num_qo_heads, num_kv_heads, head_dim, page_size, sm_scale, causal,
                         q, k_cache, v_cache, qo_indptr, kv_indptr, kv_indices,
                         kv_last_page_len, batch, 0, INT64_MAX, NULL, 0, NULL, NULL,
                         NULL, NULL};
    int b = owner_of_token(&pb, t);
    int64_t kv_len = request_kv_len(&pb, b);
    if (probs_len < kv_len)
        return ORACLE_BAD_ARG;
    const int D = head_dim;
    const int g = h / (num_qo_heads / num_kv_heads);
    const int64_t q_len = (int64_t)qo_indptr[b + 1] - qo_indptr[b];
    const int64_t p = kv_len - q_len + (t - qo_indptr[b]);
    int64_t last = causal ? p : kv_len - 1;
    if (last > kv_len - 1)
        last = kv_len - 1;
    for (int64_t j = 0; j < probs_len; j++)
        probs[j] = 0.0;
    if (last < 0)
        return ORACLE_OK;
    const uint16_t *qrow = q + (t * num_qo_heads + h) * D;
    double m = -INFINITY;
    for (int64_t j = 0; j <= last; j++) {
        const uint16_t *krow = paged_row(&pb, k_cache, b, j, g);
        double dot = 0.0;
        for (int d = 0; d < D; d++)
            dot += bf16_value(qrow[d]) * bf16_value(krow[d]);
        probs[j] = sm_scale * dot;
        if (probs[j] > m)
            m = probs[j];
    }
    double denom = 0.0;
    for (int64_t j = 0; j <= last; j++) {
        probs[j] = exp(probs[j] - m);
        denom += probs[j];
    }
    for (int64_t j = 0; j <= last; j++)
        probs[j] /= denom;
    return ORACLE_OK;
}

/*
 * Merge of attention states by their log-sum-exp, written as its plain
 * definition rather than as a fold: for row (i, h) with states s < S_i,
 *   LSE = ln sum_s e^{lse_s},  out = sum_s e^{lse_s - LSE} v_s.
 * States with lse = -inf carry no weight; a row with none has out 0 and
 * lse -inf.  v: [n, S, H, D] fp32, lse_in: [n, S, H] fp32 (natural log),
 * num_states: [n] or NULL (all S).  out: [n, H, D] fp64, lse_out: [n, H].
 * The pages fix only that the merge order is fixed ("sglang PR #10417",
 * Modifications: fixed split-KV); the value merged to is this one.
 */
int oracle_merge_states(const float *v, const float *lse_in, const int32_t *num_states,
                        int64_t n, int32_t S, int32_t H, int32_t D, double *out,
                        double *lse_out)
{
    if (!v || !lse_in || !out || !lse_out || n < 0 || S <= 0 || H <= 0 || D <= 0)
        return ORACLE_BAD_ARG;
    for (int64_t i = 0; i < n; i++) {
        int32_t cnt = num_states ? num_states[i] : S;
        if (cnt < 0 || cnt > S)
            return ORACLE_BAD_ARG;
        for (int h = 0; h < H; h++) {
            double m = -INFINITY;
            for (int s = 0; s < cnt; s++) {
                double l = lse_in[(i * S + s) * H + h];
                if (l > m)
                    m = l;
            }
            double *o = out + (i * H + h) * D;
            for (int d = 0; d < D; d++)
                o[d] = 0.0;
            if (m == -INFINITY) {
                lse_out[i * H + h] = -INFINITY;
                continue;
            }
            double sum = 0.0;
            for (int s = 0; s < cnt; s++)
                sum += exp((double)lse_in[(i * S + s) * H + h] - m);
            double total = m + log(sum);
            for (int s = 0; s < cnt; s++) {
                double w = exp((double)lse_in[(i * S + s) * H + h] - total);
                if (w == 0.0)
                    continue;
                const float *vs = v + ((i * S + s) * H + h) * D;
                for (int d = 0; d < D; d++)
                    o[d] += w * (double)vs[d];
            }
            lse_out[i * H + h] = total;
        }
    }
    return ORACLE_OK;
}

/*
 * Multi-head latent attention (MLA) over a paged latent cache, by its
 * definition.  The pages name the paged MLA wrapper their serving stack uses
 * for chunked extends of Kimi-Linear and note that it has no deterministic
 * mode ("sglang PR #43612", Summary); what it computes, in the absorbed form
 * paged MLA kernels take, is plain attention of every q head over one shared
 * latent cache:
 *   s_j = sm_scale * (<q_nope, ckv_j> + <q_pe, kpe_j>),
 *   out = sum_j softmax(s)_j * ckv_j   (the latent row doubles as the value),
 *   lse = m + ln sum_j e^{s_j - m}.
 * Token t of request b sits at position kv_len - q_len + t and, causal, sees
 * keys 0..that position.  q_nope [total_q, H, Dc], q_pe [total_q, H, Dp],
 * ckv_cache [num_pages, P, Dc], kpe_cache [num_pages, P, Dp] (bf16 bits);
 * out [total_q, H, Dc] fp64, lse [total_q, H] fp64.  key_lo / key_hi bound the
 * visible keys (a split partial).
 */
int oracle_mla(int32_t num_heads, int32_t dc, int32_t dp, int32_t page_size, double sm_scale,
               int32_t causal, const uint16_t *q_nope, const uint16_t *q_pe,
               const uint16_t *ckv_cache, const uint16_t *kpe_cache, const int32_t *qo_indptr,
               const int32_t *kv_indptr, const int32_t *kv_indices,
               const int32_t *kv_last_page_len, int32_t batch, int64_t key_lo, int64_t key_hi,
               double *out, double *lse)
{
    if (num_heads <= 0 || dc <= 0 || dp < 0 || page_size <= 0 || batch <= 0 || !q_nope ||
        (dp > 0 && (!q_pe || !kpe_cache)) || !ckv_cache || !qo_indptr || !kv_indptr ||
        !kv_indices || !kv_last_page_len || !out || !lse)
        return ORACLE_BAD_ARG;
    int64_t max_kv = 1;
    for (int b = 0; b < batch; b++) {
        int64_t pages = (int64_t)kv_indptr[b + 1] - kv_indptr[b];
        int64_t kv = pages > 0 ? (pages - 1) * page_size + kv_last_page_len[b] : 0;
        if (kv > max_kv)
            max_kv = kv;
    }
    double *scores = (double *)malloc((size_t)max_kv * sizeof(double));
    if (!scores)
        return ORACLE_NO_MEM;
    for (int b = 0; b < batch; b++) {
        int64_t pages = (int64_t)kv_indptr[b + 1] - kv_indptr[b];
        int64_t kv_len = pages > 0 ? (pages - 1) * page_size + kv_last_page_len[b] : 0;
        int64_t q_len = (int64_t)qo_indptr[b + 1] - qo_indptr[b];
        for (int64_t tl = 0; tl < q_len; tl++) {
            int64_t t = qo_indptr[b] + tl;
            int64_t p = kv_len - q_len + tl;
            int64_t last = causal ? p : kv_len - 1;
            if (last > kv_len - 1)
                last = kv_len - 1;
            if (key_hi - 1 < last)
                last = key_hi - 1;
            int64_t first = key_lo > 0 ? key_lo : 0;
            for (int h = 0; h < num_heads; h++) {
                const uint16_t *qn = q_nope + (t * num_heads + h) * dc;
                const uint16_t *qp = dp > 0 ? q_pe + (t * num_heads + h) * dp : NULL;
                double *o = out + (t * num_heads + h) * dc;
                for (int d = 0; d < dc; d++)
                    o[d] = 0.0;
                if (last < first) {
                    lse[t * num_heads + h] = -INFINITY;
                    continue;
                }
                double m = -INFINITY;
                for (int64_t j = first; j <= last; j++) {
                    int64_t page = kv_indices[kv_indptr[b] + j / page_size];
                    int64_t slot = j % page_size;
                    const uint16_t *c = ckv_cache + (page * page_size + slot) * dc;
                    double dot = 0.0;
                    for (int d = 0; d < dc; d++)
                        dot += bf16_value(qn[d]) * bf16_value(c[d]);
                    if (dp > 0) {
                        const uint16_t *kp = kpe_cache + (page * page_size + slot) * dp;
                        for (int d = 0; d < dp; d++)
                            dot += bf16_value(qp[d]) * bf16_value(kp[d]);
                    }
                    scores[j - first] = sm_scale * dot;
                    if (scores[j - first] > m)
                        m = scores[j - first];
                }
                double denom = 0.0;
                for (int64_t j = first; j <= last; j++) {
                    scores[j - first] = exp(scores[j - first] - m);
                    denom += scores[j - first];
                }
                for (int64_t j = first; j <= last; j++) {
                    int64_t page = kv_indices[kv_indptr[b] + j / page_size];
                    int64_t slot = j % page_size;
                    const uint16_t *c = ckv_cache + (page * page_size + slot) * dc;
                    double w = scores[j - first] / denom;
                    for (int d = 0; d < dc; d++)
                        o[d] += w * bf16_value(c[d]);
                }
                lse[t * num_heads + h] = m + log(denom);
            }
        }
    }
    free(scores);
    return ORACLE_OK;
}
