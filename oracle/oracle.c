/*
 * CPU fp64 oracle for paged KV append + causal attention with a cache offset.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the test suite, the smoke check and the CPU-baseline leg
 * of the benchmark use it.  It shares no code, header or constant with the CUDA
 * library; it is written as the plain definition, with no blocking, fusion or
 * reordering, so that it can be checked against the pages by eye.
 *
 * Sources (web pages, cited by title and section):
 *  - "Chunked prefill" (k4i.top), section "Why chunking does not change the
 *    result" (#correctness): token i attends to every position j <= i; the
 *    cached prefix and the current chunk are two parts of one softmax; after a
 *    chunk the new k, v vectors are appended to the KV cache
 *    (K_cache += [k_{(s-1)C+1} .. k_{sC}]).
 *  - same page, "IO overhead" (#io-overhead): the append writes C x 2 (K and V)
 *    x n_h x d_h x 2 bytes per layer.
 *  - "Accelerating Sonar through speculation" (Perplexity), section EAGLE:
 *    verifying a tree of draft tokens needs a custom attention mask; each
 *    draft token is scored against the accepted prefix and its own branch.
 *  - "Disaggregated prefill and decode" (Perplexity), section "Sharded KV cache
 *    transfers" and its figure "NHD and HND KV cache layouts": in the HND
 *    layout the head dimension precedes the token dimension inside a page, so
 *    each head's slice of a page is contiguous and a page is one block.
 *
 * Layout read here: the pool is [num_pages][2 (K, V)][Hkv][page_size][d] bf16.
 * Page table: request r owns page_indices[kv_indptr[r] .. kv_indptr[r+1]);
 * its length is kv_len = (npages-1)*page_size + last_page_len[r] (0 if no page).
 * kv_len counts the tokens present AFTER the append (cached + new).
 * Causal alignment: new token i (0-based within the request's qo_len) sits at
 * absolute position kv_len - qo_len + i and attends to keys j <= that position.
 * GQA: query head h reads kv head floor(h * Hkv / Hq).
 *
 * Parity pins live in tests/test_oracle.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
    OR_OK = 0,
    OR_ERR_ARG = -1,
    OR_ERR_SHAPE = -2,
    OR_ERR_PAGE = -3,
};

/* bf16 bit pattern -> exact double (bf16 is the top half of an IEEE float). */
static double bf16_to_f64(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Flat element index of pool[page][kv][head][slot][c] in the HND layout. */
static int64_t hnd_index(int64_t page, int kv, int head, int slot, int c,
                         int Hkv, int P, int d)
{
    return ((((page * 2 + kv) * (int64_t)Hkv + head) * P + slot) * (int64_t)d) + c;
}

/* kv_len of request r from its page count and last-page fill. */
static int64_t request_kv_len(const int32_t *kv_indptr, const int32_t *last_page_len,
                              int r, int P)
{
    int64_t np = (int64_t)kv_indptr[r + 1] - kv_indptr[r];
    if (np <= 0)
        return 0;
    return (np - 1) * P + last_page_len[r];
}

static int check_table(const int32_t *qo_indptr, const int32_t *kv_indptr,
                       const int32_t *page_indices, const int32_t *last_page_len,
                       int batch, int64_t num_pages, int P)
{
    if (batch < 0)
        return OR_ERR_ARG;
    if (qo_indptr[0] != 0 || kv_indptr[0] != 0)
        return OR_ERR_SHAPE;
    for (int r = 0; r < batch; ++r) {
        int64_t nq = (int64_t)qo_indptr[r + 1] - qo_indptr[r];
        int64_t np = (int64_t)kv_indptr[r + 1] - kv_indptr[r];
        if (nq < 0 || np < 0)
            return OR_ERR_SHAPE;
        if (np > 0 && (last_page_len[r] < 1 || last_page_len[r] > P))
            return OR_ERR_SHAPE;
        if (nq > request_kv_len(kv_indptr, last_page_len, r, P))
            return OR_ERR_SHAPE;
        for (int64_t i = kv_indptr[r]; i < kv_indptr[r + 1]; ++i)
            if (page_indices[i] < 0 || page_indices[i] >= num_pages)
                return OR_ERR_PAGE;
    }
    return OR_OK;
}

/*
 * Page append ("Chunked prefill", #correctness: K_cache += [k ...]).
 * For each request r and each of its n_new = append_indptr[r+1]-append_indptr[r]
 * new tokens t, the token lands at position pos = kv_len - n_new + t, i.e. in
 * page page_indices[kv_indptr[r] + pos / P] at slot pos % P, for every kv head.
 * A bit copy: the bf16 patterns are stored unchanged.
 */
int oracle_kv_append(uint16_t *pool, int64_t num_pages,
                     const uint16_t *k_new, const uint16_t *v_new,
                     const int32_t *append_indptr, const int32_t *page_indices,
                     const int32_t *kv_indptr, const int32_t *last_page_len,
                     int batch, int Hkv, int d, int P)
{
    int st = check_table(append_indptr, kv_indptr, page_indices, last_page_len,
                         batch, num_pages, P);
    if (st != OR_OK)
        return st;
    for (int r = 0; r < batch; ++r) {
        int64_t n_new = (int64_t)append_indptr[r + 1] - append_indptr[r];
        int64_t kv_len = request_kv_len(kv_indptr, last_page_len, r, P);
        for (int64_t t = 0; t < n_new; ++t) {
            int64_t pos = kv_len - n_new + t;
            int64_t page = page_indices[kv_indptr[r] + pos / P];
            int slot = (int)(pos % P);
            int64_t row = (int64_t)append_indptr[r] + t;
            for (int h = 0; h < Hkv; ++h)
                for (int c = 0; c < d; ++c) {
                    int64_t src = (row * Hkv + h) * (int64_t)d + c;
                    pool[hnd_index(page, 0, h, slot, c, Hkv, P, d)] = k_new[src];
                    pool[hnd_index(page, 1, h, slot, c, Hkv, P, d)] = v_new[src];
                }
        }
    }
    return OR_OK;
}

/* Paged gather of one key or value vector: token j of request r, kv head h. */
static const uint16_t *paged_row(const uint16_t *pool, const int32_t *page_indices,
                                 const int32_t *kv_indptr, int r, int64_t j, int kv,
                                 int h, int Hkv, int P, int d)
{
    int64_t page = page_indices[kv_indptr[r] + j / P];
    return pool + hnd_index(page, kv, h, (int)(j % P), 0, Hkv, P, d);
}

/*
 * Visibility of key j under a draft-tree mask (EAGLE section: tree
 * verification uses a custom attention mask).  The request's new tokens
 * t = 0 .. qo_len-1 sit at absolute positions draft0 + t.  New token `tok`
 * sees every cached key (j < draft0), itself, and each earlier new token
 * t < tok whose bit is set in its mask row (word t / 32, bit t % 32), and no
 * later new token.  mrow == NULL: every key is visible.
 */
static int tree_visible(const uint32_t *mrow, int64_t draft0, int64_t tok, int64_t j)
{
    if (!mrow || j < draft0)
        return 1;
    int64_t t = j - draft0;
    if (t == tok)
        return 1;
    if (t > tok)
        return 0;
    return (int)((mrow[t / 32] >> (t % 32)) & 1u);
}

/*
 * softmax(q . K^T * sm_scale) V over the visible keys in [lo, hi) of request
 * r, kv head h (all of them when mrow is NULL; see tree_visible):
 *   s_j = sm_scale * sum_c q_c K[j][c]
 *   w_j = exp(s_j - max s) / sum_j' exp(s_j' - max s)
 *   o   = sum_j w_j V[j]          lse = max s + ln sum_j exp(s_j - max s)
 * An empty set gives o = 0 and lse = -inf (the identity of softmax_merge).
 * When w is non-NULL the weights are stored at w[j - lo] (0 for hidden keys).
 */
static void attend(const double *qv, const uint16_t *pool, const int32_t *page_indices,
                   const int32_t *kv_indptr, int r, int h_kv, int64_t lo, int64_t hi,
                   double sm_scale, int Hkv, int P, int d, const uint32_t *mrow,
                   int64_t draft0, int64_t tok, double *o, double *lse, double *w,
                   double *scratch)
{
    for (int c = 0; c < d; ++c)
        o[c] = 0.0;
    double m = -INFINITY;
    int64_t seen = 0;
    for (int64_t j = lo; j < hi; ++j) {
        if (!tree_visible(mrow, draft0, tok, j))
            continue;
        const uint16_t *k = paged_row(pool, page_indices, kv_indptr, r, j, 0, h_kv, Hkv, P, d);
        double s = 0.0;
        for (int c = 0; c < d; ++c)
            s += qv[c] * bf16_to_f64(k[c]);
        s *= sm_scale;
        scratch[j - lo] = s;
        if (s > m)
            m = s;
        ++seen;
    }
    if (seen == 0) {
        *lse = -INFINITY;
        for (int64_t j = lo; w && j < hi; ++j)
            w[j - lo] = 0.0;
        return;
    }
    double z = 0.0;
    for (int64_t j = lo; j < hi; ++j) {
        if (!tree_visible(mrow, draft0, tok, j))
            continue;
        double e = exp(scratch[j - lo] - m);
        scratch[j - lo] = e;
        z += e;
    }
    for (int64_t j = lo; j < hi; ++j) {
        if (!tree_visible(mrow, draft0, tok, j)) {
            if (w)
                w[j - lo] = 0.0;
            continue;
        }
        double wj = scratch[j - lo] / z;
        if (w)
            w[j - lo] = wj;
        const uint16_t *v = paged_row(pool, page_indices, kv_indptr, r, j, 1, h_kv, Hkv, P, d);
        for (int c = 0; c < d; ++c)
            o[c] += wj * bf16_to_f64(v[c]);
    }
    *lse = m + log(z);
}

/* Request that owns q row `row` (binary search over qo_indptr). */
static int row_request(const int32_t *qo_indptr, int batch, int64_t row)
{
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (qo_indptr[mid] <= row)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

/*
 * Batch attention by definition.  q: [nnz_qo][Hq][d] bf16.  out: [nnz_qo][Hq][d]
 * fp64, lse: [nnz_qo][Hq] fp64 (natural log; may be NULL).  When sel_rows is
 * non-NULL only the n_sel listed q rows are computed (all heads of each); the
 * outputs are then packed [n_sel][Hq][d].  pairs_out (may be NULL) receives the
 * number of (query token, key) pairs attended, summed over the computed rows
 * (per query head group, i.e. not multiplied by Hq).
 * tree_mask (may be NULL): uint32 [nnz_qo][mask_words] draft-tree mask rows
 * (see tree_visible); it needs causal = 1 and qo_len <= 32 * mask_words.
 */
int oracle_attention(const uint16_t *q, const uint16_t *pool, int64_t num_pages,
                     const int32_t *qo_indptr, const int32_t *kv_indptr,
                     const int32_t *page_indices, const int32_t *last_page_len,
                     int batch, int Hq, int Hkv, int d, int P, int causal,
                     const uint32_t *tree_mask, int mask_words,
                     double sm_scale, const int64_t *sel_rows, int64_t n_sel,
                     double *out, double *lse, int64_t *pairs_out)
{
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || P <= 0)
        return OR_ERR_ARG;
    int st = check_table(qo_indptr, kv_indptr, page_indices, last_page_len, batch,
                         num_pages, P);
    if (st != OR_OK)
        return st;
    if (tree_mask) {
        if (!causal || mask_words < 1)
            return OR_ERR_ARG;
        for (int r = 0; r < batch; ++r)
            if ((int64_t)qo_indptr[r + 1] - qo_indptr[r] > 32 * (int64_t)mask_words)
                return OR_ERR_SHAPE;
    }
    int64_t nnz = batch > 0 ? qo_indptr[batch] : 0;
    int64_t nrows = sel_rows ? n_sel : nnz;
    int64_t max_kv = 0;
    for (int r = 0; r < batch; ++r) {
        int64_t kv = request_kv_len(kv_indptr, last_page_len, r, P);
        if (kv > max_kv)
            max_kv = kv;
    }
    for (int64_t i = 0; sel_rows && i < n_sel; ++i)
        if (sel_rows[i] < 0 || sel_rows[i] >= nnz)
            return OR_ERR_ARG;
    int64_t pairs = 0;
#pragma omp parallel reduction(+ : pairs)
    {
        double *scratch = (double *)malloc(sizeof(double) * (size_t)(max_kv > 0 ? max_kv : 1));
        double *qv = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int64_t task = 0; task < nrows * Hq; ++task) {
            int64_t idx = task / Hq;
            int h = (int)(task % Hq);
            int64_t row = sel_rows ? sel_rows[idx] : idx;
            int r = row_request(qo_indptr, batch, row);
            int64_t qo_len = (int64_t)qo_indptr[r + 1] - qo_indptr[r];
            int64_t kv_len = request_kv_len(kv_indptr, last_page_len, r, P);
            int64_t i = row - qo_indptr[r];
            int64_t pos = kv_len - qo_len + i;            /* absolute position */
            int64_t hi = causal ? pos + 1 : kv_len;       /* keys j <= pos */
            int h_kv = (int)((int64_t)h * Hkv / Hq);
            for (int c = 0; c < d; ++c)
                qv[c] = bf16_to_f64(q[(row * Hq + h) * (int64_t)d + c]);
            const uint32_t *mrow = tree_mask ? tree_mask + row * (int64_t)mask_words : NULL;
            double l;
            attend(qv, pool, page_indices, kv_indptr, r, h_kv, 0, hi, sm_scale, Hkv, P, d,
                   mrow, kv_len - qo_len, i, out + (idx * Hq + h) * (int64_t)d, &l, NULL,
                   scratch);
            if (lse)
                lse[idx * Hq + h] = l;
            if (h == 0)
                for (int64_t j = 0; j < hi; ++j)
                    pairs += tree_visible(mrow, kv_len - qo_len, i, j);
        }
        free(scratch);
        free(qv);
    }
    if (pairs_out)
        *pairs_out = pairs;
    return OR_OK;
}

/*
 * One query vector (row `row`, head h) over an explicit key range [lo, hi) of its
 * request, with no causal rule applied: the building block of the
 * "softmax_merge" decomposition of #correctness (attention over the cache, then
 * over the chunk).  w (may be NULL) receives hi-lo weights.
 */
int oracle_attention_keyrange(const uint16_t *q, const uint16_t *pool, int64_t num_pages,
                              const int32_t *qo_indptr, const int32_t *kv_indptr,
                              const int32_t *page_indices, const int32_t *last_page_len,
                              int batch, int Hq, int Hkv, int d, int P, double sm_scale,
                              int64_t row, int h, int64_t lo, int64_t hi,
                              double *o, double *lse, double *w)
{
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || h < 0 || h >= Hq)
        return OR_ERR_ARG;
    int st = check_table(qo_indptr, kv_indptr, page_indices, last_page_len, batch,
                         num_pages, P);
    if (st != OR_OK)
        return st;
    if (row < 0 || batch <= 0 || row >= qo_indptr[batch])
        return OR_ERR_ARG;
    int r = row_request(qo_indptr, batch, row);
    int64_t kv_len = request_kv_len(kv_indptr, last_page_len, r, P);
    if (lo < 0 || hi > kv_len || lo > hi)
        return OR_ERR_ARG;
    double *qv = (double *)malloc(sizeof(double) * (size_t)d);
    double *scratch = (double *)malloc(sizeof(double) * (size_t)(hi - lo > 0 ? hi - lo : 1));
    for (int c = 0; c < d; ++c)
        qv[c] = bf16_to_f64(q[(row * Hq + h) * (int64_t)d + c]);
    attend(qv, pool, page_indices, kv_indptr, r, (int)((int64_t)h * Hkv / Hq), lo, hi,
           sm_scale, Hkv, P, d, NULL, 0, 0, o, lse, w, scratch);
    free(qv);
    free(scratch);
    return OR_OK;
}

/*
 * softmax_merge of n partial attentions ("Chunked prefill", #correctness): each
 * part p holds o_p (normalised over its own keys) and lse_p; the merged result
 * over the union of the keys is
 *   lse = m + ln sum_p exp(lse_p - m),  m = max_p lse_p
 *   o   = sum_p exp(lse_p - lse) o_p.
 * Parts with lse = -inf (no keys) contribute nothing.  parts_o: [n][d].
 */
void oracle_softmax_merge(const double *parts_o, const double *parts_lse, int n, int d,
                          double *o, double *lse)
{
    double m = -INFINITY;
    for (int p = 0; p < n; ++p)
        if (parts_lse[p] > m)
            m = parts_lse[p];
    for (int c = 0; c < d; ++c)
        o[c] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double z = 0.0;
    for (int p = 0; p < n; ++p)
        z += exp(parts_lse[p] - m);
    double l = m + log(z);
    for (int p = 0; p < n; ++p) {
        double a = exp(parts_lse[p] - l);
        for (int c = 0; c < d; ++c)
            o[c] += a * parts_o[(int64_t)p * d + c];
    }
    *lse = l;
}
