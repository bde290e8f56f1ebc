/*
 * Paged-attention oracle: a plain, slow fp64 CPU restatement of what attention
 * over a paged K/V cache computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links, loads or calls this
 * file; only the test suite, the smoke check and the benchmark's CPU-baseline
 * arm use it.  It shares no code with the CUDA path.
 *
 * Sources (page titles and sections):
 *   [P1] rocMLIR PR #2222 "Paged Attention: rocmlir-gen changes", Key Changes 1
 *        (view [batch, numPages, pageSize] -> [G, seqK, headDim]) and 3 (the
 *        CPU validator works on logically ordered K/V, not on pages).
 *   [P3] rocm-libraries PR #14349, Motivation and Technical Details: page ids
 *        come from a per-sequence block table; the in-page offset has a
 *        kv-head term; page size is counted in tokens; GQA shapes 32/8, 64/4.
 *   [P4] rocMLIR PR #2371 "Fix split-kv attention masking...", Technical
 *        Details: ceil-divided split partition with the end clamped so trailing
 *        splits are empty; an empty or fully masked partition contributes
 *        zero; a 0/0 row stores 0; the split combine is a reduce-max, exp,
 *        weighted sum and normalisation; causal reach is per query row and
 *        includes the prefix offset.
 *
 * Readings where the pages leave a step open (each is also listed in the
 * design notes):
 *   - the split unit is a page of the sequence's own length L_b;
 *   - q_offset[b] defaults to L_b - Sq (queries are the last Sq tokens);
 *   - key j is valid for query row i iff j < L_b and, when causal,
 *     j <= q_offset[b] + i;
 *   - GQA: query head h reads kv head h / (Hq / Hkv);
 *   - lse is the natural log of the sum of exp(scaled score);
 *   - a split's partial output is normalised by its own sum; a split with no
 *     valid key yields output 0 and lse -inf;
 *   - quantized pools (the pages' sweeps include i8 attention: rocMLIR PR #2222,
 *     reviewed files; rocMLIR PR #2371, Motivation) are read as FP8 E4M3 or as
 *     two's-complement int8 elements with one float scale per (page, kv head):
 *     value = element x scale.
 *
 * Everything is evaluated from the definition: scores in double, the maximum
 * over all valid keys, then exp, sum and weighted sum.  No online rescaling,
 * no blocking.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2, ORACLE_FP8E4M3 = 3, ORACLE_INT8 = 4 };
enum { ORACLE_OK = 0, ORACLE_EINVAL = -1, ORACLE_EBOUNDS = -5, ORACLE_ENOMEM = -6 };

/* Shape of one problem.  Layouts (all dense, row-major):
 *   q            [B, Sq, Hq, D]
 *   k/v cache    [num_pages, page_size, Hkv, D]
 *   block_table  [B, bt_stride] int32
 *   seq_lens     [B] int32, q_offset [B] int32 (optional) */
typedef struct {
    int32_t B, Sq, Hq, Hkv, D, page_size, bt_stride, dtype;
    int64_t num_pages;
} oracle_dims;

/* ---------------------------------------------------------------- widening */

/* IEEE binary16 -> double, exactly, from the format's definition. */
static double half_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);
    return sign ? -v : v;
}

/* bfloat16 -> double: the 16 bits are the top half of a binary32. */
static double bf16_bits_to_double(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* FP8 E4M3 (OCP "fn" variant: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent
 * 1111 with mantissa 111 is NaN; no infinities) -> double, exactly, from the format's definition. */
static double e4m3_bits_to_double(uint8_t h)
{
    int sign = (h >> 7) & 1;
    int e = (h >> 3) & 0xF;
    int m = h & 7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);          /* m/8 * 2^(1-7) */
    else
        v = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* int8 (two's complement: bit 7 weighs -128) -> double. */
static double int8_bits_to_double(uint8_t h)
{
    return (double)(h & 0x7F) - ((h & 0x80) ? 128.0 : 0.0);
}

static double widen(const void *base, int dtype, int64_t idx)
{
    if (dtype == ORACLE_INT8)
        return int8_bits_to_double(((const uint8_t *)base)[idx]);
    if (dtype == ORACLE_FP8E4M3)
        return e4m3_bits_to_double(((const uint8_t *)base)[idx]);
    if (dtype == ORACLE_F32)
        return (double)((const float *)base)[idx];
    if (dtype == ORACLE_BF16)
        return bf16_bits_to_double(((const uint16_t *)base)[idx]);
    return half_bits_to_double(((const uint16_t *)base)[idx]);
}

static int dims_ok(const oracle_dims *d)
{
    if (!d || d->B < 0 || d->Sq < 0 || d->Hq <= 0 || d->Hkv <= 0 || d->D <= 0 || d->page_size <= 0)
        return 0;
    if (d->Hq % d->Hkv != 0)
        return 0;
    if (d->dtype != ORACLE_F32 && d->dtype != ORACLE_F16 && d->dtype != ORACLE_BF16)
        return 0;
    return d->num_pages >= 0 && d->bt_stride >= 0;
}

/* The K and V pools as stored: element type, and for quantized pools one float scale per
 * (page, kv head), [num_pages, Hkv]; a stored element times its page's scale is the value. */
typedef struct {
    const void *k_cache, *v_cache;
    int kv_dtype;
    const float *k_scale, *v_scale;  /* NULL: no scaling */
} oracle_kv;

/* ---------------------------------------------------------------- split plan */

/* [P4] split-KV iteration math: blocks per split is the ceiling of
 * blocks / split_kv; a split's start and end are clamped to the block count, so
 * trailing splits are empty.  Here a block is a page of sequence b.
 * plan is [B, split_kv, 2] = {first page, one past the last page}. */
int oracle_plan(const int32_t *seq_lens, int32_t B, int32_t page_size, int32_t split_kv, int32_t *plan)
{
    if (B < 0 || page_size <= 0 || split_kv <= 0)
        return ORACLE_EINVAL;
    for (int32_t b = 0; b < B; ++b) {
        int64_t L = seq_lens[b] > 0 ? seq_lens[b] : 0;
        int64_t nblk = (L + page_size - 1) / page_size;
        int64_t per = (nblk + split_kv - 1) / split_kv;
        for (int32_t s = 0; s < split_kv; ++s) {
            int64_t start = (int64_t)s * per;
            int64_t end = (int64_t)(s + 1) * per;
            if (start > nblk) start = nblk;
            if (end > nblk) end = nblk;
            plan[((int64_t)b * split_kv + s) * 2 + 0] = (int32_t)start;
            plan[((int64_t)b * split_kv + s) * 2 + 1] = (int32_t)end;
        }
    }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------- gather */

/* [P1][P3] element (token j, kv head kvh, dim e) of sequence b: the page is
 * block_table[b][j / page_size]; inside the page the token sits at row
 * j % page_size and the kv head adds kvh * D.  Returns the flat index or -1 if
 * the page id is not a page of the pool. */
static int32_t table_page(const oracle_dims *d, const int32_t *block_table, int32_t b, int64_t j)
{
    return block_table[(int64_t)b * d->bt_stride + j / d->page_size];
}

static int64_t logical_index(const oracle_dims *d, const int32_t *block_table, int32_t b, int64_t j,
                             int32_t kvh, int32_t e)
{
    int32_t page = table_page(d, block_table, b, j);
    if (page < 0 || (int64_t)page >= d->num_pages)
        return -1;
    int64_t tok = (int64_t)page * d->page_size + j % d->page_size;
    return (tok * d->Hkv + kvh) * d->D + e;
}

/* Logically ordered K (or V) of sequence b: out[L_b, Hkv, D] in double. */
int oracle_gather(const void *cache, const int32_t *block_table, const int32_t *seq_lens,
                  const oracle_dims *d, int32_t b, double *out)
{
    if (!dims_ok(d) || b < 0 || b >= d->B)
        return ORACLE_EINVAL;
    int64_t L = seq_lens[b] > 0 ? seq_lens[b] : 0;
    if ((L + d->page_size - 1) / d->page_size > d->bt_stride)
        return ORACLE_EINVAL;
    for (int64_t j = 0; j < L; ++j)
        for (int32_t kvh = 0; kvh < d->Hkv; ++kvh)
            for (int32_t e = 0; e < d->D; ++e) {
                int64_t idx = logical_index(d, block_table, b, j, kvh, e);
                if (idx < 0)
                    return ORACLE_EBOUNDS;
                out[(j * d->Hkv + kvh) * d->D + e] = widen(cache, d->dtype, idx);
            }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------- masking */

/* Number of keys query row i of sequence b may see: keys j < L_b and, when
 * causal, j <= q_offset[b] + i ([P4] per-row causal reach with the prefix
 * offset).  Valid keys always form the prefix [0, limit). */
static int64_t key_limit(const oracle_dims *d, const int32_t *seq_lens, const int32_t *q_offset,
                         int32_t causal, int32_t b, int32_t i)
{
    int64_t L = seq_lens[b] > 0 ? seq_lens[b] : 0;
    if (!causal)
        return L;
    int64_t qoff = q_offset ? (int64_t)q_offset[b] : L - d->Sq;
    int64_t reach = qoff + i + 1;
    if (reach < 0) reach = 0;
    return reach < L ? reach : L;
}

int64_t oracle_key_limit(const int32_t *seq_lens, const int32_t *q_offset, int32_t causal,
                         const oracle_dims *d, int32_t b, int32_t i)
{
    return key_limit(d, seq_lens, q_offset, causal, b, i);
}

/* ---------------------------------------------------------------- softmax */

/* Value of the element at flat index idx (token j, kv head kvh of sequence b) in pool k
 * (which = 0) or v (1): the stored element, times its (page, kv head) scale for quantized pools. */
static double kv_value(const oracle_dims *d, const oracle_kv *kv, int which, const int32_t *block_table, int32_t b,
                       int64_t j, int32_t kvh, int64_t idx)
{
    const void *cache = which ? kv->v_cache : kv->k_cache;
    double x = widen(cache, kv->kv_dtype, idx);
    const float *sc = which ? kv->v_scale : kv->k_scale;
    if (sc)
        x *= (double)sc[(int64_t)table_page(d, block_table, b, j) * d->Hkv + kvh];
    return x;
}

/* softmax(scale * q.k_j) . v_j over the keys j in [lo, hi), from the definition.
 * No keys: out = 0, lse = -inf.  scratch has room for hi - lo doubles. */
static int attend_keys(const oracle_dims *d, const double *qrow, const oracle_kv *kv,
                       const int32_t *block_table, int32_t b, int32_t kvh, int64_t lo, int64_t hi,
                       double scale, double *scratch, double *out, double *lse)
{
    const int32_t D = d->D;
    for (int32_t e = 0; e < D; ++e)
        out[e] = 0.0;
    if (hi <= lo) {
        *lse = -INFINITY;
        return ORACLE_OK;
    }
    double m = -INFINITY;
    for (int64_t j = lo; j < hi; ++j) {
        double s = 0.0;
        for (int32_t e = 0; e < D; ++e) {
            int64_t idx = logical_index(d, block_table, b, j, kvh, e);
            if (idx < 0)
                return ORACLE_EBOUNDS;
            s += qrow[e] * kv_value(d, kv, 0, block_table, b, j, kvh, idx);
        }
        s *= scale;
        scratch[j - lo] = s;
        if (s > m)
            m = s;
    }
    double l = 0.0;
    for (int64_t j = lo; j < hi; ++j) {
        double p = exp(scratch[j - lo] - m);
        l += p;
        for (int32_t e = 0; e < D; ++e) {
            int64_t idx = logical_index(d, block_table, b, j, kvh, e);
            out[e] += p * kv_value(d, kv, 1, block_table, b, j, kvh, idx);
        }
    }
    for (int32_t e = 0; e < D; ++e)
        out[e] /= l;
    *lse = m + log(l);
    return ORACLE_OK;
}

/* ---------------------------------------------------------------- combine */

/* [P4] split combine: M = max_s lse_s; w_s = exp(lse_s - M); out = sum w_s O_s /
 * sum w_s; lse = M + log(sum w_s).  All splits empty (M = -inf): out 0, lse -inf.
 * part_out [S, D] and part_lse [S] belong to one row. */
static void combine_row(const double *part_out, const double *part_lse, int32_t S, int32_t D,
                        double *out, double *lse)
{
    double M = -INFINITY;
    for (int32_t s = 0; s < S; ++s)
        if (part_lse[s] > M)
            M = part_lse[s];
    for (int32_t e = 0; e < D; ++e)
        out[e] = 0.0;
    if (M == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double wsum = 0.0;
    for (int32_t s = 0; s < S; ++s) {
        double w = exp(part_lse[s] - M);
        wsum += w;
        for (int32_t e = 0; e < D; ++e)
            out[e] += w * part_out[(int64_t)s * D + e];
    }
    for (int32_t e = 0; e < D; ++e)
        out[e] /= wsum;
    *lse = M + log(wsum);
}

/* Combine many rows: part_out [n, S, D], part_lse [n, S] -> out [n, D], lse [n]. */
void oracle_combine(const double *part_out, const double *part_lse, int64_t n, int32_t S, int32_t D,
                    double *out, double *lse)
{
    for (int64_t r = 0; r < n; ++r)
        combine_row(part_out + r * S * D, part_lse + r * S, S, D, out + r * D, lse + r);
}

/* ---------------------------------------------------------------- rows */

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Attention for the query rows (row_b[r], row_i[r], row_h[r]).
 *   out/lse            unsplit result over every valid key      [n, D] / [n]
 *   part_out/part_lse  per-split results of the page plan       [n, S, D] / [n, S]
 *   comb_out/comb_lse  those partials combined                  [n, D] / [n]
 * Any of the split outputs may be NULL (then split_kv is only used for them).
 * n_threads <= 0 uses the OpenMP default.  Returns ORACLE_EBOUNDS if a page id
 * inside a sequence's first ceil(L_b / page_size) table slots is not a pool page. */
static int rows_impl(const void *q, const oracle_kv *kv, const int32_t *block_table,
                     const int32_t *seq_lens, const int32_t *q_offset, int32_t causal, const oracle_dims *d,
                     double scale, int32_t split_kv, const int32_t *row_b, const int32_t *row_i,
                     const int32_t *row_h, int64_t n_rows, int32_t n_threads, double *out, double *lse,
                     double *part_out, double *part_lse, double *comb_out, double *comb_lse)
{
    if (!dims_ok(d) || split_kv <= 0 || n_rows < 0)
        return ORACLE_EINVAL;
    const int32_t D = d->D, S = split_kv, G = d->Hq / d->Hkv;
    int64_t maxL = 0;
    for (int32_t b = 0; b < d->B; ++b) {
        int64_t L = seq_lens[b] > 0 ? seq_lens[b] : 0;
        if ((L + d->page_size - 1) / d->page_size > d->bt_stride)
            return ORACLE_EINVAL;
        if (L > maxL) maxL = L;
    }
    for (int64_t r = 0; r < n_rows; ++r)
        if (row_b[r] < 0 || row_b[r] >= d->B || row_i[r] < 0 || row_i[r] >= d->Sq || row_h[r] < 0 ||
            row_h[r] >= d->Hq)
            return ORACLE_EINVAL;
    int32_t *plan = (int32_t *)malloc(sizeof(int32_t) * 2 * (size_t)(d->B > 0 ? d->B : 1) * S);
    if (!plan)
        return ORACLE_ENOMEM;
    oracle_plan(seq_lens, d->B, d->page_size, S, plan);
    int status = ORACLE_OK;
#ifdef _OPENMP
    if (n_threads > 0)
        omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel
    {
        double *qrow = (double *)malloc(sizeof(double) * D);
        double *scratch = (double *)malloc(sizeof(double) * (size_t)(maxL > 0 ? maxL : 1));
        double *pout = (double *)malloc(sizeof(double) * (size_t)S * D);
        double *plse = (double *)malloc(sizeof(double) * (size_t)S);
        if (!qrow || !scratch || !pout || !plse) {
#pragma omp critical
            status = ORACLE_ENOMEM;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < n_rows; ++r) {
                const int32_t b = row_b[r], i = row_i[r], h = row_h[r];
                const int32_t kvh = h / G;
                const int64_t qbase = (((int64_t)b * d->Sq + i) * d->Hq + h) * D;
                for (int32_t e = 0; e < D; ++e)
                    qrow[e] = widen(q, d->dtype, qbase + e);
                const int64_t lim = key_limit(d, seq_lens, q_offset, causal, b, i);
                int st = ORACLE_OK;
                double tlse;
                if (out && lse) {
                    st = attend_keys(d, qrow, kv, block_table, b, kvh, 0, lim, scale, scratch, out + r * D, lse + r);
                }
                if (st == ORACLE_OK && (part_out || comb_out)) {
                    const int64_t L = seq_lens[b] > 0 ? seq_lens[b] : 0;
                    for (int32_t s = 0; s < S && st == ORACLE_OK; ++s) {
                        int64_t lo = (int64_t)plan[((int64_t)b * S + s) * 2 + 0] * d->page_size;
                        int64_t hi = (int64_t)plan[((int64_t)b * S + s) * 2 + 1] * d->page_size;
                        if (hi > L) hi = L;
                        if (hi > lim) hi = lim;   /* causal reach inside the split */
                        if (lo > hi) lo = hi;
                        st = attend_keys(d, qrow, kv, block_table, b, kvh, lo, hi, scale, scratch,
                                         pout + (int64_t)s * D, &tlse);
                        plse[s] = tlse;
                    }
                    if (st == ORACLE_OK) {
                        if (part_out)
                            memcpy(part_out + r * S * D, pout, sizeof(double) * (size_t)S * D);
                        if (part_lse)
                            memcpy(part_lse + r * S, plse, sizeof(double) * (size_t)S);
                        if (comb_out && comb_lse)
                            combine_row(pout, plse, S, D, comb_out + r * D, comb_lse + r);
                    }
                }
                if (st != ORACLE_OK) {
#pragma omp critical
                    status = st;
                }
            }
        }
        free(qrow);
        free(scratch);
        free(pout);
        free(plse);
    }
    free(plan);
    return status;
}

/* Attention for the chosen rows with K/V pools of element type dtype (see oracle_rows). */
int oracle_rows(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
                const int32_t *seq_lens, const int32_t *q_offset, int32_t causal, const oracle_dims *d,
                double scale, int32_t split_kv, const int32_t *row_b, const int32_t *row_i,
                const int32_t *row_h, int64_t n_rows, int32_t n_threads, double *out, double *lse,
                double *part_out, double *part_lse, double *comb_out, double *comb_lse)
{
    if (!dims_ok(d))
        return ORACLE_EINVAL;
    const oracle_kv kv = {k_cache, v_cache, d->dtype, NULL, NULL};
    return rows_impl(q, &kv, block_table, seq_lens, q_offset, causal, d, scale, split_kv, row_b, row_i, row_h,
                     n_rows, n_threads, out, lse, part_out, part_lse, comb_out, comb_lse);
}

/* The same with quantized K/V pools: elements of kv_dtype (ORACLE_FP8E4M3 or ORACLE_INT8) times the float scale
 * of their (page, kv head), k_scale / v_scale [num_pages, Hkv]; q and the results as in oracle_rows. */
int oracle_rows_kvq(const void *q, const void *k_cache, const void *v_cache, int32_t kv_dtype,
                    const float *k_scale, const float *v_scale, const int32_t *block_table,
                    const int32_t *seq_lens, const int32_t *q_offset, int32_t causal, const oracle_dims *d,
                    double scale, int32_t split_kv, const int32_t *row_b, const int32_t *row_i,
                    const int32_t *row_h, int64_t n_rows, int32_t n_threads, double *out, double *lse,
                    double *part_out, double *part_lse, double *comb_out, double *comb_lse)
{
    if (!dims_ok(d) || (kv_dtype != ORACLE_FP8E4M3 && kv_dtype != ORACLE_INT8) || !k_scale || !v_scale)
        return ORACLE_EINVAL;
    const oracle_kv kv = {k_cache, v_cache, kv_dtype, k_scale, v_scale};
    return rows_impl(q, &kv, block_table, seq_lens, q_offset, causal, d, scale, split_kv, row_b, row_i, row_h,
                     n_rows, n_threads, out, lse, part_out, part_lse, comb_out, comb_lse);
}

/* Dequantized logical gather of one quantized pool: out[L_b, Hkv, D] (see oracle_gather). */
int oracle_gather_kvq(const void *cache, int32_t kv_dtype, const float *scales, const int32_t *block_table,
                      const int32_t *seq_lens, const oracle_dims *d, int32_t b, double *out)
{
    if (!dims_ok(d) || b < 0 || b >= d->B || (kv_dtype != ORACLE_FP8E4M3 && kv_dtype != ORACLE_INT8) || !scales)
        return ORACLE_EINVAL;
    const oracle_kv kv = {cache, cache, kv_dtype, scales, scales};
    int64_t L = seq_lens[b] > 0 ? seq_lens[b] : 0;
    if ((L + d->page_size - 1) / d->page_size > d->bt_stride)
        return ORACLE_EINVAL;
    for (int64_t j = 0; j < L; ++j)
        for (int32_t kvh = 0; kvh < d->Hkv; ++kvh)
            for (int32_t e = 0; e < d->D; ++e) {
                int64_t idx = logical_index(d, block_table, b, j, kvh, e);
                if (idx < 0)
                    return ORACLE_EBOUNDS;
                out[(j * d->Hkv + kvh) * d->D + e] = kv_value(d, &kv, 0, block_table, b, j, kvh, idx);
            }
    return ORACLE_OK;
}
