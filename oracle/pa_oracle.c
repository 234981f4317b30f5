/*
 * pa_oracle.c -- plain f64 CPU oracle for fused paged-attention decode v2.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / --impl reference legs of bench.py load this library.  The
 * product path (paged_attention_decode_gb300, libpa_v2.so) never links,
 * imports or calls it, and it shares no code, header or table with it.
 *
 * What it computes, and where the pages define it:
 *
 *  - Page resolution.  Issue #898 ("Fused paged-attention decode v2: CSR page
 *    table, cross-CTA split-KV, and variable-length merge kernels"), design
 *    piece 1 (CSR page table), and sparse-paged-decode.md (issue #904), first
 *    paragraph: visible token i of request r lives in physical page
 *    indices[indptr[r] + (first_page_offset[r] + i) / page_size], at entry
 *    (first_page_offset[r] + i) % page_size of that page.  Issue #898, Task 1,
 *    fixes the pool layout [num_blocks, block_size, n_kv_heads, head_dim].
 *
 *  - Geometry identity.  PR #984 ("fused paged-attention decode v2 with CSR
 *    page table and cross-CTA split-KV"), What changed 1 (CSR view builder):
 *    (pages - 1) * page_size + last_page_len - first_page_offset == seq_len,
 *    and an exactly full final page has last_page_len == page_size.
 *
 *  - Attention.  The method computes plain softmax attention over the visible
 *    tokens (cascade-attention.md, issue #903: the composed states are
 *    "exactly the attention over the whole range").  Query head h reads KV
 *    head h / (Hq / Hkv) (same page, head-stacking paragraph).  The oracle is
 *    that definition written out in f64: s_i = scale * q.K_i,
 *    out = sum_i softmax(s)_i V_i, and the log-sum-exp reported in base 2
 *    (PR #984, What changed 2: the LSE is emitted in log2 units).
 *
 *  - Partials.  PR #984, What changed 2 and 4: a chunk is a run of
 *    pages_per_chunk page slots of one request; its state is the normalized
 *    attention over the chunk's tokens plus the chunk's log2-LSE.  An empty
 *    chunk is (0, -inf).
 *
 *  - Merge.  Issue #898, design piece 3: m = max lse_i, w_i = 2^(lse_i - m),
 *    out = sum w_i v_i / sum w_i, lse_out = log2(sum w_i) + m, generalized to
 *    a variable-length group given by o_indptr (PR #984, What changed 3).  A
 *    -inf partial contributes nothing; a group with no finite partial gives
 *    zeros and -inf.
 *
 *  - Plan.  PR #984, What changed 4 (Plan): the largest pages_per_chunk whose
 *    CTA count (num_chunks * Hkv * q_groups) still reaches the target, a
 *    floor from the 65535 grid-z bound, at least one chunk per request,
 *    chunks emitted in request order.  The oracle evaluates every candidate
 *    by linear scan instead of the library's binary search.
 *
 * Element decoding of IEEE binary16 and bfloat16 is written from the formats'
 * definitions.  Everything is evaluated in double precision; no fused
 * multiply-add contraction (built with -ffp-contract=off).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORA_F32 = 0, ORA_F16 = 1, ORA_BF16 = 2 };

/* Geometry validation result codes (0 = valid). */
enum {
    ORA_GEOM_OK = 0,
    ORA_GEOM_BAD_ARGS = 1,        /* batch < 0 or page_size < 1 */
    ORA_GEOM_INDPTR0 = 2,         /* indptr[0] != 0 */
    ORA_GEOM_INDPTR_ORDER = 3,    /* indptr decreases */
    ORA_GEOM_LAST_PAGE_LEN = 4,   /* non-empty request with lpl outside [1, ps] */
    ORA_GEOM_FIRST_OFFSET = 5,    /* non-empty request with fpo outside [0, ps) */
    ORA_GEOM_SINGLE_PAGE = 6,     /* one page with fpo >= lpl (no visible token) */
    ORA_GEOM_EMPTY_REQUEST = 7,   /* zero pages but lpl or fpo non-zero */
    ORA_GEOM_PAGE_ID = 8,         /* an indices entry outside [0, num_pages) */
    ORA_GEOM_IDENTITY = 9,        /* identity disagrees with the given seq_len */
};

/* ---------------------------------------------------------------------- */
/* element decoding                                                        */
/* ---------------------------------------------------------------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  Subnormals are fraction * 2^-24. */
static double ora_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -24);
    else if (expo == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + frac), expo - 25);
    return sign ? -mag : mag;
}

/* bfloat16 is the upper half of an IEEE binary32. */
static double ora_bf16_to_double(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double ora_elem(const void *base, int dtype, int64_t idx)
{
    switch (dtype) {
    case ORA_F32: return (double)((const float *)base)[idx];
    case ORA_F16: return ora_half_to_double(((const uint16_t *)base)[idx]);
    default:      return ora_bf16_to_double(((const uint16_t *)base)[idx]);
    }
}

/* Exposed so the decoding can be pinned against library conversions. */
double ora_decode_element(const void *base, int32_t dtype, int64_t idx)
{
    return ora_elem(base, dtype, idx);
}

int32_t ora_num_threads(void)
{
#ifdef _OPENMP
    return (int32_t)omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------------- */
/* CSR geometry                                                            */
/* ---------------------------------------------------------------------- */

int64_t ora_seq_len(const int32_t *indptr, const int32_t *last_page_len,
                    const int32_t *first_page_offset, int32_t page_size, int32_t r)
{
    int64_t pages = (int64_t)indptr[r + 1] - indptr[r];
    if (pages <= 0)
        return 0;
    return (pages - 1) * page_size + last_page_len[r] - first_page_offset[r];
}

int32_t ora_validate_geometry(const int32_t *indptr, const int32_t *last_page_len,
                              const int32_t *first_page_offset, int32_t batch,
                              int32_t page_size, const int32_t *indices,
                              int64_t num_pages, const int64_t *expect_seq_len)
{
    if (batch < 0 || page_size < 1)
        return ORA_GEOM_BAD_ARGS;
    if (indptr[0] != 0)
        return ORA_GEOM_INDPTR0;
    for (int32_t r = 0; r < batch; ++r) {
        int64_t pages = (int64_t)indptr[r + 1] - indptr[r];
        if (pages < 0)
            return ORA_GEOM_INDPTR_ORDER;
        if (pages == 0) {
            if (last_page_len[r] != 0 || first_page_offset[r] != 0)
                return ORA_GEOM_EMPTY_REQUEST;
        } else {
            if (last_page_len[r] < 1 || last_page_len[r] > page_size)
                return ORA_GEOM_LAST_PAGE_LEN;
            if (first_page_offset[r] < 0 || first_page_offset[r] >= page_size)
                return ORA_GEOM_FIRST_OFFSET;
            if (pages == 1 && first_page_offset[r] >= last_page_len[r])
                return ORA_GEOM_SINGLE_PAGE;
        }
        if (expect_seq_len &&
            ora_seq_len(indptr, last_page_len, first_page_offset, page_size, r) !=
                expect_seq_len[r])
            return ORA_GEOM_IDENTITY;
    }
    if (indices) {
        for (int64_t j = 0; j < indptr[batch]; ++j)
            if (indices[j] < 0 || (int64_t)indices[j] >= num_pages)
                return ORA_GEOM_PAGE_ID;
    }
    return ORA_GEOM_OK;
}

/* Pool row (page * page_size + entry) holding visible token i of request r. */
int64_t ora_resolve_row(const int32_t *indices, const int32_t *indptr,
                        const int32_t *first_page_offset, int32_t page_size,
                        int32_t r, int64_t i)
{
    int64_t t = (int64_t)first_page_offset[r] + i;
    int64_t slot = (int64_t)indptr[r] + t / page_size;
    int64_t entry = t % page_size;
    return (int64_t)indices[slot] * page_size + entry;
}

/* ---------------------------------------------------------------------- */
/* attention over a token range of one request                              */
/* ---------------------------------------------------------------------- */

typedef struct {
    const void *k_pool, *v_pool;
    int dtype;
    const int32_t *indices, *indptr, *first_page_offset;
    int32_t page_size, num_kv_heads, head_dim;
} ora_pool;

/* Softmax attention of query q (head_dim doubles) over visible tokens
 * [i0, i1) of request r, KV head kvh.  Writes the normalized output and the
 * log-sum-exp in base 2.  An empty range gives zeros and -inf. */
static void ora_attend_range(const ora_pool *p, const double *q, double scale,
                             int32_t r, int32_t kvh, int64_t i0, int64_t i1,
                             double *out, double *lse2)
{
    const int32_t D = p->head_dim;
    for (int32_t d = 0; d < D; ++d)
        out[d] = 0.0;
    if (i1 <= i0) {
        *lse2 = -INFINITY;
        return;
    }
    int64_t n = i1 - i0;
    double *s = (double *)malloc((size_t)n * sizeof(double));
    int64_t *row = (int64_t *)malloc((size_t)n * sizeof(int64_t));
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        row[j] = ora_resolve_row(p->indices, p->indptr, p->first_page_offset,
                                 p->page_size, r, i0 + j);
        int64_t base = (row[j] * p->num_kv_heads + kvh) * D;
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d)
            dot += q[d] * ora_elem(p->k_pool, p->dtype, base + d);
        s[j] = scale * dot;
        if (s[j] > m)
            m = s[j];
    }
    double den = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double e = exp(s[j] - m);
        den += e;
        int64_t base = (row[j] * p->num_kv_heads + kvh) * D;
        for (int32_t d = 0; d < D; ++d)
            out[d] += e * ora_elem(p->v_pool, p->dtype, base + d);
    }
    for (int32_t d = 0; d < D; ++d)
        out[d] /= den;
    *lse2 = (m + log(den)) / M_LN2;
    free(s);
    free(row);
}

/* Full decode attention for every (request, query head).
 * q: [batch, num_qo_heads, head_dim] f32.  Pools: [P, page_size, Hkv, D] of
 * dtype.  out: [batch, num_qo_heads, head_dim] f64, lse2: [batch, Hq] f64. */
void ora_attention(const float *q, const void *k_pool, const void *v_pool, int32_t dtype,
                   const int32_t *indices, const int32_t *indptr,
                   const int32_t *last_page_len, const int32_t *first_page_offset,
                   int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads,
                   int32_t head_dim, int32_t page_size, double scale, double *out,
                   double *lse2)
{
    ora_pool p = {k_pool, v_pool, dtype, indices, indptr, first_page_offset,
                  page_size, num_kv_heads, head_dim};
    const int32_t group = num_qo_heads / num_kv_heads;
    const int64_t pairs = (int64_t)batch * num_qo_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t rh = 0; rh < pairs; ++rh) {
        int32_t r = (int32_t)(rh / num_qo_heads), h = (int32_t)(rh % num_qo_heads);
        double *qd = (double *)malloc((size_t)head_dim * sizeof(double));
        for (int32_t d = 0; d < head_dim; ++d)
            qd[d] = (double)q[rh * head_dim + d];
        int64_t L = ora_seq_len(indptr, last_page_len, first_page_offset, page_size, r);
        ora_attend_range(&p, qd, scale, r, h / group, 0, L, out + rh * head_dim,
                         lse2 + rh);
        free(qd);
    }
}

/* Per-chunk partial states for a given chunking: chunk c is the
 * kv_tile_indices[c]-th run of pages_per_chunk page slots of request
 * request_indices[c].  out: [num_chunks, Hq, D] f64, lse2: [num_chunks, Hq]. */
void ora_partials(const float *q, const void *k_pool, const void *v_pool, int32_t dtype,
                  const int32_t *indices, const int32_t *indptr,
                  const int32_t *last_page_len, const int32_t *first_page_offset,
                  int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                  int32_t page_size, int32_t pages_per_chunk,
                  const int32_t *request_indices, const int32_t *kv_tile_indices,
                  int64_t num_chunks, double scale, double *out, double *lse2)
{
    ora_pool p = {k_pool, v_pool, dtype, indices, indptr, first_page_offset,
                  page_size, num_kv_heads, head_dim};
    const int32_t group = num_qo_heads / num_kv_heads;
    const int64_t pairs = num_chunks * num_qo_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t ch = 0; ch < pairs; ++ch) {
        int64_t c = ch / num_qo_heads;
        int32_t h = (int32_t)(ch % num_qo_heads);
        int32_t r = request_indices[c];
        int64_t k = kv_tile_indices[c];
        int64_t L = ora_seq_len(indptr, last_page_len, first_page_offset, page_size, r);
        /* token index of slot s, entry e is s * page_size + e - fpo */
        int64_t i0 = k * pages_per_chunk * page_size - first_page_offset[r];
        int64_t i1 = (k + 1) * pages_per_chunk * page_size - first_page_offset[r];
        if (i0 < 0) i0 = 0;
        if (i1 > L) i1 = L;
        double *qd = (double *)malloc((size_t)head_dim * sizeof(double));
        for (int32_t d = 0; d < head_dim; ++d)
            qd[d] = (double)q[((int64_t)r * num_qo_heads + h) * head_dim + d];
        ora_attend_range(&p, qd, scale, r, h / group, i0, i1, out + ch * head_dim,
                         lse2 + ch);
        free(qd);
    }
}

/* ---------------------------------------------------------------------- */
/* merge of attention states                                                */
/* ---------------------------------------------------------------------- */

/* v_in [N, H, D] normalized partials, lse_in [N, H] base-2 LSEs, o_indptr
 * [M + 1] groups contiguous rows.  out [M, H, D], lse_out [M, H]. */
void ora_merge(const double *v_in, const double *lse_in, const int32_t *o_indptr,
               int32_t num_rows_out, int32_t num_heads, int32_t head_dim, double *out,
               double *lse_out)
{
    for (int32_t r = 0; r < num_rows_out; ++r) {
        for (int32_t h = 0; h < num_heads; ++h) {
            double *o = out + ((int64_t)r * num_heads + h) * head_dim;
            double m = -INFINITY;
            for (int32_t i = o_indptr[r]; i < o_indptr[r + 1]; ++i) {
                double l = lse_in[(int64_t)i * num_heads + h];
                if (l > m)
                    m = l;
            }
            for (int32_t d = 0; d < head_dim; ++d)
                o[d] = 0.0;
            if (m == -INFINITY) {
                lse_out[(int64_t)r * num_heads + h] = -INFINITY;
                continue;
            }
            double wsum = 0.0;
            for (int32_t i = o_indptr[r]; i < o_indptr[r + 1]; ++i) {
                double l = lse_in[(int64_t)i * num_heads + h];
                double w = (l == -INFINITY) ? 0.0 : exp2(l - m);
                wsum += w;
                const double *v = v_in + ((int64_t)i * num_heads + h) * head_dim;
                for (int32_t d = 0; d < head_dim; ++d)
                    o[d] += w * v[d];
            }
            for (int32_t d = 0; d < head_dim; ++d)
                o[d] /= wsum;
            lse_out[(int64_t)r * num_heads + h] = log2(wsum) + m;
        }
    }
}

/* ---------------------------------------------------------------------- */
/* plan: chunk-size choice by linear scan                                   */
/* ---------------------------------------------------------------------- */

static int64_t ora_num_chunks(const int32_t *indptr, int32_t batch, int64_t ppc)
{
    int64_t n = 0;
    for (int32_t r = 0; r < batch; ++r) {
        int64_t pages = (int64_t)indptr[r + 1] - indptr[r];
        int64_t c = 0;
        /* ceil(pages / ppc) written as repeated subtraction-free division */
        if (pages > 0)
            c = pages / ppc + (pages % ppc != 0);
        n += c > 1 ? c : 1;
    }
    return n;
}

/* Returns 0 on success, 1 if no chunk size fits max_chunks, 2 if the
 * override does not fit, 3 if cap is too small (needed count in *n_out).
 * On success writes pages_per_chunk, the search bounds, the chunk count and
 * the request_indices / kv_tile_indices / o_indptr arrays. */
int32_t ora_plan(const int32_t *indptr, int32_t batch, int32_t num_kv_heads,
                 int32_t q_groups, int64_t target_ctas, int32_t ppc_override,
                 int64_t max_chunks, int32_t *ppc_out, int32_t *lo_out, int32_t *hi_out,
                 int64_t *n_out, int32_t *request_indices, int32_t *kv_tile_indices,
                 int64_t cap, int32_t *o_indptr)
{
    int64_t hi = 1;
    for (int32_t r = 0; r < batch; ++r) {
        int64_t pages = (int64_t)indptr[r + 1] - indptr[r];
        if (pages > hi)
            hi = pages;
    }
    int64_t lo = -1;
    for (int64_t p = 1; p <= hi; ++p) {
        if (ora_num_chunks(indptr, batch, p) <= max_chunks) {
            lo = p;
            break;
        }
    }
    if (lo < 0)
        return 1;
    int64_t ppc;
    if (ppc_override > 0) {
        if (ora_num_chunks(indptr, batch, ppc_override) > max_chunks)
            return 2;
        ppc = ppc_override;
    } else {
        ppc = lo;
        for (int64_t p = lo; p <= hi; ++p)
            if (ora_num_chunks(indptr, batch, p) * num_kv_heads * q_groups >= target_ctas)
                ppc = p;
    }
    int64_t n = ora_num_chunks(indptr, batch, ppc);
    *ppc_out = (int32_t)ppc;
    *lo_out = (int32_t)lo;
    *hi_out = (int32_t)hi;
    *n_out = n;
    if (n > cap)
        return 3;
    int64_t c = 0;
    o_indptr[0] = 0;
    for (int32_t r = 0; r < batch; ++r) {
        int64_t pages = (int64_t)indptr[r + 1] - indptr[r];
        int64_t nr = pages > 0 ? pages / ppc + (pages % ppc != 0) : 1;
        for (int64_t k = 0; k < nr; ++k) {
            request_indices[c] = r;
            kv_tile_indices[c] = (int32_t)k;
            ++c;
        }
        o_indptr[r + 1] = (int32_t)c;
    }
    return 0;
}
