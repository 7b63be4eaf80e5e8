/*
 * Oracle for the DLRM sparse hot path.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the test suite, the
 * smoke check in __graft_entry__ and the CPU-baseline leg of bench.py may
 * load or call this code.  It shares nothing with the CUDA library: no
 * headers, no helpers, no constants.
 *
 * Every function below is the plain definition of one step of the path,
 * written as simple loops and computed in fp64.  Next to every floating
 * point result it also returns a "magnitude": the same computation carried
 * out on absolute values (for a sum of products, the sum of the absolute
 * products).  The magnitude bounds the rounding error of any summation order,
 * so a GPU value x passes when |x - value| <= rel * magnitude.  Magnitudes of
 * inputs may be passed in (to chain stages); a NULL magnitude means |x|.
 *
 * Sources (web pages describing the Deep Learning Recommendation Model):
 *  - "Notes/DLRM" (vault-aram.pages.dev), section 2 "The Architecture": one
 *    embedding table per categorical feature; the lookup turns an ID into a
 *    learned vector; the bottom-MLP output e0 has the embedding dimension.
 *  - same page, section 3 "The Pairwise Interaction Layer": a dot product
 *    e_i^T e_j for each unordered pair, self pairs optional, the resulting
 *    vector concatenated with e0.
 *  - same page, section 9 "Weaknesses": multi-valued features must be
 *    aggregated before they are passed in (here: sum pooling over a bag).
 *  - same page, section 5 "Training": the tables are trained by an optimizer
 *    (here: row-wise SGD on the rows a batch touched).
 *  - "Terabyte Embedding Tables ... Force Meta's DLRM to Split Training"
 *    (factlen.com), section "The memory wall of sparse features": the model
 *    adjusts the vectors as it trains.
 * Where the pages are silent (pooling operator, CSR layout, pair order,
 * which side of the concatenation e0 sits on, the optimizer's exact form),
 * the readings used are stated at each function.
 *
 * Build: gcc -O2 -ffp-contract=off -shared -fPIC (no fused multiply-add, so
 * results are identical on x86-64 and AArch64 hosts).  The same source built
 * with -fopenmp spreads the outer loops (tables and samples, samples, unique
 * keys) over the host's cores; every output element is still computed by one
 * thread in the order written here, so both builds give identical results.
 * The parallel build exists only to time the oracle on all cores.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2, ORACLE_INT4 = 3 };
enum {
    ORACLE_OK = 0,
    ORACLE_INVALID_ARG = -1,
    ORACLE_INDEX_OOB = -4,
    ORACLE_BAD_OFFSETS = -5,
    ORACLE_NO_MEMORY = -8
};

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_binary16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24); /* subnormal: frac * 2^-14 * 2^-10 */
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), expo - 25); /* (1 + frac/2^10) * 2^(expo-15) */
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
static double decode_bfloat16(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * Row-wise 4-bit tables.  The factlen.com page ("...Force Meta's DLRM to Split
 * Training", section "Scaling limits and the reality of production") reports
 * 4-bit integer quantization of the vectors without a format; the reading here is the
 * common row-wise affine codec: each row stores d 4-bit codes q (element 2j
 * in the low nibble of byte j, element 2j+1 in the high nibble), then its
 * fp32 scale s and fp32 bias b; the row is padded to a multiple of 16 bytes.
 * An element's value is b + s q.
 */
static int64_t int4_row_bytes(int d)
{
    return ((int64_t)d / 2 + 8 + 15) / 16 * 16;
}

static void int4_params(const void *table, int d, int64_t r, float *scale, float *bias)
{
    const uint8_t *row = (const uint8_t *)table + r * int4_row_bytes(d);
    memcpy(scale, row + d / 2, 4);
    memcpy(bias, row + d / 2 + 4, 4);
}

static int int4_code(const void *table, int d, int64_t r, int e)
{
    const uint8_t *row = (const uint8_t *)table + r * int4_row_bytes(d);
    return (row[e / 2] >> (4 * (e & 1))) & 15;
}

/* Element pos = r * d + e of a table; int4 tables need d to find the row. */
static double table_element(const void *table, int dtype, int d, int64_t pos)
{
    if (dtype == ORACLE_F32)
        return (double)((const float *)table)[pos];
    if (dtype == ORACLE_F16)
        return decode_binary16(((const uint16_t *)table)[pos]);
    if (dtype == ORACLE_INT4) {
        float s, b;
        int64_t r = pos / d;
        int e = (int)(pos % d);
        int4_params(table, d, r, &s, &b);
        return (double)b + (double)s * int4_code(table, d, r, e);
    }
    return decode_bfloat16(((const uint16_t *)table)[pos]);
}

/* The element's magnitude: |value|, or |b| + |s q| for a decoded int4 code. */
static double table_element_mag(const void *table, int dtype, int d, int64_t pos)
{
    if (dtype == ORACLE_INT4) {
        float s, b;
        int64_t r = pos / d;
        int4_params(table, d, r, &s, &b);
        return fabs((double)b) + fabs((double)s * int4_code(table, d, r, (int)(pos % d)));
    }
    return fabs(table_element(table, dtype, d, pos));
}

static double mag_or_abs(const double *mag, const double *val, int64_t i)
{
    return mag ? mag[i] : fabs(val[i]);
}

/* Decodes n elements of a table in its storage type to fp64 (test helper). */
int oracle_decode(int dtype, const void *src, int64_t n, double *dst)
{
    if (dtype < ORACLE_F32 || dtype > ORACLE_BF16 || n < 0)
        return ORACLE_INVALID_ARG;
    for (int64_t i = 0; i < n; i++)
        dst[i] = table_element(src, dtype, 1, i);
    return ORACLE_OK;
}

/*
 * Offsets are table-major CSR: bag (t, b) holds the lookups
 * indices[offsets[t*B + b] .. offsets[t*B + b + 1]).  (Reading: the pages give
 * no layout.)  Checks offsets[0] == 0, offsets[T*B] == nnz and monotonicity.
 */
static int check_offsets(int T, int64_t B, const int64_t *offsets, int64_t nnz)
{
    if (offsets[0] != 0 || offsets[(int64_t)T * B] != nnz)
        return ORACLE_BAD_OFFSETS;
    for (int64_t i = 0; i < (int64_t)T * B; i++)
        if (offsets[i + 1] < offsets[i])
            return ORACLE_BAD_OFFSETS;
    return ORACLE_OK;
}

/*
 * Embedding-bag forward: pooled[b][t][:] = sum over the lookups k of bag
 * (t, b) of row indices[k] of table t.  Sum pooling is the reading of
 * "aggregated" in section 9 of the DLRM notes; an empty bag pools to zero.
 * Output layout [B][T][d] (fp64) with its magnitude.
 */
int oracle_emb_bag_fwd(int T, int d, int dtype, const void *const *tables, const int64_t *rows,
                       int64_t B, const int64_t *offsets, const int64_t *indices, int64_t nnz,
                       double *pooled, double *pooled_mag)
{
    if (T <= 0 || d <= 0 || B < 0 || dtype < ORACLE_F32 || dtype > ORACLE_INT4 ||
        (dtype == ORACLE_INT4 && d % 2 != 0))
        return ORACLE_INVALID_ARG;
    int st = check_offsets(T, B, offsets, nnz);
    if (st != ORACLE_OK)
        return st;
    for (int t = 0; t < T; t++)
        for (int64_t k = offsets[(int64_t)t * B]; k < offsets[(int64_t)(t + 1) * B]; k++)
            if (indices[k] < 0 || indices[k] >= rows[t])
                return ORACLE_INDEX_OOB;
#pragma omp parallel for collapse(2) schedule(dynamic, 64)
    for (int t = 0; t < T; t++) {
        for (int64_t b = 0; b < B; b++) {
            double *out = pooled + (b * T + t) * (int64_t)d;
            double *mag = pooled_mag + (b * T + t) * (int64_t)d;
            for (int e = 0; e < d; e++) {
                out[e] = 0.0;
                mag[e] = 0.0;
            }
            for (int64_t k = offsets[(int64_t)t * B + b]; k < offsets[(int64_t)t * B + b + 1]; k++) {
                int64_t r = indices[k];
                for (int e = 0; e < d; e++) {
                    out[e] += table_element(tables[t], dtype, d, r * d + e);
                    mag[e] += table_element_mag(tables[t], dtype, d, r * d + e);
                }
            }
        }
    }
    return ORACLE_OK;
}

/*
 * Number of interaction terms over F = N + 1 vectors (e0 and the N pooled
 * embeddings): F(F-1)/2 strict pairs, F(F+1)/2 with self pairs.
 */
int64_t oracle_num_pairs(int N, int include_self)
{
    int64_t F = (int64_t)N + 1;
    return (include_self & 1) ? F * (F + 1) / 2 : F * (F - 1) / 2;
}

/*
 * Width of an interaction output row.  mode bit 0: self pairs; bit 1: the
 * original embeddings are concatenated alongside (section 3 of the DLRM notes
 * names this variant: "some include the original embeddings concatenated
 * alongside the interaction vector"; read here as [e0 | e_1 .. e_N | pairs]).
 */
static int64_t interact_width(int N, int d, int mode)
{
    return (int64_t)d * ((mode & 2) ? N + 1 : 1) + oracle_num_pairs(N, mode & 1);
}

/*
 * Interaction forward (DLRM notes, section 3).  The vectors are z_0 = e0 and
 * z_i = pooled embedding i-1 for i = 1..N.  Output row of sample b:
 *   [ e0 (d values) | z_i . z_j for i = 0..N, j = 0..i-1 (strict) or
 *                     j = 0..i (self-inclusive), i outer, j inner ].
 * Readings: e0 takes part in the pairs (the architecture figure feeds the
 * bottom-MLP output into the interaction); "element-wise dot product" is the
 * scalar dot product; e0 is placed first in the concatenation; pairs are
 * listed by row i, then column j.
 */
int oracle_interact_fwd(int N, int d, int64_t B, int mode,
                        const double *e0, const double *e0_mag,
                        const double *emb, const double *emb_mag,
                        double *y, double *y_mag)
{
    if (N < 0 || d <= 0 || B < 0)
        return ORACLE_INVALID_ARG;
    int F = N + 1;
    int include_self = mode & 1;
    int64_t width = interact_width(N, d, mode);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t b = 0; b < B; b++) {
        double *yr = y + b * width;
        double *ym = y_mag + b * width;
        for (int e = 0; e < d; e++) {
            yr[e] = e0[b * d + e];
            ym[e] = mag_or_abs(e0_mag, e0, b * d + e);
        }
        int64_t p = d;
        if (mode & 2) { /* the original embeddings, in order */
            for (int i = 0; i < N; i++)
                for (int e = 0; e < d; e++) {
                    int64_t k = (b * N + i) * (int64_t)d + e;
                    yr[p] = emb[k];
                    ym[p] = mag_or_abs(emb_mag, emb, k);
                    p++;
                }
        }
        for (int i = 0; i < F; i++) {
            int jmax = include_self ? i : i - 1;
            for (int j = 0; j <= jmax; j++) {
                double dot = 0.0, mag = 0.0;
                for (int e = 0; e < d; e++) {
                    int64_t ii = (i == 0) ? b * d + e : (b * N + (i - 1)) * (int64_t)d + e;
                    int64_t jj = (j == 0) ? b * d + e : (b * N + (j - 1)) * (int64_t)d + e;
                    double zi = (i == 0) ? e0[ii] : emb[ii];
                    double zj = (j == 0) ? e0[jj] : emb[jj];
                    double mi = (i == 0) ? mag_or_abs(e0_mag, e0, ii) : mag_or_abs(emb_mag, emb, ii);
                    double mj = (j == 0) ? mag_or_abs(e0_mag, e0, jj) : mag_or_abs(emb_mag, emb, jj);
                    dot += zi * zj;
                    mag += mi * mj;
                }
                yr[p] = dot;
                ym[p] = mag;
                p++;
            }
        }
    }
    return ORACLE_OK;
}

/*
 * Interaction backward, by the product rule applied pair by pair: for an
 * upstream gradient g of the term z_i . z_j (i != j), z_i receives g * z_j
 * and z_j receives g * z_i; for a self term z_i . z_i, z_i receives
 * 2 * g * z_i.  e0 also receives the gradient of its copy in the output.
 * de0 is [B][d]; demb is [B][N][d].
 */
int oracle_interact_bwd(int N, int d, int64_t B, int mode,
                        const double *e0, const double *e0_mag,
                        const double *emb, const double *emb_mag,
                        const double *dy, const double *dy_mag,
                        double *de0, double *de0_mag, double *demb, double *demb_mag)
{
    if (N < 0 || d <= 0 || B < 0)
        return ORACLE_INVALID_ARG;
    int F = N + 1;
    int include_self = mode & 1;
    int64_t width = interact_width(N, d, mode);
    int failed = 0;
    /* one scratch pair per thread (a single one in the serial build) */
#pragma omp parallel
    {
        double *dz = (double *)calloc((size_t)F * d, sizeof(double));
        double *dzm = (double *)calloc((size_t)F * d, sizeof(double));
        if (!dz || !dzm) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t b = 0; b < B; b++) {
            if (!dz || !dzm)
                continue;
            memset(dz, 0, sizeof(double) * (size_t)F * d);
            memset(dzm, 0, sizeof(double) * (size_t)F * d);
            int64_t p = (mode & 2) ? (int64_t)F * d : d;
            for (int i = 0; i < F; i++) {
                int jmax = include_self ? i : i - 1;
                for (int j = 0; j <= jmax; j++) {
                    double g = dy[b * width + p];
                    double gm = mag_or_abs(dy_mag, dy, b * width + p);
                    p++;
                    for (int e = 0; e < d; e++) {
                        int64_t ii = (i == 0) ? b * d + e : (b * N + (i - 1)) * (int64_t)d + e;
                        int64_t jj = (j == 0) ? b * d + e : (b * N + (j - 1)) * (int64_t)d + e;
                        double zi = (i == 0) ? e0[ii] : emb[ii];
                        double zj = (j == 0) ? e0[jj] : emb[jj];
                        double mi = (i == 0) ? mag_or_abs(e0_mag, e0, ii) : mag_or_abs(emb_mag, emb, ii);
                        double mj = (j == 0) ? mag_or_abs(e0_mag, e0, jj) : mag_or_abs(emb_mag, emb, jj);
                        if (i == j) {
                            dz[(int64_t)i * d + e] += 2.0 * g * zi;
                            dzm[(int64_t)i * d + e] += 2.0 * gm * mi;
                        } else {
                            dz[(int64_t)i * d + e] += g * zj;
                            dzm[(int64_t)i * d + e] += gm * mj;
                            dz[(int64_t)j * d + e] += g * zi;
                            dzm[(int64_t)j * d + e] += gm * mi;
                        }
                    }
                }
            }
            for (int e = 0; e < d; e++) {
                de0[b * d + e] = dy[b * width + e] + dz[e];
                de0_mag[b * d + e] = mag_or_abs(dy_mag, dy, b * width + e) + dzm[e];
            }
            for (int i = 1; i < F; i++)
                for (int e = 0; e < d; e++) {
                    /* with the embeddings alongside, each also receives the gradient of its copy */
                    double cp = 0.0, cpm = 0.0;
                    if (mode & 2) {
                        cp = dy[b * width + (int64_t)i * d + e];
                        cpm = mag_or_abs(dy_mag, dy, b * width + (int64_t)i * d + e);
                    }
                    demb[(b * N + (i - 1)) * (int64_t)d + e] = cp + dz[(int64_t)i * d + e];
                    demb_mag[(b * N + (i - 1)) * (int64_t)d + e] = cpm + dzm[(int64_t)i * d + e];
                }
        }
        free(dz);
        free(dzm);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/* One lookup, keyed by (table, row) and tagged with its position. */
typedef struct {
    int64_t table;
    int64_t row;
    int64_t pos;
} lookup_key;

static int compare_lookup(const void *pa, const void *pb)
{
    const lookup_key *a = (const lookup_key *)pa, *b = (const lookup_key *)pb;
    if (a->table != b->table)
        return a->table < b->table ? -1 : 1;
    if (a->row != b->row)
        return a->row < b->row ? -1 : 1;
    if (a->pos != b->pos)
        return a->pos < b->pos ? -1 : 1;
    return 0;
}

/*
 * Coalescing of duplicate lookups before the sparse update: a stable sort of
 * the lookup positions by the key (table, row) -- ties keep their original
 * position order, which the position in the comparison makes explicit --
 * followed by run-length encoding of the sorted keys.
 * Outputs: sorted_pos[nnz], sorted_row[nnz]; for each unique key u (at most
 * nnz of them): uniq_table[u], uniq_row[u], seg_off[u] (first sorted
 * position of the run); seg_off[U] = nnz; *num_unique = U.
 */
int oracle_coalesce(int T, int64_t B, const int64_t *rows, const int64_t *offsets,
                    const int64_t *indices, int64_t nnz,
                    int64_t *sorted_pos, int64_t *sorted_row, int32_t *uniq_table,
                    int64_t *uniq_row, int64_t *seg_off, int64_t *num_unique)
{
    if (T <= 0 || B < 0 || nnz < 0)
        return ORACLE_INVALID_ARG;
    int st = check_offsets(T, B, offsets, nnz);
    if (st != ORACLE_OK)
        return st;
    lookup_key *keys = (lookup_key *)malloc(sizeof(lookup_key) * (size_t)(nnz > 0 ? nnz : 1));
    if (!keys)
        return ORACLE_NO_MEMORY;
    for (int t = 0; t < T; t++)
        for (int64_t b = 0; b < B; b++)
            for (int64_t k = offsets[(int64_t)t * B + b]; k < offsets[(int64_t)t * B + b + 1]; k++) {
                if (indices[k] < 0 || indices[k] >= rows[t]) {
                    free(keys);
                    return ORACLE_INDEX_OOB;
                }
                keys[k].table = t;
                keys[k].row = indices[k];
                keys[k].pos = k;
            }
    qsort(keys, (size_t)nnz, sizeof(lookup_key), compare_lookup);
    int64_t U = 0;
    for (int64_t j = 0; j < nnz; j++) {
        sorted_pos[j] = keys[j].pos;
        sorted_row[j] = keys[j].row;
        if (j == 0 || keys[j].table != keys[j - 1].table || keys[j].row != keys[j - 1].row) {
            uniq_table[U] = (int32_t)keys[j].table;
            uniq_row[U] = keys[j].row;
            seg_off[U] = j;
            U++;
        }
    }
    seg_off[U] = nnz;
    *num_unique = U;
    free(keys);
    return ORACLE_OK;
}

/*
 * Backward of the sum pooling plus row-wise SGD.  The gradient of row
 * uniq_row[u] of table uniq_table[u] is the sum, over the lookups of that
 * row (its run of the sorted order, summed in that order), of the gradient
 * of the pooled vector of the lookup's bag: grad[u] = sum_j dpooled[bag][t].
 * The updated row is W - lr * grad[u] (plain SGD on the touched rows only:
 * the reading of section 5 of the DLRM notes adopted for this path; rows no
 * lookup touched are left as they are).
 * dpooled is [B][T][d]; grad and new_row are [U][d].
 */
int oracle_sgd(int T, int d, int dtype, const void *const *tables, const int64_t *rows,
               int64_t B, const int64_t *offsets, int64_t nnz,
               const double *dpooled, const double *dpooled_mag, double lr,
               const int64_t *sorted_pos, const int32_t *uniq_table, const int64_t *uniq_row,
               const int64_t *seg_off, int64_t U,
               double *grad, double *grad_mag, double *new_row, double *new_row_mag)
{
    if (T <= 0 || d <= 0 || B < 0 || nnz < 0 || U < 0)
        return ORACLE_INVALID_ARG;
    int st = check_offsets(T, B, offsets, nnz);
    if (st != ORACLE_OK)
        return st;
    /* bag of each lookup position, from the CSR offsets */
    int64_t *bag_of = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nnz > 0 ? nnz : 1));
    if (!bag_of)
        return ORACLE_NO_MEMORY;
    for (int t = 0; t < T; t++)
        for (int64_t b = 0; b < B; b++)
            for (int64_t k = offsets[(int64_t)t * B + b]; k < offsets[(int64_t)t * B + b + 1]; k++)
                bag_of[k] = b;
    for (int64_t u = 0; u < U; u++)
        if (uniq_table[u] < 0 || uniq_table[u] >= T || uniq_row[u] < 0 || uniq_row[u] >= rows[uniq_table[u]]) {
            free(bag_of);
            return ORACLE_INDEX_OOB;
        }
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t u = 0; u < U; u++) {
        int t = uniq_table[u];
        int64_t r = uniq_row[u];
        for (int e = 0; e < d; e++) {
            double g = 0.0, gm = 0.0;
            for (int64_t j = seg_off[u]; j < seg_off[u + 1]; j++) {
                int64_t i = (bag_of[sorted_pos[j]] * T + t) * (int64_t)d + e;
                g += dpooled[i];
                gm += mag_or_abs(dpooled_mag, dpooled, i);
            }
            double w = table_element(tables[t], dtype, d, r * d + e);
            grad[u * d + e] = g;
            grad_mag[u * d + e] = gm;
            new_row[u * d + e] = w - lr * g;
            new_row_mag[u * d + e] = fabs(w) + fabs(lr) * gm;
        }
    }
    free(bag_of);
    return ORACLE_OK;
}

/*
 * Row-wise AdaGrad on the coalesced gradient.  The notes name AdaGrad as the
 * usual optimizer ("Notes/DLRM", section 5, Training) without its formula;
 * this is AdaGrad (Duchi, Hazan and Singer, 2011) with one accumulator per
 * row: the accumulator grows by the mean over the row of the squared
 * gradient, and every element of the row takes the same step size.
 *
 *   g[u]       = sum over the lookups of key u of dpooled    (as in oracle_sgd)
 *   s'         = s + (1/d) sum_e g[u][e]^2
 *   w'[e]      = w[e] - lr * g[u][e] / (sqrt(s') + eps)
 *
 * state[u] is s for key u (in), new_state[u] is s'.  Magnitudes bound the
 * effect of any summation order to first order, so that a result may differ
 * from the fp64 value by at most rel * magnitude:
 *   grad_mag   sum of |terms| (as in oracle_sgd);
 *   state_mag  s + (1/d) sum_e (2 |g| grad_mag + g^2): a change of g by
 *              rel * grad_mag moves g^2 by 2 |g| rel * grad_mag; g^2 covers
 *              the rounding of the squares and of their sum;
 *   row_mag    |w| + k (grad_mag + |g|) + |g| lr state_mag / (2 sqrt(s') r^2)
 *              with r = sqrt(s') + eps and k = lr / r: the first terms cover
 *              the change of g and the rounding of k g, the last the change
 *              of k when s' moves by rel * state_mag.
 * A row whose gradient is zero everywhere keeps w (its step is 0 / r).
 */
int oracle_adagrad(int T, int d, int dtype, const void *const *tables, const int64_t *rows,
                   int64_t B, const int64_t *offsets, int64_t nnz,
                   const double *dpooled, const double *dpooled_mag, double lr, double eps,
                   const int64_t *sorted_pos, const int32_t *uniq_table, const int64_t *uniq_row,
                   const int64_t *seg_off, int64_t U, const double *state,
                   double *grad, double *grad_mag, double *new_state, double *new_state_mag,
                   double *new_row, double *new_row_mag)
{
    if (T <= 0 || d <= 0 || B < 0 || nnz < 0 || U < 0 || !(eps >= 0.0))
        return ORACLE_INVALID_ARG;
    /* the gradients, exactly as the SGD oracle sums them */
    int st = oracle_sgd(T, d, dtype, tables, rows, B, offsets, nnz, dpooled, dpooled_mag, 0.0, sorted_pos,
                        uniq_table, uniq_row, seg_off, U, grad, grad_mag, new_row, new_row_mag);
    if (st != ORACLE_OK)
        return st;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t u = 0; u < U; u++) {
        const int t = uniq_table[u];
        const int64_t r = uniq_row[u];
        const double *g = grad + u * d, *gm = grad_mag + u * d;
        double q = 0.0, qm = 0.0;
        for (int e = 0; e < d; e++) {
            q += g[e] * g[e];
            qm += 2.0 * fabs(g[e]) * gm[e] + g[e] * g[e];
        }
        const double s1 = state[u] + q / d;
        new_state[u] = s1;
        new_state_mag[u] = fabs(state[u]) + qm / d;
        const double root = sqrt(s1), den = root + eps;
        for (int e = 0; e < d; e++) {
            const double w = table_element(tables[t], dtype, d, r * d + e);
            if (g[e] == 0.0) {
                new_row[u * d + e] = w;
                new_row_mag[u * d + e] = fabs(w) + (den > 0.0 ? fabs(lr) / den * gm[e] : 0.0);
                continue;
            }
            const double k = lr / den;
            new_row[u * d + e] = w - k * g[e];
            new_row_mag[u * d + e] = fabs(w) + fabs(k) * (gm[e] + fabs(g[e])) +
                                     fabs(g[e]) * fabs(lr) * new_state_mag[u] / (2.0 * root * den * den);
        }
    }
    return ORACLE_OK;
}

/*
 * Encodes a table of R rows of d values (fp32, fp16 or bf16; d even) into
 * the row-wise int4 layout above.  Per row, in fp32 arithmetic (the codes
 * are integers decided by floating point, so they are decided in one stated
 * precision): lo and hi are the row's minimum and maximum, s = (hi - lo) / 15,
 * b = lo (a zero minimum stored as +0), and q = the nearest integer (ties to
 * even) to (w - lo) / s, kept in 0 .. 15; a constant row (s = 0) gets q = 0.
 * Padding bytes are zero.  Rows are expected to be finite.
 */
int oracle_quantize_int4(int64_t R, int d, int src_dtype, const void *src, uint8_t *dst)
{
    if (R < 0 || d <= 0 || d % 2 != 0 || src_dtype < ORACLE_F32 || src_dtype > ORACLE_BF16)
        return ORACLE_INVALID_ARG;
    const int64_t rb = int4_row_bytes(d);
    for (int64_t r = 0; r < R; r++) {
        uint8_t *row = dst + r * rb;
        memset(row, 0, (size_t)rb);
        float lo = (float)table_element(src, src_dtype, d, r * d), hi = lo;
        for (int e = 1; e < d; e++) {
            float w = (float)table_element(src, src_dtype, d, r * d + e);
            if (w < lo)
                lo = w;
            if (w > hi)
                hi = w;
        }
        lo = lo + 0.0f; /* -0 becomes +0, so that the stored bias and scale are unique */
        hi = hi + 0.0f;
        float range = hi - lo;
        float scale = range / 15.0f;
        for (int e = 0; e < d; e++) {
            int q = 0;
            if (scale > 0.0f) {
                float w = (float)table_element(src, src_dtype, d, r * d + e);
                float diff = w - lo;
                float x = diff / scale;
                q = (int)rintf(x);
                q = q < 0 ? 0 : (q > 15 ? 15 : q);
            }
            row[e / 2] |= (uint8_t)(q << (4 * (e & 1)));
        }
        memcpy(row + d / 2, &scale, 4);
        memcpy(row + d / 2 + 4, &lo, 4);
    }
    return ORACLE_OK;
}

int64_t oracle_int4_row_bytes(int d)
{
    return int4_row_bytes(d);
}

