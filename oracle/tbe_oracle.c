/*
 * Plain CPU oracle for the table-batched embedding (TBE) hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library calls or links this
 * file; only the tests, the package's smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header or helper with the CUDA path.
 *
 * What it computes (sources are the pages' sections, by page title):
 *
 *  - Forward pooled sum over KeyedJagged CSR input.  FBTriton TBE redesign
 *    (accesspath.com), "Backward kernels", problem statement and notation
 *    (T, E, D, L, B); TorchEasyRec analysis (39.107.221.112 article 1724244),
 *    section 1 "KeyedJaggedTensor" (all ids concatenated, one length per
 *    sample per feature, one fused lookup for all features).
 *  - Per-sample weights: FBTriton TBE redesign, "Backward kernels",
 *    weighted-tables paragraph (each gradient row is scaled by its per-sample
 *    weight before accumulation); the forward is read as the matching
 *    weighted pooled sum.
 *  - Batch inversion: FBTriton TBE redesign, "transpose_embedding_input"
 *    (linearise (table,row), sort, run-length encode into runs of one unique
 *    row with all positions touching it) and decision checklist item 6
 *    (int32 keys when the linearised range is below 2^31).
 *  - Backward: FBTriton TBE redesign, "Backward kernels": for every unique
 *    (table,row) touched by the batch, sum the upstream gradient rows of all
 *    positions touching it, then apply exactly one optimizer update to that
 *    row.
 *  - Optimizer: exact rowwise Adagrad (named in FBTriton TBE redesign,
 *    "Forward state reuse and preprocessing"):
 *        m[r] += mean_d(g[r,d]^2);  w[r,d] -= lr * g[r,d] / (sqrt(m[r]) + eps)
 *    with the updated m in the denominator, eps outside the square root.
 *  - Small-table histogram: FBTriton TBE redesign, "Forward state reuse and
 *    preprocessing" (forward histogram counts saved for backward) and
 *    decision checklist item 2 (E<=64, 64<=D<=128, L>=64, FP16, unweighted).
 *    The histogram path computes the same values as the generic path; the
 *    oracle for it is the generic definition plus the plain count function
 *    below.
 *
 * Arithmetic: every sum is accumulated in double, and every stored result is
 * rounded once from double to its stored type (float32 outputs and momentum;
 * the table dtype for weights, round-to-nearest-even).  The pages fix the
 * kernel's accumulation precision (decision checklist item 1: FP32 for
 * FP16/BF16 weights, FP64 for FP32 weights); the oracle is at least as
 * accurate as either, so a comparison measures the kernel's own rounding.
 *
 * Tables and bags.  Table t owns linearised rows [table_offset[t],
 * table_offset[t+1]) and is described by a layout record of 7 int64
 * (layout[t*7 + k]):
 *   k = 0  first byte of its rows in the weight buffer W (row r of the
 *          table, element d: byte 0 + ((r - table_offset[t]) * D + d) * size)
 *   k = 1  index in out / grad_out of bag 0's first element
 *   k = 2  elements from one bag's row to the next in out / grad_out
 *   k = 3  CSR bag index of its bag 0 (tables follow one another)
 *   k = 4  B_t, its bags in this batch
 *   k = 5  D_t, elements per row
 *   k = 6  dtype of its weights
 * One layout covers the uniform problem of the pages' notation (every table
 * with the same D, dtype and B; out = [B, T*D]), tables of different D and
 * dtype in one fused call (TorchEasyRec analysis, section 1: one lookup for
 * all features of a KeyedJagged batch), and variable batch size per table
 * (VBE, which the FBTriton TBE redesign names in decision checklist item 5;
 * read here as table t having its own B_t, its bags' rows packed one after
 * another in out and grad_out).
 *
 * Out-of-range indices (idx < 0 or idx >= E_t) are counted, contribute
 * nothing to the forward and take no part in the backward.
 *
 * Malformed offsets (the pages say nothing about them; this is the reading
 * both sides implement):
 *  - a bag g is well formed when 0 <= offsets[g] <= offsets[g+1] <= N; any
 *    other bag is malformed, counted, and empty;
 *  - lookups outside every well-formed bag (before offsets[0], after
 *    offsets[NB], or inside a malformed bag) take no part in the forward or
 *    the backward;
 *  - offsets that decrease anywhere (some bag with end < start) leave no
 *    single bag for a lookup that two well-formed bags both cover, so such a
 *    batch gets no backward update at all (its forward still pools each
 *    well-formed bag over its own range).
 *
 * Dtype codes: 0 = float32, 1 = float16, 2 = bfloat16.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Stored-type conversions, written from the IEEE 754 binary16 and the  */
/* bfloat16 (float32 with the low 16 bits dropped) encodings.           */

static double half_bits_to_double(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m | 1024), e - 25);     /* 1.m * 2^(e-15) */
    return s ? -v : v;
}

/* nearest binary16, ties to even (nearbyint in the default rounding mode) */
static uint16_t double_to_half_bits(double x)
{
    uint16_t s = signbit(x) ? 0x8000 : 0;
    if (isnan(x))
        return 0x7E00;
    double a = fabs(x);
    if (isinf(a))
        return s | 0x7C00;
    if (a < ldexp(1.0, -14)) {                     /* subnormal quantum 2^-24 */
        double q = nearbyint(ldexp(a, 24));        /* q == 1024 is the smallest normal */
        return s | (uint16_t)q;
    }
    int e;
    frexp(a, &e);                                  /* a in [2^(e-1), 2^e) */
    int E = e - 1;
    double q = nearbyint(ldexp(a, 10 - E));        /* significand in [1024, 2048] */
    if (q == 2048.0) {
        q = 1024.0;
        E += 1;
    }
    if (E > 15)
        return s | 0x7C00;
    return s | (uint16_t)((E + 15) << 10) | (uint16_t)((int)q - 1024);
}

static double bf16_bits_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* nearest bfloat16 (8-bit exponent, 7 stored significand bits), ties to even */
static uint16_t double_to_bf16_bits(double x)
{
    uint16_t s = signbit(x) ? 0x8000 : 0;
    if (isnan(x))
        return s | 0x7FC0;
    double a = fabs(x);
    if (isinf(a))
        return s | 0x7F80;
    if (a < ldexp(1.0, -126)) {                    /* subnormal quantum 2^-133 */
        double q = nearbyint(ldexp(a, 133));       /* q == 128 is the smallest normal */
        return s | (uint16_t)q;
    }
    int e;
    frexp(a, &e);
    int E = e - 1;
    double q = nearbyint(ldexp(a, 7 - E));         /* significand in [128, 256] */
    if (q == 256.0) {
        q = 128.0;
        E += 1;
    }
    if (E > 127)
        return s | 0x7F80;
    return s | (uint16_t)((E + 127) << 7) | (uint16_t)((int)q - 128);
}

static double load_w(const void *W, int dtype, int64_t i)
{
    if (dtype == 0)
        return (double)((const float *)W)[i];
    if (dtype == 1)
        return half_bits_to_double(((const uint16_t *)W)[i]);
    return bf16_bits_to_double(((const uint16_t *)W)[i]);
}

static void store_w(void *W, int dtype, int64_t i, double v)
{
    if (dtype == 0)
        ((float *)W)[i] = (float)v;
    else if (dtype == 1)
        ((uint16_t *)W)[i] = double_to_half_bits(v);
    else
        ((uint16_t *)W)[i] = double_to_bf16_bits(v);
}


/* exported for the conversion pins */
uint16_t tbe_oracle_to_half(double x) { return double_to_half_bits(x); }
uint16_t tbe_oracle_to_bf16(double x) { return double_to_bf16_bits(x); }
double tbe_oracle_from_half(uint16_t h) { return half_bits_to_double(h); }
double tbe_oracle_from_bf16(uint16_t h) { return bf16_bits_to_double(h); }

/* ------------------------------------------------------------------ */
/* Tables                                                              */

#define LAY(t, k) layout[(int64_t)(t) * 7 + (k)]

static int64_t elem_size(int64_t dtype) { return dtype == 0 ? 4 : 2; }

/* byte address of element 0 of linearised row `row` of table t */
static unsigned char *row_ptr(const void *W, const int64_t *layout, const int64_t *table_offset,
                              int64_t t, int64_t row)
{
    return (unsigned char *)W + LAY(t, 0) + (row - table_offset[t]) * LAY(t, 5) * elem_size(LAY(t, 6));
}

/* table of CSR bag g: the t with LAY(t,3) <= g < LAY(t,3) + LAY(t,4) */
static int64_t table_of_bag(const int64_t *layout, int32_t T, int64_t g)
{
    for (int64_t t = 0; t < T; ++t)
        if (g >= LAY(t, 3) && g < LAY(t, 3) + LAY(t, 4))
            return t;
    return -1;
}

/* table of linearised row `row` */
static int64_t table_of_row(const int64_t *table_offset, int32_t T, int64_t row)
{
    int64_t t = 0;
    while (t + 1 < T && table_offset[t + 1] <= row)
        ++t;
    return t;
}

static double sample_weight(const float *psw, const uint8_t *weighted, int64_t t, int64_t p)
{
    if (psw == NULL)
        return 1.0;
    if (weighted != NULL && !weighted[t])
        return 1.0;
    return (double)psw[p];
}

static int well_formed(const int64_t *offsets, int64_t g, int64_t N)
{
    int64_t s = offsets[g], e = offsets[g + 1];
    return 0 <= s && s <= e && e <= N;
}

/*
 * Forward pooled sum for a list of bags (all NB bags when bags == NULL).
 *
 *   out[row of bag (t,b) + d] = sum_{p in bag, 0 <= idx_p < E_t} w_p * W_t[idx_p, d]
 *
 * indices[N] and offsets[NB+1] are int64 (callers widen int32 inputs).  With
 * bags == NULL bag (t,b) writes its D_t elements at out[LAY(t,1) +
 * b*LAY(t,2) + d]; with a bag list, row k of out ([nbags, Dmax]) belongs to
 * bags[k].  abs_sum (nullable) receives sum |w_p * W[.., d]| in the same
 * layout: the scale that bounds any summation-order rounding of out.
 * Returns the number of out-of-range lookups in the bags visited;
 * *bad_bags (nullable) the number of malformed bags among them.
 */
int64_t tbe_oracle_forward(int32_t T, int64_t NB, const int64_t *layout, int32_t Dmax,
                           const void *W, const int64_t *table_offset, const int64_t *indices,
                           const int64_t *offsets, int64_t N, const float *psw,
                           const uint8_t *weighted, const int64_t *bags, int64_t nbags,
                           float *out, double *abs_sum, int64_t *bad_bags)
{
    int64_t oob = 0, bad = 0;
    int64_t n = bags ? nbags : NB;
    double *acc = (double *)malloc(sizeof(double) * (size_t)Dmax);
    double *aab = (double *)malloc(sizeof(double) * (size_t)Dmax);
    for (int64_t k = 0; k < n; ++k) {
        int64_t g = bags ? bags[k] : k;
        int64_t t = table_of_bag(layout, T, g), b = g - LAY(t, 3);
        int64_t E = table_offset[t + 1] - table_offset[t];
        int64_t D = LAY(t, 5), dtype = LAY(t, 6);
        for (int64_t d = 0; d < D; ++d)
            acc[d] = aab[d] = 0.0;
        int64_t start = offsets[g], end = offsets[g + 1];
        if (!well_formed(offsets, g, N)) {
            ++bad;                       /* malformed bag: empty */
            start = end = 0;
        }
        for (int64_t p = start; p < end; ++p) {
            int64_t idx = indices[p];
            if (idx < 0 || idx >= E) {
                ++oob;
                continue;
            }
            double w = sample_weight(psw, weighted, t, p);
            const unsigned char *wr = row_ptr(W, layout, table_offset, t, table_offset[t] + idx);
            for (int64_t d = 0; d < D; ++d) {
                double v = w * load_w(wr, (int)dtype, d);
                acc[d] += v;
                aab[d] += fabs(v);
            }
        }
        int64_t o = bags ? k * Dmax : LAY(t, 1) + b * LAY(t, 2);
        for (int64_t d = 0; d < D; ++d) {
            out[o + d] = (float)acc[d];
            if (abs_sum)
                abs_sum[o + d] = aab[d];
        }
    }
    free(acc);
    free(aab);
    if (bad_bags)
        *bad_bags = bad;
    return oob;
}

/* ------------------------------------------------------------------ */
/* Batch inversion: linearise, stable sort, run-length encode.          */

typedef struct {
    int64_t key;
    int64_t pos;
} kp_t;

static int cmp_key_pos(const void *a, const void *b)
{
    const kp_t *x = (const kp_t *)a, *y = (const kp_t *)b;
    if (x->key != y->key)
        return x->key < y->key ? -1 : 1;
    if (x->pos != y->pos)
        return x->pos < y->pos ? -1 : 1;
    return 0;
}

/*
 * Shape of the offsets array: *bad_bags = malformed bags (not
 * 0 <= offsets[g] <= offsets[g+1] <= N), *decreasing = 1 when some bag has
 * end < start, *span = 1 when offsets[0] != 0 or offsets[NB] != N.
 * Returns 1 when any of the three holds (the batch's offsets are malformed).
 */
int32_t tbe_oracle_offsets_check(int64_t NB, const int64_t *offsets, int64_t N,
                                 int64_t *bad_bags, int32_t *decreasing, int32_t *span)
{
    int64_t bad = 0;
    int32_t dec = 0;
    for (int64_t g = 0; g < NB; ++g) {
        if (offsets[g + 1] < offsets[g])
            dec = 1;
        if (!well_formed(offsets, g, N))
            ++bad;
    }
    int32_t sp = offsets[0] != 0 || offsets[NB] != N;
    if (bad_bags)
        *bad_bags = bad;
    if (decreasing)
        *decreasing = dec;
    if (span)
        *span = sp;
    return bad > 0 || dec || sp;
}

/*
 * CSR bag of every position p for the backward; -1 for positions in no
 * well-formed bag.  Offsets that decrease anywhere give -1 everywhere (such
 * a batch has no backward update).
 */
static int64_t *bag_of_positions(int64_t NB, const int64_t *offsets, int64_t N)
{
    int64_t *bag = (int64_t *)malloc(sizeof(int64_t) * (size_t)(N > 0 ? N : 1));
    for (int64_t p = 0; p < N; ++p)
        bag[p] = -1;
    int32_t dec = 0;
    tbe_oracle_offsets_check(NB, offsets, N, NULL, &dec, NULL);
    if (dec)
        return bag;
    for (int64_t g = 0; g < NB; ++g) {
        if (!well_formed(offsets, g, N))
            continue;
        for (int64_t p = offsets[g]; p < offsets[g + 1]; ++p)
            bag[p] = g;
    }
    return bag;
}

/*
 * key_p = table_offset[t] + idx_p for every in-range lookup p of a
 * well-formed bag (t its table; see bag_of_positions), sorted by (key, p)
 * -- a stable sort by key -- then run-length encoded:
 *   unique_keys[r], run_len[r], seg_off[r] (exclusive prefix sum of run_len,
 *   seg_off[U] = N' = number of in-range lookups).
 * sorted_keys/sorted_pos have N' entries.  Any output may be NULL.
 * Returns U.
 */
int64_t tbe_oracle_preprocess(int32_t T, int64_t NB, const int64_t *layout,
                              const int64_t *table_offset, const int64_t *indices,
                              const int64_t *offsets, int64_t N, int64_t *sorted_keys,
                              int64_t *sorted_pos, int64_t *unique_keys, int64_t *run_len,
                              int64_t *seg_off, int64_t *n_valid)
{
    int64_t *bag = bag_of_positions(NB, offsets, N);
    kp_t *kp = (kp_t *)malloc(sizeof(kp_t) * (size_t)(N > 0 ? N : 1));
    int64_t nv = 0;
    for (int64_t p = 0; p < N; ++p) {
        if (bag[p] < 0)
            continue;
        int64_t t = table_of_bag(layout, T, bag[p]);
        int64_t E = table_offset[t + 1] - table_offset[t];
        int64_t idx = indices[p];
        if (idx < 0 || idx >= E)
            continue;
        kp[nv].key = table_offset[t] + idx;
        kp[nv].pos = p;
        ++nv;
    }
    qsort(kp, (size_t)nv, sizeof(kp_t), cmp_key_pos);
    int64_t U = 0;
    for (int64_t i = 0; i < nv; ++i) {
        if (sorted_keys)
            sorted_keys[i] = kp[i].key;
        if (sorted_pos)
            sorted_pos[i] = kp[i].pos;
        if (i == 0 || kp[i].key != kp[i - 1].key) {
            if (unique_keys)
                unique_keys[U] = kp[i].key;
            if (seg_off)
                seg_off[U] = i;
            ++U;
        }
        if (run_len)
            run_len[U - 1] = (i == 0 || kp[i].key != kp[i - 1].key) ? 1 : run_len[U - 1] + 1;
    }
    if (seg_off)
        seg_off[U] = nv;
    if (n_valid)
        *n_valid = nv;
    free(kp);
    free(bag);
    return U;
}

/* ------------------------------------------------------------------ */
/* Backward with the fused exact rowwise Adagrad update.                 */

/* One exact rowwise Adagrad step on one row (D elements of dtype at wr,
 * its momentum *m) with row gradient g[0..D). */
static void adagrad_row(unsigned char *wr, float *m, int64_t D, int dtype, const double *g,
                        float lr, float eps)
{
    double ss = 0.0;
    for (int64_t d = 0; d < D; ++d)
        ss += g[d] * g[d];
    *m = (float)((double)*m + ss / (double)D);
    double den = sqrt((double)*m) + (double)eps;
    for (int64_t d = 0; d < D; ++d) {
        double w = load_w(wr, dtype, d);
        store_w(wr, dtype, d, w - (double)lr * g[d] / den);
    }
}

/*
 * Full backward in the pages' order: batch inversion (linearise, stable
 * sort, RLE), then for every run r (one unique row of table t) the row
 * gradient
 *     g[d] = sum_{p in run r, sorted order} w_p * grad_out[row of bag(p) + d]
 * and exactly one Adagrad update of that row.  W (bytes, laid out as the
 * layout says) and momentum are updated in place; rows no in-range lookup
 * touches are not written.
 * run_grad (nullable, [U, Dmax]) receives g of run r (rows in ascending key
 * order, the order of tbe_oracle_preprocess's unique_keys); run_abs
 * (nullable, [U, Dmax]) the sum |w_p * grad_out[..]| of the same terms (the
 * scale that bounds a summation-order rounding of g); update_count
 * (nullable, [rows_total]) counts updates applied per row.
 * Returns U, the number of rows updated.
 */
int64_t tbe_oracle_backward_adagrad(int32_t T, int64_t NB, const int64_t *layout, int32_t Dmax,
                                    void *W, float *momentum, const int64_t *table_offset,
                                    const int64_t *indices, const int64_t *offsets, int64_t N,
                                    const float *psw, const uint8_t *weighted,
                                    const float *grad_out, float lr, float eps,
                                    double *run_grad, double *run_abs, int32_t *update_count)
{
    int64_t *skeys = (int64_t *)malloc(sizeof(int64_t) * (size_t)(N > 0 ? N : 1));
    int64_t *spos = (int64_t *)malloc(sizeof(int64_t) * (size_t)(N > 0 ? N : 1));
    int64_t *ukeys = (int64_t *)malloc(sizeof(int64_t) * (size_t)(N > 0 ? N : 1));
    int64_t *soff = (int64_t *)malloc(sizeof(int64_t) * (size_t)(N + 1));
    int64_t U = tbe_oracle_preprocess(T, NB, layout, table_offset, indices, offsets, N, skeys, spos,
                                      ukeys, NULL, soff, NULL);
    int64_t *bag = bag_of_positions(NB, offsets, N);
    double *g = (double *)malloc(sizeof(double) * (size_t)Dmax);
    double *ga = (double *)malloc(sizeof(double) * (size_t)Dmax);
    for (int64_t r = 0; r < U; ++r) {
        int64_t row = ukeys[r];
        int64_t t = table_of_row(table_offset, T, row);
        int64_t D = LAY(t, 5);
        for (int64_t d = 0; d < D; ++d)
            g[d] = ga[d] = 0.0;
        for (int64_t i = soff[r]; i < soff[r + 1]; ++i) {
            int64_t p = spos[i];
            int64_t b = bag[p] - LAY(t, 3);
            double w = sample_weight(psw, weighted, t, p);
            const float *grow = grad_out + LAY(t, 1) + b * LAY(t, 2);
            for (int64_t d = 0; d < D; ++d) {
                g[d] += w * (double)grow[d];
                ga[d] += fabs(w * (double)grow[d]);
            }
        }
        if (run_grad)
            for (int64_t d = 0; d < D; ++d)
                run_grad[r * Dmax + d] = g[d];
        if (run_abs)
            for (int64_t d = 0; d < D; ++d)
                run_abs[r * Dmax + d] = ga[d];
        adagrad_row(row_ptr(W, layout, table_offset, t, row), momentum + row, D, (int)LAY(t, 6), g,
                    lr, eps);
        if (update_count)
            update_count[row] += 1;
    }
    free(g);
    free(ga);
    free(bag);
    free(soff);
    free(ukeys);
    free(spos);
    free(skeys);
    return U;
}

/* ------------------------------------------------------------------ */
/* Sampled rows, for full-size checks.                                   */

static int cmp_i64(const void *a, const void *b)
{
    int64_t x = *(const int64_t *)a, y = *(const int64_t *)b;
    return x < y ? -1 : (x > y ? 1 : 0);
}

/*
 * For k sampled linearised rows (sorted ascending, distinct) compute by one
 * scan over all lookups of the well-formed bags their lookup count, row
 * gradient (summed in position order, double; row_abs, nullable, the sum of
 * the terms' magnitudes) and the Adagrad result.  W_rows ([k] rows of
 * row_bytes bytes, each in its table's dtype and D) and mom_rows ([k]) hold
 * the rows' values before the update and are updated in place; rows with
 * count 0 are left untouched.  row_grad ([k, Dmax]) and counts ([k]) are
 * outputs.  Returns the number of in-range lookups scanned.
 */
int64_t tbe_oracle_rows_update(int32_t T, int64_t NB, const int64_t *layout, int32_t Dmax,
                               const int64_t *table_offset, const int64_t *indices,
                               const int64_t *offsets, int64_t N, const float *psw,
                               const uint8_t *weighted, const float *grad_out, float lr,
                               float eps, const int64_t *rows, int64_t k, void *W_rows,
                               int64_t row_bytes, float *mom_rows, double *row_grad,
                               double *row_abs, int64_t *counts)
{
    int64_t nv = 0;
    for (int64_t i = 0; i < k * Dmax; ++i) {
        row_grad[i] = 0.0;
        if (row_abs)
            row_abs[i] = 0.0;
    }
    for (int64_t i = 0; i < k; ++i)
        counts[i] = 0;
    int32_t dec = 0;
    tbe_oracle_offsets_check(NB, offsets, N, NULL, &dec, NULL);
    if (dec)
        return 0;                        /* decreasing offsets: no update */
    for (int64_t g = 0; g < NB; ++g) {
        if (!well_formed(offsets, g, N))
            continue;                    /* malformed bag */
        int64_t t = table_of_bag(layout, T, g), b = g - LAY(t, 3);
        int64_t E = table_offset[t + 1] - table_offset[t];
        int64_t D = LAY(t, 5);
        for (int64_t p = offsets[g]; p < offsets[g + 1]; ++p) {
            int64_t idx = indices[p];
            if (idx < 0 || idx >= E)
                continue;
            ++nv;
            int64_t key = table_offset[t] + idx;
            const int64_t *hit = (const int64_t *)bsearch(&key, rows, (size_t)k, sizeof(int64_t), cmp_i64);
            if (!hit)
                continue;
            int64_t r = hit - rows;
            double w = sample_weight(psw, weighted, t, p);
            const float *grow = grad_out + LAY(t, 1) + b * LAY(t, 2);
            for (int64_t d = 0; d < D; ++d) {
                row_grad[r * Dmax + d] += w * (double)grow[d];
                if (row_abs)
                    row_abs[r * Dmax + d] += fabs(w * (double)grow[d]);
            }
            counts[r] += 1;
        }
    }
    for (int64_t r = 0; r < k; ++r) {
        if (counts[r] == 0)
            continue;
        int64_t t = table_of_row(table_offset, T, rows[r]);
        adagrad_row((unsigned char *)W_rows + r * row_bytes, mom_rows + r, LAY(t, 5), (int)LAY(t, 6),
                    row_grad + r * Dmax, lr, eps);
    }
    return nv;
}

/* ------------------------------------------------------------------ */
/* Small-table histogram counts.                                         */

/*
 * counts[g*Emax + e] = #{p in bag g : idx_p == e}, for 0 <= e < E_t
 * (out-of-range lookups and malformed bags are not counted).  Emax >= every
 * E_t.  These are the forward's counts: a lookup that two well-formed bags
 * cover counts in both.  Returns the number of lookups counted.
 */
int64_t tbe_oracle_histogram(int32_t T, int64_t NB, const int64_t *layout, int32_t Emax,
                             const int64_t *table_offset, const int64_t *indices,
                             const int64_t *offsets, int64_t N, int32_t *counts)
{
    int64_t total = 0;
    memset(counts, 0, sizeof(int32_t) * (size_t)NB * (size_t)Emax);
    for (int64_t g = 0; g < NB; ++g) {
        if (!well_formed(offsets, g, N))
            continue;                    /* malformed bag: empty */
        int64_t t = table_of_bag(layout, T, g);
        int64_t E = table_offset[t + 1] - table_offset[t];
        for (int64_t p = offsets[g]; p < offsets[g + 1]; ++p) {
            int64_t idx = indices[p];
            if (idx < 0 || idx >= E)
                continue;
            counts[g * Emax + idx] += 1;
            ++total;
        }
    }
    return total;
}
