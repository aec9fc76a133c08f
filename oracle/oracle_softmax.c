/*
 * oracle_softmax.c -- CPU reference for the row softmax.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle that the GPU library is
 * checked against.  Only the tests, the smoke check and the bench's CPU-baseline
 * leg may load it; the library itself never does.  It shares no code, header or
 * constant with the CUDA path: its own storage decoding, its own loops, libm's
 * double-precision exp.
 *
 * What it computes is the plain definition of the numerically stable softmax,
 * written out step by step with no blocking, fusion or reordering:
 *
 *     m   = max_c x[c]                      (row max)
 *     e_c = exp(x[c] - m)                   (shifted exponentials)
 *     l   = sum_c e_c                       (normaliser, sequential sum)
 *     y_c = e_c / l
 *
 * Sources (page titles; sections):
 *   - "Dissecting Memory Bandwidth & SRAM Tiling in Triton: From GEMM to
 *     FlashAttention-3", section "The Mathematical Remedy: Online Softmax
 *     Tiling": the two-step definition (max, then shifted exponentials over
 *     their sum) and the merge rule for two partial (max, normaliser) states.
 *   - "I Wrote My First GPU Kernel -- Here's What Changed", sections "Why Naive
 *     Softmax Is Slow" and "What Fusion Actually Does": the four steps and the
 *     max subtraction that keeps exp from overflowing.
 *   - "GPU Kernels - Implementing and optimizing Softmax", "Baseline & Triton
 *     Softmax kernel": row-major rows addressed with a row stride, padded lanes
 *     read as -inf so that exp gives 0; "The tree reduction": stride-halving
 *     pairwise reduction of per-thread partials.
 *
 * Readings where the pages are silent (each also stated in the design notes):
 *   R1  a row whose entries are all -inf has no finite max; every output of
 *       that row is NaN (what -inf - (-inf) gives in every page's kernel);
 *   R2  a NaN anywhere in a row makes the whole row NaN;
 *   R3  a +inf entry makes the whole row NaN (IEEE: inf - inf);
 *   R4  the oracle returns exact-as-double results; rounding to the output
 *       dtype is the library's business and the tests' tolerance covers it.
 *
 * Storage: f32 rows are IEEE binary32; f16 rows are IEEE binary16 bit patterns;
 * bf16 rows are the top 16 bits of a binary32.  All are decoded here exactly
 * into double.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_F16 1
#define ORACLE_BF16 2

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0)              /* zero or subnormal: frac * 2^-24 */
        v = ldexp((double)frac, -24);
    else if (expo == 0x1f)      /* inf or NaN */
        v = frac ? NAN : INFINITY;
    else                        /* (1024 + frac) * 2^(expo - 15 - 10) */
        v = ldexp((double)(1024 + frac), expo - 25);
    return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_decode_bf16(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int expo = (b >> 7) & 0xff;
    int frac = b & 0x7f;
    double v;
    if (expo == 0)              /* zero or subnormal: frac * 2^(-126-7) */
        v = ldexp((double)frac, -133);
    else if (expo == 0xff)
        v = frac ? NAN : INFINITY;
    else                        /* (128 + frac) * 2^(expo - 127 - 7) */
        v = ldexp((double)(128 + frac), expo - 134);
    return sign ? -v : v;
}

static double load_elem(const void *base, int64_t idx, int dtype)
{
    if (dtype == ORACLE_F32) {
        float f;
        memcpy(&f, (const char *)base + idx * 4, 4);
        return (double)f;
    } else {
        uint16_t h;
        memcpy(&h, (const char *)base + idx * 2, 2);
        return dtype == ORACLE_F16 ? oracle_decode_f16(h) : oracle_decode_bf16(h);
    }
}

/*
 * Softmax of rows [row_begin, row_end) of a (rows x row_stride) matrix whose
 * first `cols` columns are valid.  Row r's result goes to
 * out[(r - row_begin) * cols + c] as double.  `scratch` holds `cols` doubles.
 * Returns 0, or -1 on bad arguments.
 */
int oracle_softmax_rows(const void *in, double *out, double *scratch,
                        int64_t row_begin, int64_t row_end, int64_t cols,
                        int64_t row_stride, int dtype)
{
    if (cols < 1 || row_stride < cols || row_begin > row_end)
        return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_F16 && dtype != ORACLE_BF16)
        return -1;
    for (int64_t r = row_begin; r < row_end; ++r) {
        double *y = out + (r - row_begin) * cols;
        double *x = scratch;
        int has_nan = 0;

        /* widen every valid entry of the row to double (exact) */
        for (int64_t c = 0; c < cols; ++c) {
            x[c] = load_elem(in, r * row_stride + c, dtype);
            if (isnan(x[c]))
                has_nan = 1;
        }

        /* step 1: the row max */
        double m = -INFINITY;
        for (int64_t c = 0; c < cols; ++c)
            if (x[c] > m)
                m = x[c];

        /* readings R1-R3: no finite shift exists, the row is NaN */
        if (has_nan || m == -INFINITY || m == INFINITY) {
            for (int64_t c = 0; c < cols; ++c)
                y[c] = NAN;
            continue;
        }

        /* step 2: shifted exponentials and their sequential sum */
        double l = 0.0;
        for (int64_t c = 0; c < cols; ++c) {
            y[c] = exp(x[c] - m);
            l += y[c];
        }

        /* step 3: normalise */
        for (int64_t c = 0; c < cols; ++c)
            y[c] = y[c] / l;
    }
    return 0;
}

/*
 * Scaled, causally masked softmax.  Page "Dissecting Memory Bandwidth & SRAM
 * Tiling in Triton: From GEMM to FlashAttention-3", section "Writing the
 * Kernel in OpenAI Triton": a score row is (Q_i K_j^T) * scale, and the causal
 * mask keeps key j only when j <= query i, the others becoming -inf before the
 * softmax (so their outputs are exp(-inf) = 0).
 *
 * Row r is query (r mod rows_per_seq) of its group of rows_per_seq rows
 * (rows_per_seq <= 0: one group holding every row) and keeps the columns
 * c <= query + causal_offset, i.e. n = clamp(query + causal_offset + 1, 0,
 * cols) of them.  The kept entries are multiplied by `scale` (in double) and
 * go through the steps of oracle_softmax_rows; the other outputs are 0, and
 * the masked inputs are never read.  A row that keeps no column is NaN
 * (reading R1).  scale must be finite and > 0.  Returns 0, or -1 on bad
 * arguments.
 */
int oracle_softmax_masked_rows(const void *in, double *out, double *scratch,
                               int64_t row_begin, int64_t row_end, int64_t cols,
                               int64_t row_stride, int dtype, double scale,
                               int64_t causal_offset, int64_t rows_per_seq)
{
    if (cols < 1 || row_stride < cols || row_begin > row_end || !(scale > 0.0) || isinf(scale))
        return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_F16 && dtype != ORACLE_BF16)
        return -1;
    for (int64_t r = row_begin; r < row_end; ++r) {
        double *y = out + (r - row_begin) * cols;
        double *x = scratch;
        const int64_t query = rows_per_seq > 0 ? r % rows_per_seq : r;
        int64_t n = query + causal_offset + 1;
        if (n < 0)
            n = 0;
        if (n > cols)
            n = cols;

        /* the masked outputs */
        for (int64_t c = n; c < cols; ++c)
            y[c] = 0.0;
        if (n == 0) {                       /* nothing kept: reading R1 */
            for (int64_t c = 0; c < cols; ++c)
                y[c] = NAN;
            continue;
        }

        /* widen and scale the kept entries */
        int has_nan = 0;
        for (int64_t c = 0; c < n; ++c) {
            x[c] = load_elem(in, r * row_stride + c, dtype) * scale;
            if (isnan(x[c]))
                has_nan = 1;
        }

        double m = -INFINITY;
        for (int64_t c = 0; c < n; ++c)
            if (x[c] > m)
                m = x[c];
        if (has_nan || m == -INFINITY || m == INFINITY) {
            for (int64_t c = 0; c < cols; ++c)
                y[c] = NAN;
            continue;
        }

        double l = 0.0;
        for (int64_t c = 0; c < n; ++c) {
            y[c] = exp(x[c] - m);
            l += y[c];
        }
        for (int64_t c = 0; c < n; ++c)
            y[c] = y[c] / l;
    }
    return 0;
}

/*
 * Attention forward for one head.  Page "Dissecting Memory Bandwidth & SRAM
 * Tiling in Triton: From GEMM to FlashAttention-3", sections "Memory
 * Hierarchy: Why Standard Attention Collapses" and "Writing the Kernel in
 * OpenAI Triton": scores S = Q K^T * scale, the causal mask (key j kept for
 * query i only when j <= i + causal_offset), P = the row softmax of S, and
 * O = P V.  Written out as the plain definition, one query row at a time in
 * double precision: the scores of the kept keys, their max, the shifted
 * exponentials and their sequential sum, then the weighted sum of the value
 * rows.
 *
 * q: n_q x d, k and v: n_k x d, row-major, dense, in the storage dtype;
 * out: n_q x d doubles.  `scratch` holds n_k doubles.  causal == 0 keeps
 * every key.  A query that keeps no key gets NaN (reading R1).  Returns 0, or
 * -1 on bad arguments.
 */
int oracle_attention_fwd(const void *q, const void *k, const void *v, double *out, double *scratch,
                         int64_t n_q, int64_t n_k, int64_t d, int dtype, double scale, int causal,
                         int64_t causal_offset)
{
    if (n_q < 0 || n_k < 1 || d < 1 || !(scale > 0.0) || isinf(scale))
        return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_F16 && dtype != ORACLE_BF16)
        return -1;
    for (int64_t i = 0; i < n_q; ++i) {
        double *o = out + i * d;
        double *p = scratch;
        int64_t n = n_k;
        if (causal) {
            n = i + causal_offset + 1;
            if (n < 0)
                n = 0;
            if (n > n_k)
                n = n_k;
        }
        if (n == 0) {
            for (int64_t c = 0; c < d; ++c)
                o[c] = NAN;
            continue;
        }
        /* scores of the kept keys */
        for (int64_t j = 0; j < n; ++j) {
            double acc = 0.0;
            for (int64_t c = 0; c < d; ++c)
                acc += load_elem(q, i * d + c, dtype) * load_elem(k, j * d + c, dtype);
            p[j] = acc * scale;
        }
        /* their softmax */
        double m = -INFINITY;
        int has_nan = 0;
        for (int64_t j = 0; j < n; ++j) {
            if (isnan(p[j]))
                has_nan = 1;
            if (p[j] > m)
                m = p[j];
        }
        if (has_nan || m == -INFINITY || m == INFINITY) {
            for (int64_t c = 0; c < d; ++c)
                o[c] = NAN;
            continue;
        }
        double l = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            p[j] = exp(p[j] - m);
            l += p[j];
        }
        /* the weighted sum of the value rows */
        for (int64_t c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int64_t j = 0; j < n; ++j)
                acc += p[j] * load_elem(v, j * d + c, dtype);
            o[c] = acc / l;
        }
    }
    return 0;
}

/*
 * The (max, normaliser) state of one row taken directly: m = max x,
 * l = sum exp(x - m).  Out: stats[0] = m, stats[1] = l.  Same readings as above
 * (a row with no finite shift gives m = NaN-or-inf, l = NaN).
 */
int oracle_row_stats(const void *in, int64_t row, int64_t c_begin, int64_t c_end,
                     int64_t row_stride, int dtype, double *stats)
{
    double m = -INFINITY, l = 0.0;
    int has_nan = 0;
    for (int64_t c = c_begin; c < c_end; ++c) {
        double v = load_elem(in, row * row_stride + c, dtype);
        if (isnan(v))
            has_nan = 1;
        else if (v > m)
            m = v;
    }
    if (has_nan || m == INFINITY) {
        stats[0] = m;
        stats[1] = NAN;
        return 0;
    }
    if (m == -INFINITY) {       /* empty or fully masked range: the merge identity */
        stats[0] = -INFINITY;
        stats[1] = 0.0;
        return 0;
    }
    for (int64_t c = c_begin; c < c_end; ++c)
        l += exp(load_elem(in, row * row_stride + c, dtype) - m);
    stats[0] = m;
    stats[1] = l;
    return 0;
}

/*
 * Merge of two partial states (page 4, "Online Softmax Tiling"):
 *     m = max(m1, m2),   l = l1 * exp(m1 - m) + l2 * exp(m2 - m).
 * A state with m = -inf is empty (l = 0) and leaves the other unchanged.
 */
void oracle_merge(double m1, double l1, double m2, double l2, double *m_out, double *l_out)
{
    if (m1 == -INFINITY) { *m_out = m2; *l_out = l2; return; }
    if (m2 == -INFINITY) { *m_out = m1; *l_out = l1; return; }
    double m = m1 > m2 ? m1 : m2;
    *m_out = m;
    *l_out = l1 * exp(m1 - m) + l2 * exp(m2 - m);
}

/*
 * Online (chunked) row statistics: the row's columns are split at the
 * `nbounds` increasing boundaries in `bounds` (bounds[0] = 0,
 * bounds[nbounds-1] = cols); each chunk's state is taken directly and folded
 * into a running state left to right with oracle_merge.  stats[0] = m,
 * stats[1] = l.
 */
int oracle_online_stats(const void *in, int64_t row, const int64_t *bounds, int64_t nbounds,
                        int64_t row_stride, int dtype, double *stats)
{
    double m = -INFINITY, l = 0.0, s[2];
    for (int64_t k = 0; k + 1 < nbounds; ++k) {
        oracle_row_stats(in, row, bounds[k], bounds[k + 1], row_stride, dtype, s);
        oracle_merge(m, l, s[0], s[1], &m, &l);
    }
    stats[0] = m;
    stats[1] = l;
    return 0;
}

/*
 * Stride-halving tree over n (a power of two) partial states, in the order of
 * the shared-memory tree on page 3 ("The tree reduction"): at stride
 * s = n/2, n/4, ..., 1, slot i < s becomes merge(slot i, slot i + s).
 * m and l are updated in place; after the call slot 0 holds the result.
 * If `trace` is non-null, after each round the first s maxima are appended to
 * it (so the caller can see every round's surviving values).
 */
int oracle_tree_merge(double *m, double *l, int64_t n, double *trace)
{
    if (n < 1 || (n & (n - 1)) != 0)
        return -1;
    int64_t t = 0;
    for (int64_t s = n / 2; s > 0; s /= 2) {
        for (int64_t i = 0; i < s; ++i)
            oracle_merge(m[i], l[i], m[i + s], l[i + s], &m[i], &l[i]);
        if (trace)
            for (int64_t i = 0; i < s; ++i)
                trace[t++] = m[i];
    }
    return 0;
}
