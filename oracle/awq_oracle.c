/*
 * awq_oracle.c -- plain CPU oracle for the AWQ W4A16 linear forward.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
 * CPU-baseline leg of the benchmark load this file. The library's GPU path
 * never calls it, and the two share no code, headers, tables or constants.
 *
 * What it computes, and where that is stated (Predibase Lorax "AWQ WQLinear"
 * page unless noted):
 *   - I/O Contract: qweight is int32 [in_features, out_features / 8], eight
 *     4-bit values per int32; qzeros are packed zero points; scales are
 *     per-group scale factors; bias is optional.
 *   - Description, __init__ bullets: in_features = rows of qweight,
 *     out_features = 8 x columns of qweight, group_size -1 means a single
 *     group spanning in_features, in_features % group_size == 0 and
 *     out_features % 8 == 0.
 *   - Overview and Description: the GEMM uses group-wise scaling, i.e. every
 *     block of group_size input rows is dequantised with its own zero point
 *     and scale: W[k, n] = (q[k, n] - zero[k / g, n]) * scale[k / g, n].
 *   - Description, forward steps 1-3: flatten x to 2-D, quantised GEMM,
 *     then add the optional bias.
 *
 * Readings where the page is silent (each one is listed with its reason in
 * the design notes):
 *   - nibble order: nibble i (bits 4i..4i+3, lowest first) of int32 j holds
 *     column 8j + i; qzeros use the same order, shape [K / g, N / 8].
 *   - scales are fp16, shape [K / g, N]; x, bias and y are fp16.
 *   - dequantised weights are rounded once to fp16 (round to nearest even),
 *     because that is the operand precision of an fp16 x fp16 matmul.
 *   - the matmul and the bias add are done here in fp64, with no rounding of
 *     the result: y_ref is an fp64 array.
 *
 * Everything is the plain definition: loops in the order the formula is
 * written, one double accumulator per output, k ascending. Threads only split
 * the output columns between them; every output is computed by one thread in
 * the same order as a single-threaded run would use.
 */
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#include <pthread.h>

#define ORACLE_OK 0
#define ORACLE_INVALID 1
#define ORACLE_NOMEM 2

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16, written out from its definition.                        */
/*   bits: sign (1) | exponent (5, bias 15) | fraction (10)                   */
/*   exponent 0      : subnormal, value = fraction * 2^-24                    */
/*   exponent 1..30  : normal, value = (1024 + fraction) * 2^(exponent - 25)  */
/*   exponent 31     : infinity (fraction 0) or NaN                           */
/* ------------------------------------------------------------------------ */

double awq_oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1F;
    int frac = h & 0x3FF;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), expo - 25);
    return sign ? -v : v;
}

/* Round a non-negative double to the nearest integer, ties to even. Every
 * caller passes y < 2^12, so floor(y) and y - floor(y) are exact. */
static double round_half_even(double y)
{
    double r = floor(y);
    double d = y - r;
    if (d > 0.5)
        return r + 1.0;
    if (d < 0.5)
        return r;
    return (fmod(r, 2.0) == 0.0) ? r : r + 1.0;
}

/* double -> binary16, round to nearest, ties to even (IEEE default mode). */
uint16_t awq_oracle_f64_to_f16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v))
        return (uint16_t)(sign | 0x7E00);
    /* The largest finite half is 65504; halfway to the next binade step
     * (65536) is 65520, which ties to the even neighbour 65536 = overflow. */
    if (a >= 65520.0)
        return (uint16_t)(sign | 0x7C00);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: value = m * 2^-24, m in [0, 1024]; m == 1024 is
         * the smallest normal, whose bit pattern is exactly 0x0400. */
        double m = round_half_even(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)m);
    }
    int e2;
    double f = frexp(a, &e2);   /* a = f * 2^e2, f in [0.5, 1) */
    int expo = e2 - 1;          /* a = (2f) * 2^expo, 2f in [1, 2) */
    /* significand with 10 fraction bits: a = s * 2^(expo - 10), s in [1024, 2048) */
    double s = round_half_even(ldexp(a, 10 - expo));
    if (s >= 2048.0) {          /* rounding carried into the next binade */
        s = 1024.0;
        expo += 1;
    }
    if (expo > 15)
        return (uint16_t)(sign | 0x7C00);
    return (uint16_t)(sign | (uint16_t)((expo + 15) << 10) | (uint16_t)((int)s - 1024));
}

void awq_oracle_f64_to_f16_array(const double *v, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = awq_oracle_f64_to_f16(v[i]);
}

void awq_oracle_f16_to_f64_array(const uint16_t *h, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = awq_oracle_f16_to_f64(h[i]);
}

/* ------------------------------------------------------------------------ */
/* Shape rules (WQLinear page, Description, __init__ bullets).               */
/* ------------------------------------------------------------------------ */

/* Resolves group_size: -1 means in_features. Returns ORACLE_INVALID for any
 * shape the page's assertions reject. */
int awq_oracle_resolve_group(int64_t in_features, int64_t out_features,
                             int64_t group_size, int64_t *g_out)
{
    if (in_features <= 0 || out_features <= 0)
        return ORACLE_INVALID;
    if (out_features % 8 != 0)
        return ORACLE_INVALID;
    int64_t g = (group_size == -1) ? in_features : group_size;
    if (g <= 0)
        return ORACLE_INVALID;
    if (in_features % g != 0)
        return ORACLE_INVALID;
    *g_out = g;
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Unpack: eight 4-bit codes per int32, nibble i of word j -> column 8j + i. */
/* ------------------------------------------------------------------------ */

int awq_oracle_unpack(const int32_t *packed, int64_t rows, int64_t out_features,
                      uint8_t *codes)
{
    if (rows < 0 || out_features <= 0 || out_features % 8 != 0)
        return ORACLE_INVALID;
    int64_t words = out_features / 8;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < words; ++j) {
            uint32_t w = (uint32_t)packed[r * words + j];
            for (int i = 0; i < 8; ++i)
                codes[r * out_features + 8 * j + i] = (uint8_t)((w >> (4 * i)) & 0xFu);
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Dequant: W16[k, n] = fp16_rn((q[k, n] - z[k / g, n]) * scale[k / g, n]).    */
/* (q - z) is an integer in [-15, 15] and scale an fp16 value, so the product */
/* is exact in double; the only rounding is the final one to fp16.           */
/* ------------------------------------------------------------------------ */

int awq_oracle_dequant(const int32_t *qweight, const int32_t *qzeros,
                       const uint16_t *scales, int64_t in_features,
                       int64_t out_features, int64_t group_size, uint16_t *W16)
{
    int64_t K = in_features, N = out_features, g;
    if (awq_oracle_resolve_group(K, N, group_size, &g) != ORACLE_OK)
        return ORACLE_INVALID;
    int64_t G = K / g;
    uint8_t *q = (uint8_t *)malloc((size_t)(K * N));
    uint8_t *z = (uint8_t *)malloc((size_t)(G * N));
    if (!q || !z) {
        free(q);
        free(z);
        return ORACLE_NOMEM;
    }
    awq_oracle_unpack(qweight, K, N, q);
    awq_oracle_unpack(qzeros, G, N, z);
    for (int64_t k = 0; k < K; ++k) {
        int64_t gi = k / g;
        for (int64_t n = 0; n < N; ++n) {
            int d = (int)q[k * N + n] - (int)z[gi * N + n];
            double s = awq_oracle_f16_to_f64(scales[gi * N + n]);
            W16[k * N + n] = awq_oracle_f64_to_f16((double)d * s);
        }
    }
    free(q);
    free(z);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Forward: y[m, n] = sum_k x[m, k] * W16[k, n]  (+ bias[n]), all in fp64.     */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t *x;
    const uint16_t *W16;
    const uint16_t *bias;
    const int64_t *rows;
    int64_t n_rows, K, N, n0, n1;
    double *y;
} fwd_job;

static void *fwd_worker(void *arg)
{
    fwd_job *j = (fwd_job *)arg;
    int64_t K = j->K, N = j->N, width = j->n1 - j->n0;
    if (width <= 0)
        return NULL;
    double *acc = (double *)malloc(sizeof(double) * (size_t)width);
    if (!acc)
        return (void *)1;
    for (int64_t r = 0; r < j->n_rows; ++r) {
        int64_t m = j->rows[r];
        for (int64_t n = 0; n < width; ++n)
            acc[n] = 0.0;
        /* for every output column, the terms are added for k = 0, 1, ..., K-1 */
        for (int64_t k = 0; k < K; ++k) {
            double xv = awq_oracle_f16_to_f64(j->x[m * K + k]);
            const uint16_t *wrow = j->W16 + k * N + j->n0;
            for (int64_t n = 0; n < width; ++n)
                acc[n] += xv * awq_oracle_f16_to_f64(wrow[n]);
        }
        for (int64_t n = 0; n < width; ++n) {
            double b = j->bias ? awq_oracle_f16_to_f64(j->bias[j->n0 + n]) : 0.0;
            j->y[r * N + j->n0 + n] = acc[n] + b;
        }
    }
    free(acc);
    return NULL;
}

/* The matmul and bias add of the forward, given the fp16 weights W16 [K, N]:
 * y[r, n] = sum_k x[rows[r], k] * W16[k, n] + bias[n] in fp64. rows: which
 * rows of x to evaluate (NULL = all M, in order); y: fp64 [n_rows, N].
 * threads <= 0 means one thread. */
static int forward_from_w16(const uint16_t *x, const uint16_t *W16, const uint16_t *bias,
                            int64_t M, int64_t K, int64_t N, const int64_t *rows,
                            int64_t n_rows, int threads, double *y)
{
    int64_t *all_rows = NULL;
    if (!rows) {
        n_rows = M;
        all_rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(M > 0 ? M : 1));
        if (!all_rows)
            return ORACLE_NOMEM;
        for (int64_t m = 0; m < M; ++m)
            all_rows[m] = m;
        rows = all_rows;
    }
    for (int64_t r = 0; r < n_rows; ++r) {
        if (rows[r] < 0 || rows[r] >= M) {
            free(all_rows);
            return ORACLE_INVALID;
        }
    }
    int rc = ORACLE_OK;
    if (threads < 1)
        threads = 1;
    if (threads > 256)
        threads = 256;
    /* split the output columns into equal blocks, one per thread */
    fwd_job jobs[256];
    pthread_t tids[256];
    int started[256];
    int64_t per = (N + threads - 1) / threads;
    for (int t = 0; t < threads; ++t) {
        int64_t n0 = (int64_t)t * per, n1 = n0 + per;
        if (n0 > N) n0 = N;
        if (n1 > N) n1 = N;
        fwd_job jb = {x, W16, bias, rows, n_rows, K, N, n0, n1, y};
        jobs[t] = jb;
        started[t] = (threads > 1) && pthread_create(&tids[t], NULL, fwd_worker, &jobs[t]) == 0;
        if (!started[t] && fwd_worker(&jobs[t]) != NULL)
            rc = ORACLE_NOMEM;
    }
    for (int t = 0; t < threads; ++t) {
        if (started[t]) {
            void *ret = NULL;
            pthread_join(tids[t], &ret);
            if (ret != NULL)
                rc = ORACLE_NOMEM;
        }
    }
    free(all_rows);
    return rc;
}

/* x: fp16 bits [M, K]; rows: which rows of x to evaluate (NULL = all M, in
 * order); y: fp64 [n_rows, N]. threads <= 0 means one thread. */
int awq_oracle_forward(const uint16_t *x, const int32_t *qweight,
                       const int32_t *qzeros, const uint16_t *scales,
                       const uint16_t *bias, int64_t M, int64_t in_features,
                       int64_t out_features, int64_t group_size,
                       const int64_t *rows, int64_t n_rows, int threads,
                       double *y)
{
    int64_t K = in_features, N = out_features, g;
    if (M < 0 || awq_oracle_resolve_group(K, N, group_size, &g) != ORACLE_OK)
        return ORACLE_INVALID;
    uint16_t *W16 = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(K * N));
    if (!W16)
        return ORACLE_NOMEM;
    int rc = awq_oracle_dequant(qweight, qzeros, scales, K, N, group_size, W16);
    if (rc == ORACLE_OK)
        rc = forward_from_w16(x, W16, bias, M, K, N, rows, n_rows, threads, y);
    free(W16);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Grouping by table (the "g_idx" variant): the group of input row k is       */
/* g_idx[k] instead of k / group_size, with G groups of scales and zeros:     */
/*   W16[k, n] = fp16_rn((q[k, n] - z[g_idx[k], n]) * scale[g_idx[k], n]).     */
/* Every g_idx[k] must lie in [0, G).                                          */
/* ------------------------------------------------------------------------ */

int awq_oracle_dequant_gidx(const int32_t *qweight, const int32_t *qzeros,
                            const uint16_t *scales, const int32_t *g_idx,
                            int64_t in_features, int64_t out_features, int64_t groups,
                            uint16_t *W16)
{
    int64_t K = in_features, N = out_features, G = groups;
    if (K <= 0 || N <= 0 || N % 8 != 0 || G <= 0)
        return ORACLE_INVALID;
    for (int64_t k = 0; k < K; ++k)
        if (g_idx[k] < 0 || g_idx[k] >= G)
            return ORACLE_INVALID;
    uint8_t *q = (uint8_t *)malloc((size_t)(K * N));
    uint8_t *z = (uint8_t *)malloc((size_t)(G * N));
    if (!q || !z) {
        free(q);
        free(z);
        return ORACLE_NOMEM;
    }
    awq_oracle_unpack(qweight, K, N, q);
    awq_oracle_unpack(qzeros, G, N, z);
    for (int64_t k = 0; k < K; ++k) {
        const int64_t row_group = g_idx[k];
        for (int64_t n = 0; n < N; ++n) {
            int diff = (int)q[k * N + n] - (int)z[row_group * N + n];
            double sc = awq_oracle_f16_to_f64(scales[row_group * N + n]);
            W16[k * N + n] = awq_oracle_f64_to_f16((double)diff * sc);
        }
    }
    free(q);
    free(z);
    return ORACLE_OK;
}

int awq_oracle_forward_gidx(const uint16_t *x, const int32_t *qweight,
                            const int32_t *qzeros, const uint16_t *scales,
                            const int32_t *g_idx, const uint16_t *bias, int64_t M,
                            int64_t in_features, int64_t out_features, int64_t groups,
                            const int64_t *rows, int64_t n_rows, int threads, double *y)
{
    int64_t K = in_features, N = out_features;
    if (M < 0 || K <= 0 || N <= 0)
        return ORACLE_INVALID;
    uint16_t *W16 = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(K * N));
    if (!W16)
        return ORACLE_NOMEM;
    int rc = awq_oracle_dequant_gidx(qweight, qzeros, scales, g_idx, K, N, groups, W16);
    if (rc == ORACLE_OK)
        rc = forward_from_w16(x, W16, bias, M, K, N, rows, n_rows, threads, y);
    free(W16);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Pack: the inverse of unpack. Code c of row r, column 8j + i goes to bits   */
/* 4i..4i+3 of int32 j of row r; only the low 4 bits of a code are used.      */
/* ------------------------------------------------------------------------ */

int awq_oracle_pack(const uint8_t *codes, int64_t rows, int64_t cols, int32_t *packed)
{
    if (rows < 0 || cols <= 0 || cols % 8 != 0)
        return ORACLE_INVALID;
    int64_t words = cols / 8;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < words; ++j) {
            uint32_t w = 0;
            for (int i = 0; i < 8; ++i)
                w |= (uint32_t)(codes[r * cols + 8 * j + i] & 0xFu) << (4 * i);
            packed[r * words + j] = (int32_t)w;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Round-to-nearest quantisation with given scales and zero points, the      */
/* inverse of the dequantisation above:                                      */
/*   q[k, n] = clamp(round_half_even(W[k, n] / s[k / g, n]) + z[k / g, n],    */
/*                   0, 15)                                                   */
/* The quotient of two fp16 values is computed in double. It is exact when   */
/* it is representable; otherwise it lies at least 2^-13 from any half        */
/* integer of magnitude up to 64 (numerator and denominator have 11-bit      */
/* significands), far more than a double rounding error, so rounding the     */
/* double quotient decides exactly as rounding the exact quotient would.     */
/* A NaN quotient (0 / 0) counts as 0. Clamping the quotient to [-64, 64]   */
/* before rounding (which also handles an infinite quotient) changes no      */
/* result: after the zero point is added the code is clamped to 0..15.       */
/* ------------------------------------------------------------------------ */

/* Nearest integer, ties to even, for |y| <= 64 (floor and y - floor exact). */
static double round_half_even_signed(double y)
{
    const double lo = floor(y);
    const double frac = y - lo;
    if (frac != 0.5)
        return frac < 0.5 ? lo : lo + 1.0;
    return (fmod(lo, 2.0) != 0.0) ? lo + 1.0 : lo;   /* a tie: the even neighbour */
}

int awq_oracle_quantize_rtn(const uint16_t *W16, const uint16_t *scales, const int32_t *qzeros,
                            int64_t in_features, int64_t out_features, int64_t group_size,
                            int32_t *qweight)
{
    int64_t K = in_features, N = out_features, g;
    if (awq_oracle_resolve_group(K, N, group_size, &g) != ORACLE_OK)
        return ORACLE_INVALID;
    int64_t G = K / g;
    uint8_t *q = (uint8_t *)malloc((size_t)(K * N));
    uint8_t *z = (uint8_t *)malloc((size_t)(G * N));
    if (!q || !z) {
        free(q);
        free(z);
        return ORACLE_NOMEM;
    }
    awq_oracle_unpack(qzeros, G, N, z);
    for (int64_t k = 0; k < K; ++k) {
        const int64_t grp = k / g;
        const uint16_t *srow = scales + grp * N;
        const uint8_t *zrow = z + grp * N;
        for (int64_t n = 0; n < N; ++n) {
            double w = awq_oracle_f16_to_f64(W16[k * N + n]);
            double t = w / awq_oracle_f16_to_f64(srow[n]);
            if (isnan(t))
                t = 0.0;
            if (t < -64.0)
                t = -64.0;
            if (t > 64.0)
                t = 64.0;
            int c = (int)round_half_even_signed(t) + (int)zrow[n];
            q[k * N + n] = (uint8_t)(c < 0 ? 0 : (c > 15 ? 15 : c));
        }
    }
    awq_oracle_pack(q, K, N, qweight);
    free(q);
    free(z);
    return ORACLE_OK;
}
