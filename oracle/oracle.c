/*
 * oracle.c -- plain CPU oracle for batch-one N:M bitmask SpMV (C99, double).
 *
 * TEST INFRASTRUCTURE: only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this file's library.  It shares no code, header,
 * table or constant with the CUDA library and includes no CUDA header.
 *
 * Sources (SparseDecoding pages):
 *   [K]  aimodeling.com article, section "The Kernel Is the Other Half of the
 *        Answer" -- bitmask format: one 32-bit mask word per 32 input columns,
 *        exactly 16 set bits per word at 50%, in place of per-nonzero 32-bit
 *        column indices; patterns 2:4, 4:8, 8:16, 16:32 all keep 50%.
 *   [W]  news.bitwarelabs.com summary, section "What's new" -- decoding is
 *        memory-bound and dominated by the sparse matrix-vector product.
 *   [A]  weekinpapers.com, Abstract -- "N:M sparse matrix-vector kernel with
 *        bitmask indexing and fixed-step traversal".
 * The method reaches exactly the plain product y = W_pruned x (up to the
 * order of rounding), so this file is that definition written out.
 *
 * Nothing here is blocked, fused or reordered: every loop walks its data in
 * the natural order so that it can be checked against the definition by eye.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16, written from the format's definition:                  */
/*   1 sign bit, 5 exponent bits (bias 15), 10 fraction bits;                */
/*   exponent 0 -> subnormal  (-1)^s * frac * 2^-24;                         */
/*   exponent 31 -> inf (frac 0) or NaN;                                     */
/*   otherwise (-1)^s * (1024 + frac) * 2^(exp - 25).                        */
/* ------------------------------------------------------------------------ */

double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1F;
    int frac = h & 0x3FF;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -24);
    } else if (expo == 31) {
        mag = (frac == 0) ? INFINITY : NAN;
    } else {
        mag = ldexp((double)(1024 + frac), expo - 25);
    }
    return sign ? -mag : mag;
}

/* Round a non-negative double to the nearest integer, ties to even. */
static double round_half_even(double n)
{
    double fl = floor(n);
    double diff = n - fl;
    if (diff > 0.5) return fl + 1.0;
    if (diff < 0.5) return fl;
    /* exactly halfway: pick the even neighbour */
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

uint16_t orc_f16_from_f64(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v)) return (uint16_t)(sign | 0x7E00u);
    double a = fabs(v);
    /* 65504 is the largest finite binary16; the midpoint to 2^16 is 65520,
     * and ties go to the even neighbour 2^16, which overflows to inf. */
    if (a >= 65520.0) return (uint16_t)(sign | 0x7C00u);

    /* quantum (spacing of binary16 values) at the magnitude of a */
    double q;
    if (a < ldexp(1.0, -14)) {
        q = ldexp(1.0, -24);                 /* subnormal spacing */
    } else {
        int e;
        (void)frexp(a, &e);                  /* a = m * 2^e, m in [0.5, 1) */
        q = ldexp(1.0, (e - 1) - 10);        /* 10 fraction bits */
    }
    double r = round_half_even(a / q) * q;   /* the rounded magnitude, exact */

    if (r == 0.0) return sign;
    if (r < ldexp(1.0, -14)) {
        /* subnormal: frac * 2^-24 */
        return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, -24)));
    }
    int e;
    double m = frexp(r, &e);                 /* r = m * 2^e, m in [0.5, 1) */
    int expo = (e - 1) + 15;
    int frac = (int)(m * 2048.0) - 1024;
    if (expo >= 31) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)(expo << 10) | (uint16_t)frac);
}

/* ------------------------------------------------------------------------ */
/* Pattern and shape checks                                                  */
/* ------------------------------------------------------------------------ */

static int valid_pattern(int N, int M)
{
    /* [K]: the four 50% patterns named on the page */
    return (N == 2 && M == 4) || (N == 4 && M == 8) || (N == 8 && M == 16) ||
           (N == 16 && M == 32);
}

static int popcount32(uint32_t w)
{
    int c = 0;
    for (int b = 0; b < 32; ++b) c += (int)((w >> b) & 1u);
    return c;
}

/* ------------------------------------------------------------------------ */
/* Prune + pack  ([K]; selection rule is the synthetic top-N-magnitude       */
/* pruner: key = bits & 0x7FFF as unsigned, larger first, lower column on a  */
/* tie).                                                                     */
/* ------------------------------------------------------------------------ */

int orc_prune_pack(const uint16_t *W, int64_t rows, int64_t cols, int64_t ld,
                   int N, int M, uint16_t *values, uint32_t *masks)
{
    if (!W || !values || !masks) return ORC_EINVAL;
    if (rows < 0 || cols < 0 || cols % 32 != 0 || ld < cols) return ORC_EINVAL;
    if (!valid_pattern(N, M)) return ORC_EINVAL;

    const int64_t words = cols / 32;
    int order[32];

    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t *row = W + r * ld;
        uint32_t *mrow = masks + r * words;
        for (int64_t w = 0; w < words; ++w) mrow[w] = 0u;

        /* 1. choose the kept columns of every M-group */
        for (int64_t g0 = 0; g0 < cols; g0 += M) {
            /* stable insertion sort of the group's positions by key,
             * descending; equal keys keep ascending column order */
            for (int i = 0; i < M; ++i) {
                int j = i;
                unsigned key_i = row[g0 + i] & 0x7FFFu;
                while (j > 0 && (unsigned)(row[g0 + order[j - 1]] & 0x7FFFu) < key_i) {
                    order[j] = order[j - 1];
                    --j;
                }
                order[j] = i;
            }
            /* keep the first N */
            for (int k = 0; k < N; ++k) {
                int64_t c = g0 + order[k];
                mrow[c / 32] |= 1u << (c % 32);
            }
        }

        /* 2. write the kept values in ascending column order; word w's
         *    values begin at 16*w within the row */
        uint16_t *vrow = values + r * (cols / 2);
        for (int64_t w = 0; w < words; ++w) {
            int k = 0;
            for (int b = 0; b < 32; ++b) {
                if ((mrow[w] >> b) & 1u) {
                    vrow[16 * w + k] = row[32 * w + b];
                    ++k;
                }
            }
            if (k != 16) return ORC_EINVAL; /* cannot happen for a 50% pattern */
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Unpack ([K]: the mask bits say which columns the compact values belong    */
/* to; with 16 values per word the k-th set bit takes value 16*w + k).       */
/* ------------------------------------------------------------------------ */

static int unpack_row(const uint16_t *vrow, const uint32_t *mrow, int64_t cols,
                      uint16_t *out)
{
    const int64_t words = cols / 32;
    for (int64_t w = 0; w < words; ++w) {
        if (popcount32(mrow[w]) != 16) return ORC_EINVAL;
        int k = 0;
        for (int b = 0; b < 32; ++b) {
            if ((mrow[w] >> b) & 1u) {
                out[32 * w + b] = vrow[16 * w + k];
                ++k;
            } else {
                out[32 * w + b] = 0x0000u; /* +0.0 */
            }
        }
    }
    return ORC_OK;
}

int orc_unpack(const uint16_t *values, const uint32_t *masks, int64_t rows,
               int64_t cols, uint16_t *W_out, int64_t ld)
{
    if (!values || !masks || !W_out) return ORC_EINVAL;
    if (rows < 0 || cols < 0 || cols % 32 != 0 || ld < cols) return ORC_EINVAL;
    for (int64_t r = 0; r < rows; ++r) {
        int rc = unpack_row(values + r * (cols / 2), masks + r * (cols / 32), cols,
                            W_out + r * ld);
        if (rc != ORC_OK) return rc;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Matrix-vector product in double ([W]: y = W x for one token).             */
/* ------------------------------------------------------------------------ */

static void dot_row(const uint16_t *row, const uint16_t *x, int64_t cols,
                    double *y, double *s)
{
    double acc = 0.0;
    double mag = 0.0;
    for (int64_t c = 0; c < cols; ++c) {
        double w = orc_f16_to_f64(row[c]);
        double xc = orc_f16_to_f64(x[c]);
        acc += w * xc;
        mag += fabs(w) * fabs(xc);
    }
    *y = acc;
    if (s) *s = mag;
}

int orc_matvec_f64(const uint16_t *W, int64_t rows, int64_t cols, int64_t ld,
                   const uint16_t *x, double *y, double *s)
{
    if (!W || !x || !y) return ORC_EINVAL;
    if (rows < 0 || cols < 0 || ld < cols) return ORC_EINVAL;
    for (int64_t r = 0; r < rows; ++r)
        dot_row(W + r * ld, x, cols, &y[r], s ? &s[r] : NULL);
    return ORC_OK;
}

int orc_spmv_rows_f64(const uint16_t *values, const uint32_t *masks,
                      int64_t rows, int64_t cols, const uint16_t *x,
                      const int64_t *row_ids, int64_t n_ids, double *y,
                      double *s)
{
    if (!values || !masks || !x || !row_ids || !y) return ORC_EINVAL;
    if (rows < 0 || cols < 0 || cols % 32 != 0 || n_ids < 0) return ORC_EINVAL;
    uint16_t *dense = (uint16_t *)malloc((size_t)(cols > 0 ? cols : 1) * sizeof(uint16_t));
    if (!dense) return ORC_EINVAL;
    int rc = ORC_OK;
    for (int64_t i = 0; i < n_ids && rc == ORC_OK; ++i) {
        int64_t r = row_ids[i];
        if (r < 0 || r >= rows) { rc = ORC_EINVAL; break; }
        rc = unpack_row(values + r * (cols / 2), masks + r * (cols / 32), cols, dense);
        if (rc == ORC_OK) dot_row(dense, x, cols, &y[i], s ? &s[i] : NULL);
    }
    free(dense);
    return rc;
}

int64_t orc_count_bad_words(const uint32_t *masks, int64_t rows, int64_t cols)
{
    if (!masks || rows < 0 || cols < 0 || cols % 32 != 0) return ORC_EINVAL;
    int64_t bad = 0;
    for (int64_t i = 0; i < rows * (cols / 32); ++i)
        if (popcount32(masks[i]) != 16) ++bad;
    return bad;
}

/* ------------------------------------------------------------------------ */
/* SwiGLU epilogue of the fused gate+up projection (the decoder layers the    */
/* pages measure -- Llama-3.1/3.3, Qwen3 -- feed silu(gate) * up into the     */
/* down projection).                                                         */
/* ------------------------------------------------------------------------ */

int orc_silu_mul_f64(const double *g, const double *u, int64_t n, double *h)
{
    if (!g || !u || !h || n < 0) return ORC_EINVAL;
    for (int64_t i = 0; i < n; ++i) {
        double silu = g[i] / (1.0 + exp(-g[i]));
        h[i] = silu * u[i];
    }
    return ORC_OK;
}
