/*
 * oracle.h -- plain, slow, obviously-correct CPU oracle for batch-one N:M
 * bitmask SpMV.  TEST INFRASTRUCTURE ONLY: the CUDA library never includes,
 * links or calls anything declared here, and nothing here includes a CUDA
 * header.  Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load it.
 *
 * What it computes follows the SparseDecoding pages:
 *   - "The Kernel Is the Other Half of the Answer" (aimodeling.com article):
 *     the sparse format -- every 32 input columns of a row are described by
 *     one 32-bit mask word; at 50% sparsity each word has exactly 16 set bits;
 *     the mask replaces per-nonzero 32-bit column indices; the four patterns
 *     2:4, 4:8, 8:16 and 16:32 all keep 50% and carry identical metadata.
 *   - "What's new" (news.bitwarelabs.com summary) and the abstract
 *     (weekinpapers.com): batch-one decoding is dominated by the sparse
 *     matrix-vector product y = W x over the N:M-pruned weight matrix.
 * The plain result is y = W_pruned . x, so the oracle unpacks the compact
 * format back to a dense row and does a double-accumulated dot product.
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes): mask bit (c mod 32) of word c/32 describes column c (LSB = lowest
 * column); values are stored in ascending column order, row r's values start
 * at r*cols/2 and word w's 16 values start 16*w further on; an M-group is M
 * consecutive columns aligned to a multiple of M; the synthetic pruner keeps
 * the N entries of largest fp16 magnitude key (bits & 0x7FFF, compared as
 * unsigned), ties going to the lower column index.
 *
 * All fp16 data is passed as raw IEEE-754 binary16 bit patterns (uint16_t).
 * Every function returns 0 on success and a negative code on a bad argument.
 */
#ifndef NM_ORACLE_H
#define NM_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORC_OK 0
#define ORC_EINVAL (-1)

/* binary16 -> double, exact (every binary16 value is a double). */
double orc_f16_to_f64(uint16_t h);

/* double -> binary16, round to nearest, ties to even; overflow -> +-inf;
 * NaN -> quiet NaN 0x7E00 (sign kept). */
uint16_t orc_f16_from_f64(double v);

/* Prune + pack.  W is dense binary16 [rows][ld] (ld >= cols).  In every
 * M-group keep the N entries with the largest key = bits & 0x7FFF, ties to the
 * lower column.  Writes values [rows][cols/2] and masks [rows][cols/32].
 * Requires cols % 32 == 0 and N:M in {2:4, 4:8, 8:16, 16:32}. */
int orc_prune_pack(const uint16_t *W, int64_t rows, int64_t cols, int64_t ld,
                   int N, int M, uint16_t *values, uint32_t *masks);

/* Unpack: scatter values back by the masks into dense W_out [rows][ld];
 * unselected columns become +0.0 (0x0000).  Columns >= cols of each row
 * are not touched. */
int orc_unpack(const uint16_t *values, const uint32_t *masks, int64_t rows,
               int64_t cols, uint16_t *W_out, int64_t ld);

/* Dense matvec in double: y[r] = sum_c W[r][c] * x[c], summed in ascending c;
 * s[r] = sum_c |W[r][c]| * |x[c]| (the scale of the tolerance).  s may be
 * NULL. */
int orc_matvec_f64(const uint16_t *W, int64_t rows, int64_t cols, int64_t ld,
                   const uint16_t *x, double *y, double *s);

/* SpMV on the packed format for the listed rows only: each listed row is
 * unpacked to a dense scratch row and dotted with x in double (the same sum
 * as orc_matvec_f64).  row_ids[i] in [0, rows); y[i], s[i] are written for
 * row row_ids[i].  s may be NULL. */
int orc_spmv_rows_f64(const uint16_t *values, const uint32_t *masks,
                      int64_t rows, int64_t cols, const uint16_t *x,
                      const int64_t *row_ids, int64_t n_ids, double *y,
                      double *s);

/* SwiGLU of a gate/up pair of SpMV outputs, in double:
 * h[i] = silu(g[i]) * u[i], silu(t) = t / (1 + exp(-t)).  This is the
 * activation between the fused gate+up projection and the down projection of
 * the Llama/Qwen decoder layers the pages measure. */
int orc_silu_mul_f64(const double *g, const double *u, int64_t n, double *h);

/* Number of mask words whose popcount is not 16 (the 50% invariant). */
int64_t orc_count_bad_words(const uint32_t *masks, int64_t rows, int64_t cols);

#ifdef __cplusplus
}
#endif

#endif /* NM_ORACLE_H */
