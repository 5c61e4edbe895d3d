/*
 * nm_spmv.h -- C ABI of the batch-one N:M bitmask SpMV library (sm_103a).
 *
 * The operation (SparseDecoding pages):
 *   - news.bitwarelabs.com summary, "What's new": batch-one LLM decoding is
 *     memory-bandwidth bound and dominated by sparse matrix-vector products
 *     y = W x, one per linear layer per generated token.
 *   - aimodeling.com article, "The Kernel Is the Other Half of the Answer":
 *     W keeps exactly N of every M weights (2:4, 4:8, 8:16, 16:32, all 50%);
 *     every 32 input columns of a row are described by one 32-bit mask word
 *     with exactly 16 set bits, replacing per-nonzero 32-bit column indices,
 *     and the kernel walks the mask with fixed-step loops.  All four patterns
 *     carry identical metadata traffic.
 *   - weekinpapers.com, Abstract: "N:M sparse matrix-vector kernel with
 *     bitmask indexing and fixed-step traversal".
 *
 * Layout of the packed format (readings where the pages are silent):
 *   W is rows x cols (output dim x input dim), row-major; cols % 32 == 0.
 *   masks  : uint32 [rows][cols/32]; bit b of word w of row r describes
 *            column 32*w + b (least significant bit = lowest column).
 *   values : fp16   [rows][cols/2]; the kept entries of row r in ascending
 *            column order; row r starts at r*cols/2 and the 16 values of
 *            mask word w start at r*cols/2 + 16*w (the fixed step).
 *   An M-group is M consecutive columns starting at a multiple of M, so a
 *   group never straddles a mask word.  The packed bytes are the same for
 *   every pattern: rows*cols (values) + rows*cols/8 (masks).
 *
 * Conventions for every call:
 *   - fp16 means IEEE binary16 (CUDA __half); pointers marked "device" must
 *     point to device (or managed) memory of the current CUDA device.
 *   - The caller owns every buffer.  Only nm_check_masks allocates (an
 *     8-byte counter, freed before it returns); the library keeps no
 *     device memory between calls.  Host state is limited to per-device
 *     attribute caches.
 *   - stream is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls enqueue work and return at once, except where stated.
 *   - Arguments are validated on the host before anything is launched; a bad
 *     argument returns a nonzero nm_status and launches nothing.  A launch
 *     failure returns NM_ERR_CUDA (the CUDA error is left readable through
 *     cudaGetLastError's sticky state only if the context itself failed).
 *   - Calls are thread-safe; concurrent calls on different streams are fine
 *     as long as their output buffers do not overlap.
 */
#ifndef NM_SPMV_H
#define NM_SPMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NM_OK = 0,
    NM_ERR_NULL = 1,      /* a required pointer is NULL                        */
    NM_ERR_SHAPE = 2,     /* rows < 0, cols % 32 != 0, ld < cols, too large    */
    NM_ERR_PATTERN = 3,   /* (N, M) not one of 2:4, 4:8, 8:16, 16:32           */
    NM_ERR_ALIGN = 4,     /* a pointer or leading dimension is misaligned      */
    NM_ERR_WORKSPACE = 5, /* workspace missing or smaller than required        */
    NM_ERR_CUDA = 6,      /* a CUDA runtime call or kernel launch failed       */
    NM_ERR_ALIAS = 7      /* an output buffer overlaps an input buffer         */
} nm_status;

/* Human-readable name of a status code (static string, never NULL). */
const char *nm_status_string(int status);

/* Bytes of the packed arrays for a rows x cols matrix; identical for all
 * four patterns (aimodeling.com, "The Kernel Is the Other Half of the
 * Answer": identical metadata traffic).  0 for invalid shapes. */
size_t nm_values_bytes(int64_t rows, int64_t cols); /* rows*cols/2 fp16 = rows*cols bytes */
size_t nm_masks_bytes(int64_t rows, int64_t cols);  /* rows*cols/32 uint32 = rows*cols/8 bytes */

/* Device workspace nm_spmv needs for this shape, in bytes: 0 whenever
 * cols <= nm_spmv_max_cols() (every row is reduced inside one thread block);
 * longer rows are cut into column slices whose fp32 partial sums go through
 * the workspace (as nm_spmm with one token).  0 also for invalid shapes. */
size_t nm_spmv_workspace_bytes(int64_t rows, int64_t cols);

/* Largest cols for which nm_spmv keeps a whole row's x in one block's shared
 * memory (and needs no workspace) on the current device. */
int64_t nm_spmv_max_cols(void);

/* ---------------------------------------------------------------------------
 * nm_pack -- prune a dense fp16 matrix to N:M and pack it.
 *   W      : device fp16 [rows][ld], ld >= cols, row stride ld elements.
 *   N, M   : one of (2,4), (4,8), (8,16), (16,32).
 *   values : device fp16 [rows][cols/2] (output), 16-byte aligned.
 *   masks  : device uint32 [rows][cols/32] (output), 4-byte aligned.
 * Per M-group the N entries with the largest magnitude key
 * (fp16 bits & 0x7FFF, compared as unsigned; NaN ranks above inf) are kept,
 * ties going to the lower column.  Integer-only, so the result is bit-exact.
 * An input that is already N:M-sparse keeps its nonzeros (a kept zero may be
 * exchanged for a lower-column zero, which leaves the values unchanged).
 * Outputs must not overlap W.  rows == 0 is a no-op.
 * ------------------------------------------------------------------------- */
int nm_pack(const void *W, int64_t rows, int64_t cols, int64_t ld, int N, int M,
            void *values, uint32_t *masks, void *stream);

/* nm_unpack -- inverse of nm_pack: scatter values by masks into dense fp16
 * W_out [rows][ld] (device); unselected columns are written +0.0, columns
 * >= cols of each row are not touched.  Every mask word must have popcount
 * 16; a word that does not is decoded in bounds but its row is unspecified. */
int nm_unpack(const void *values, const uint32_t *masks, int64_t rows, int64_t cols,
              void *W_out, int64_t ld, void *stream);

/* ---------------------------------------------------------------------------
 * nm_spmv -- y = W x for one token (batch 1), W in the packed format.
 *   values    : device fp16 [rows][cols/2], 32-byte aligned.
 *   masks     : device uint32 [rows][cols/32], 4-byte aligned.
 *   x         : device fp16 [cols], 16-byte aligned.
 *   y         : device fp16 [rows] (output), must not overlap the inputs.
 *   workspace : device scratch, 16-byte aligned, of at least
 *               nm_spmv_workspace_bytes(rows, cols) bytes (NULL when that is 0,
 *               i.e. for cols <= nm_spmv_max_cols()).
 * Products and sums are fp32 (fp32 fused multiply-add); y is rounded to fp16
 * with round-to-nearest-even.  The summation order is fixed for a shape and
 * device, so repeated calls give bit-identical y.  Takes no N or M: the
 * packed format is the same for all four patterns.
 * Pruned weights are structural zeros and are never multiplied: a
 * non-finite x[c] reaches only the rows that keep column c (where IEEE rules
 * apply: inf * w = +-inf, NaN propagates, +inf + -inf = NaN); every other row
 * is what it would be with x[c] = 0.
 * Precondition: every mask word has popcount 16 (nm_pack guarantees it; use
 * nm_check_masks for untrusted data).  A word that breaks it is still read
 * in bounds, but the affected rows are unspecified.
 * Rows longer than nm_spmv_max_cols() run column-sliced through the
 * workspace (still deterministic); an explicit-plan nm_spmv_ex call for such
 * a shape returns NM_ERR_SHAPE.  rows == 0 is a no-op.
 * ------------------------------------------------------------------------- */
int nm_spmv(const void *values, const uint32_t *masks, int64_t rows, int64_t cols,
            const void *x, void *y, void *workspace, size_t workspace_bytes,
            void *stream);

/* ---------------------------------------------------------------------------
 * nm_spmv_swiglu -- the gate+up projection of a decoder layer with its SwiGLU
 * activation fused: h[i] = silu(g_i) * u_i, silu(t) = t / (1 + e^-t), where
 * g = W_gate x and u = W_up x.  The pages time whole decoding steps of
 * Llama/Qwen layers (aimodeling.com article, "The Kernel Is the Other Half of
 * the Answer"), whose gate and up projections feed exactly this product into
 * the down projection; fusing it saves writing and re-reading both outputs.
 *   The packed matrix interleaves the two projections: row 2i is gate row i,
 *   row 2i+1 is up row i (rows = 2 * hidden, even); pack W_gate and W_up
 *   row-interleaved with nm_pack.
 *   h : device fp16 [rows / 2], must not overlap the inputs.
 * g and u are the same fp32 sums nm_spmv would round to fp16; silu and the
 * product are evaluated in fp32 and h is rounded once to fp16 (RNE).
 * Other arguments and errors as nm_spmv (rows odd -> NM_ERR_SHAPE).
 * ------------------------------------------------------------------------- */
int nm_spmv_swiglu(const void *values, const uint32_t *masks, int64_t rows, int64_t cols,
                   const void *x, void *h, void *stream);
int nm_spmv_swiglu_ex(const void *values, const uint32_t *masks, int64_t rows, int64_t cols,
                      const void *x, void *h, int variant, int grid, int flags, void *stream);

/* ---------------------------------------------------------------------------
 * nm_spmm -- Y = W X for a small batch of tokens (1..8), W in the packed
 * format.  Decoding several tokens at once (small-batch serving, speculative
 * decoding) is the step between the batch-one SpMV and the prefill SpMM the
 * pages contrast it with (news.bitwarelabs.com summary, "What's new").  Each
 * mask word is decoded once for the whole batch.
 *   X : device fp16 [batch][ldx], 16-byte aligned, ldx % 8 == 0, ldx >= cols;
 *       token j's activations are X[j][0..cols).
 *   Y : device fp16 [batch][ldy], ldy >= rows; Y[j][r] = sum_c W[r][c] X[j][c].
 *   workspace : device scratch, 16-byte aligned, of at least
 *       nm_spmm_workspace_bytes(rows, cols, batch) bytes (0 when a whole row's
 *       x tile fits in one block's shared memory, else fp32 partial sums of
 *       column slices; for batch > 8, nm_spmm_prefill_workspace_bytes).  May
 *       be NULL when that is 0.
 * Same arithmetic, rounding, determinism and structural-zero rule as nm_spmv
 * (a non-finite activation of token j reaches only column j of Y); each column of Y is
 * within the same tolerance of the exact product (and equals nm_spmv's
 * result whenever the sums are exact).  nm_spmm with batch > 8 is served by
 * nm_spmm_prefill_ws (tensor cores; its numerics); nm_spmm_ex and
 * nm_spmm_workspace_bytes_ex take batch 1..8 only.  batch < 1 -> NM_ERR_SHAPE;
 * a short workspace -> NM_ERR_WORKSPACE.  Y must not overlap any input or the
 * workspace.
 * ------------------------------------------------------------------------- */
size_t nm_spmm_workspace_bytes(int64_t rows, int64_t cols, int batch);
int nm_spmm(const void *values, const uint32_t *masks, int64_t rows, int64_t cols,
            const void *X, int64_t ldx, int batch, void *Y, int64_t ldy,
            void *workspace, size_t workspace_bytes, void *stream);
/* Explicit plan: kernel variant (< 0: default), grid (<= 0: default), column
 * slices (<= 0: the fewest that fit), launch flags as for nm_spmv_ex.  The
 * workspace such a plan needs is nm_spmm_workspace_bytes_ex(rows, cols,
 * batch, variant, slices) (0 also for a plan that cannot run). */
int nm_spmm_variant_count(void);
size_t nm_spmm_workspace_bytes_ex(int64_t rows, int64_t cols, int batch, int variant,
                                  int slices);
int nm_spmm_ex(const void *values, const uint32_t *masks, int64_t rows, int64_t cols,
               const void *X, int64_t ldx, int batch, void *Y, int64_t ldy,
               void *workspace, size_t workspace_bytes, int variant, int grid, int slices,
               int flags, void *stream);

/* ---------------------------------------------------------------------------
 * nm_spmm24 -- Y = W X for 1..8 tokens when W is 2:4: every aligned group of
 * four columns keeps exactly two (the packing nm_pack makes with N = 2,
 * M = 4, the pattern of the pages' sparse tensor cores; aimodeling.com
 * article, "The Kernel Is the Other Half of the Answer").  Same packed
 * format and arguments as nm_spmm; with 2:4 masks each group's two values
 * are one fixed 32-bit pair of the word's values, so the kernel expands every
 * 16 x 16 tile of W to dense fp16 in registers (two byte permutes per group)
 * and multiplies it with the 8-token x tile by mma.sync.m16n8k16 (fp16 x fp16
 * products, fp32 accumulation): x is read once per 16 rows, not once per kept
 * weight, so the cost no longer grows with the batch (at 6-8 tokens it is
 * the faster of the two on the large decoder matrices).
 *   cols % 128 == 0 (any decoder shape) and ceil(rows / 16) * (cols / 128)
 *   < 2^31; X, Y, ldx, ldy, values, masks as for nm_spmm.
 *   workspace : device scratch, 16-byte aligned, of at least
 *       nm_spmm24_workspace_bytes(rows, cols, batch) bytes (fp32 partial sums
 *       of 16-row panels cut between warps -- 1 KB per warp of the grid, and
 *       per panel and column slice when the columns are sliced -- and a
 *       counter per panel), ZERO-FILLED before its first use (e.g.
 *       cudaMemsetAsync).  Every call leaves it zero-filled again, so it can
 *       be reused by any later nm_spmm24 call on the same stream; it must
 *       not overlap any argument.
 * Numerics as nm_spmm_prefill: pruned weights enter the products as +0 (a
 * non-finite X[t][c] turns every row of token t into NaN), fixed summation
 * order (identical bits across calls with the same plan), each element within
 * the nm_spmv tolerance of the exact product and equal to it whenever the
 * sums are exact.  A mask group that does not hold exactly two set bits is
 * decoded in bounds (its first two set columns take the group's two values,
 * further ones +0) and that row's result is unspecified; nm_check_masks does
 * not detect this.  rows == 0 is a no-op.  Errors: NM_ERR_SHAPE (cols not a
 * multiple of 128, batch outside 1..8, bad plan), NM_ERR_WORKSPACE, and the
 * nm_spmm ones.  One launch: each block first copies its column slice of X
 * into shared memory in operand order (16 bytes per column, at most 8192
 * columns per slice: 4 slices for the 70B down projection).
 * nm_spmm24_ex takes the plan: variant (< 0: default, 1; 0..count-1: warps
 * per block x 128-column units in flight per warp x accumulator chains =
 * 16x3x2, 20x1x4, 16x2x1, 12x4x2, 24x1x4, 20x2x1), grid (<= 0: one block per
 * SM; at most 65536; rounded down to a whole number of blocks per column
 * slice) and launch flags as for nm_spmv_ex; its workspace is
 * nm_spmm24_workspace_bytes_ex(rows, cols, batch, variant, grid).
 * ------------------------------------------------------------------------- */
size_t nm_spmm24_workspace_bytes(int64_t rows, int64_t cols, int batch);
int nm_spmm24(const void *values, const uint32_t *masks, int64_t rows, int64_t cols,
              const void *X, int64_t ldx, int batch, void *Y, int64_t ldy,
              void *workspace, size_t workspace_bytes, void *stream);
int nm_spmm24_variant_count(void);
size_t nm_spmm24_workspace_bytes_ex(int64_t rows, int64_t cols, int batch, int variant,
                                    int grid);
int nm_spmm24_ex(const void *values, const uint32_t *masks, int64_t rows, int64_t cols,
                 const void *X, int64_t ldx, int batch, void *Y, int64_t ldy,
                 void *workspace, size_t workspace_bytes, int variant, int grid, int flags,
                 void *stream);

/* ---------------------------------------------------------------------------
 * dense_gemv -- the dense baseline y = W x on an unpruned fp16 matrix
 * (aimodeling.com article, "The Kernel Is the Other Half of the Answer":
 * speedups are stated against dense decoding throughput).
 *   W : device fp16 [rows][ld], 16-byte aligned, ld % 8 == 0, ld >= cols.
 *   x : device fp16 [cols], 16-byte aligned;  y : device fp16 [rows].
 * Same arithmetic and rounding as nm_spmv.  cols <= nm_spmv_max_cols() * 2.
 * ------------------------------------------------------------------------- */
int dense_gemv(const void *W, int64_t rows, int64_t cols, int64_t ld,
               const void *x, void *y, void *stream);

/* ---------------------------------------------------------------------------
 * Launch flags (the _ex entry points take them; nm_spmv and dense_gemv use
 * NM_FLAG_PDL).
 *   NM_FLAG_PDL: launch with programmatic dependent launch, so the kernel can
 *     be scheduled while the previous kernel on the stream drains.  It waits
 *     for that kernel's completion before reading or writing any buffer, so
 *     stream order is kept for every argument.
 *   NM_FLAG_WEIGHTS_CONST: the caller promises that the weights (values and
 *     masks, or W) were not written by the previous kernel on the stream; the
 *     first weight loads are then issued before that wait.  x and y are still
 *     touched only after it.  Only meaningful with NM_FLAG_PDL.
 * ------------------------------------------------------------------------- */
#define NM_FLAG_PDL 1
#define NM_FLAG_WEIGHTS_CONST 2

/* ---------------------------------------------------------------------------
 * Launch plans.  nm_spmv and dense_gemv pick a plan from the shape and the
 * device: a kernel variant (warps per block x 256-bit steps in flight per
 * warp) and a grid (one persistent block per SM, never more blocks than
 * rows).  The _ex forms take the plan explicitly -- variant < 0 or grid <= 0
 * select the default -- for tuning sweeps and for tests that make rows be
 * cut between warps and blocks at many different places.  The result is
 * within the same tolerance for every plan; it is bit-identical across calls
 * with the same plan.  Bad variants return NM_ERR_SHAPE.
 * ------------------------------------------------------------------------- */
int nm_spmv_plan(int64_t rows, int64_t cols, int *variant, int *grid, int *warps);
int nm_spmv_variant_count(void);
int nm_spmv_ex(const void *values, const uint32_t *masks, int64_t rows, int64_t cols,
               const void *x, void *y, void *workspace, size_t workspace_bytes,
               int variant, int grid, int flags, void *stream);
int dense_gemv_variant_count(void);
int dense_gemv_ex(const void *W, int64_t rows, int64_t cols, int64_t ld,
                  const void *x, void *y, int variant, int grid, int flags, void *stream);

/* ---------------------------------------------------------------------------
 * nm_check_masks -- validator for untrusted masks (host-synchronous).
 * Returns the number of mask words whose popcount is not 16 (0 = valid), or
 * a negative nm_status on error.  Allocates and frees an 8-byte device
 * counter on the stream and waits for the stream.
 * ------------------------------------------------------------------------- */
int64_t nm_check_masks(const uint32_t *masks, int64_t rows, int64_t cols, void *stream);

/* ---------------------------------------------------------------------------
 * nm_spmm_prefill -- Y = W X for a prefill-sized batch of T tokens (any
 * T >= 1; meant for T beyond the 1..8 of nm_spmm), W in the packed format, on
 * the tensor cores.  Prefill is the compute-bound regime the pages set
 * against batch-one decoding (aimodeling.com article, "The Kernel Is the
 * Other Half of the Answer"; news.bitwarelabs.com summary, "What's new"):
 * each block expands a 128-row tile of W from values + masks into dense fp16
 * in shared memory and multiplies it with up to 512 tokens of X by
 * tcgen05.mma (fp16 x fp16 products, fp32 accumulation in tensor memory).
 *   X : device fp16 [T][ldx], 16-byte aligned, ldx % 8 == 0, ldx >= cols;
 *       token t's activations are X[t][0..cols).
 *   Y : device fp16 [T][ldy] (output), ldy >= rows; Y[t][r] = sum_c W[r][c] X[t][c],
 *       rounded once to fp16 (round-to-nearest-even).
 *   values / masks : as for nm_spmv (values 32-byte aligned).
 * Pruned weights enter the products as +0 (so, unlike nm_spmv, a non-finite
 * X[t][c] also turns the rows that do not keep column c into NaN).  The
 * tensor core's summation order is fixed, so repeated calls give identical
 * bits; each element is within the nm_spmv tolerance of the exact product.
 * Limits: rows < 2^31 and ceil(rows / 128) <= 65535; T < 2^31.  T == 0 or
 * rows == 0 is a no-op.  Y must not overlap any input.  No workspace: every
 * block multiplies whole rows of W.
 *
 * nm_spmm_prefill_ws -- the same product with a K split when it is faster:
 * when a matrix has too few 128-row tiles to fill the SMs (few rows, or few
 * tokens), the mask words of each row are cut into S slices (multiples of
 * four words) taken by different blocks.  Each writes its slice's fp32 sums
 * to the workspace ([S][T][rows] fp32), and a second kernel adds the S sums
 * in slice order and rounds once to fp16: deterministic, within the same
 * tolerance (fp32 sums of fp16 products, one rounding).
 *   workspace : device scratch, 16-byte aligned, of at least
 *       nm_spmm_prefill_workspace_bytes(rows, cols, T) bytes (0 when the plan
 *       for this shape on this device does not split); may be NULL then.  A
 *       short workspace -> NM_ERR_WORKSPACE; it must not overlap any argument.
 * nm_spmm_prefill_ex takes the plan explicitly: variant (< 0: chosen;
 * 0..nm_spmm_prefill_variant_count()-1: 512 tokens per block with 4 pipeline
 * stages, 256, 128, 64 tokens, and 512 tokens with 5 stages) and splits
 * (<= 0: chosen; 1: none; k <= 64: at most k slices -- the words are cut in
 * multiples of four, so fewer may result); the workspace it needs is
 * nm_spmm_prefill_workspace_bytes_ex(rows, cols, T, variant, splits).  The
 * chosen plan minimises a time model: waves of blocks x (a slice's stages x
 * each variant's measured time per stage + a block's fixed cost + its output
 * stores), plus the combine's launch and traffic when split; it considers at
 * most 8 slices and at most 256 MB of partial sums.  nm_spmm_prefill_plan
 * reports it.
 * ------------------------------------------------------------------------- */
int nm_spmm_prefill(const void *values, const uint32_t *masks, int64_t rows, int64_t cols,
                    const void *X, int64_t ldx, int64_t T, void *Y, int64_t ldy, void *stream);
size_t nm_spmm_prefill_workspace_bytes(int64_t rows, int64_t cols, int64_t T);
int nm_spmm_prefill_ws(const void *values, const uint32_t *masks, int64_t rows, int64_t cols,
                       const void *X, int64_t ldx, int64_t T, void *Y, int64_t ldy,
                       void *workspace, size_t workspace_bytes, void *stream);
size_t nm_spmm_prefill_workspace_bytes_ex(int64_t rows, int64_t cols, int64_t T, int variant,
                                          int splits);
int nm_spmm_prefill_ex(const void *values, const uint32_t *masks, int64_t rows, int64_t cols,
                       const void *X, int64_t ldx, int64_t T, void *Y, int64_t ldy, int variant,
                       int splits, void *workspace, size_t workspace_bytes, void *stream);
int nm_spmm_prefill_variant_count(void);
/* nm_spmm_prefill_plan -- the plan nm_spmm_prefill_ws takes for this shape on
 * a device with `sms` SMs (<= 0: the current device's count): the kernel
 * variant, the number of K slices (1: no split) and the tokens per block of
 * that variant.  Any output pointer may be NULL.  Host-only when sms > 0.
 * rows, T >= 1 and cols % 32 == 0, else NM_ERR_SHAPE. */
int nm_spmm_prefill_plan(int64_t rows, int64_t cols, int64_t T, int sms, int *variant,
                         int *slices, int *tile_tokens);

/* nm_wait_timeouts -- how many times a tensor-core kernel's bounded wait on
 * one of its own barriers gave up (each such wait ends after 2 s, after which
 * the kernel abandons its work, skips its stores and returns, rather than
 * hang).  The first wait that gives up also sets an abort flag: every other
 * pipeline wait then gives up at once (waits for the block's own copies in
 * flight still complete), and tensor-core blocks launched while the flag is
 * set return without doing anything, so their Y is left unwritten.  Zero in
 * every correct run; `reset` != 0 resets the count to zero and clears the
 * abort flag.  After a nonzero count, treat the outputs of the tensor-core
 * calls since the last reset as undefined.
 * Host-synchronous (reads a device counter); negative nm_status on error. */
int64_t nm_wait_timeouts(int reset);

/* nm_prefill_stall_selftest -- exercises the bounded-wait path of the
 * prefill kernel (self-test; no counterpart on the pages): launches it on the
 * given buffers (as for nm_spmm_prefill, 64-token variant) with its weight
 * producer disabled, so that no stage ever completes, and every wait limited
 * to wait_limit_us (1..2,000,000).  Each role's wait then runs out, is counted
 * in nm_wait_timeouts(), and the kernel returns without storing Y; the device
 * stays usable.  Asynchronous; NM_OK once launched. */
int nm_prefill_stall_selftest(const void *values, const uint32_t *masks, int64_t rows,
                              int64_t cols, const void *X, int64_t ldx, int64_t T, void *Y,
                              int64_t ldy, int64_t wait_limit_us, void *stream);

/* ---------------------------------------------------------------------------
 * nm_check_masks_noalloc -- the same count as nm_check_masks, without any
 * device allocation.  The paper has no counterpart to this entry point; it
 * exists for callers that must not allocate device memory while they run --
 * a serving process whose memory is all handed to its own caching allocator
 * or arena at start-up, or a latency-critical loop where a stream-ordered
 * allocation could stall on the memory pool.
 *   Scratch: a fixed array inside the library's device image (32 KB + 8 B),
 *   held by every GPU that loads the library until the process exits.
 *   Limit: rows * cols / 32 <= NM_CHECK_NOALLOC_MAX_WORDS mask words;
 *   larger inputs (including any whose product would overflow) return
 *   -NM_ERR_WORKSPACE without any CUDA call.
 *   The first call in a CUDA context looks up the array's device address in
 *   that context (cudaGetSymbolAddress, which also loads the module) and
 *   caches it under the context's unique id, so a context made after
 *   cudaDeviceReset gets a fresh lookup; make that first call before any
 *   stream capture.
 *   All calls share the array: calls that overlap on the GPU (different
 *   streams or host threads at the same time) race and must be serialised by
 *   the caller.  Each call writes every scratch slot it reads, so nothing
 *   carries over from one call to the next.
 *   Returns the number of words whose popcount is not 16, or a negative
 *   nm_status; host-synchronous (waits for the stream).
 * ------------------------------------------------------------------------- */
#define NM_CHECK_NOALLOC_MAX_WORDS ((int64_t)67108864) /* 4096 blocks x 16384 words */
int64_t nm_check_masks_noalloc(const uint32_t *masks, int64_t rows, int64_t cols, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* NM_SPMV_H */
