// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernels.  Not part of the public ABI.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nmk {

// ---- sparse ----------------------------------------------------------------
struct SpmvParams {
  const uint32_t* values;  // fp16 pairs, [rows][words*8] uint32
  const uint32_t* masks;   // [rows][words]
  const __half* x;         // [words*32]
  __half* y;               // [rows]
  int64_t rows;
  int words;  // cols / 32
  int steps;  // ceil(words / 32): warp-steps per row
  int pitch;  // floats per row of the transposed x tile (multiple of 32, >= words)
  int early_weights;  // 1: load the first weights before waiting on the previous kernel
  int64_t rows_q = 0;  // set by the launcher: rows (or row pairs) per block ...
  int rows_r = 0;      // ... and how many blocks take one more
};

struct SpmvPlan {
  int variant;  // kernel template instance (warps per block, steps in flight)
  int grid;     // blocks
  int warps;    // warps per block of that variant
};

int spmv_variant_warps(int variant);
int spmv_variant_count();
size_t spmv_smem_bytes(int pitch, int nw);
// epilogue 0: y = W x; 1: rows are interleaved (gate, up) pairs and y receives
// h = silu(gate) * up, rows/2 values.
cudaError_t launch_spmv(const SpmvParams& p, const SpmvPlan& plan, int flags,
                        cudaStream_t stream, int epilogue = 0);

// ---- dense -----------------------------------------------------------------
struct GemvParams {
  const __half* W;  // [rows][ld]
  const __half* x;  // [cols]
  __half* y;        // [rows]
  int64_t rows;
  int64_t ld;
  int cols;
  int steps;  // ceil(cols / 512)
  int early_weights;
  int64_t rows_q = 0;  // set by the launcher: rows per block, blocks with one more
  int rows_r = 0;
};

struct GemvPlan {
  int variant;
  int grid;
  int warps;
};

int gemv_variant_warps(int variant);
int gemv_variant_count();
size_t gemv_smem_bytes(int steps, int nw);
cudaError_t launch_gemv(const GemvParams& p, const GemvPlan& plan, int flags,
                        cudaStream_t stream);

// ---- small-batch sparse ------------------------------------------------------
struct SpmmParams {
  const uint32_t* values;
  const uint32_t* masks;
  const __half* X;  // [batch][ldx]
  int64_t ldx;
  __half* Y;        // [batch][ldy]
  int64_t ldy;
  float* partial;   // [slices][batch][rows] fp32 when slices > 1
  int64_t rows;
  int words;   // cols / 32
  int steps;   // ceil(words / 32): warp-steps per row
  int slices;  // column slices
  int pitch;   // x-tile slots per row (>= 32 * steps of the widest slice)
  int batch;   // 1..8
  int early_weights;
  int64_t rows_q = 0;  // set by the launcher: rows per block of a slice, blocks with one more
  int rows_r = 0;
  int bps = 1;         // blocks per column slice
  int steps_q = 0;     // steps per slice, and how many slices take one more
  int steps_r = 0;
};

struct SpmmPlan {
  int variant;
  int grid;
  int bp;    // padded batch: 2, 4 or 8
  int sms;
  int warps;
};

int spmm_variant_count();
int spmm_variant_warps(int variant);
int spmm_padded_batch(int batch, int xf);
int spmm_variant_xf(int variant);
size_t spmm_smem_bytes(int pitch, int nw, int bp, int xf);
// One x-slot width (2, 4, 6 or 8 tokens), any variant: explicitly instantiated
// in spmm_b<bp>.cu.
template <int BP>
cudaError_t launch_spmm_variant(const SpmmParams& p, int variant, int grid, int flags,
                                cudaStream_t stream);
cudaError_t launch_spmm(const SpmmParams& p, const SpmmPlan& plan, int flags,
                        cudaStream_t stream);

// ---- small batches of a 2:4 matrix on the tensor cores (spmm24.cu) ----------
struct Spmm24Params {
  const uint32_t* values;
  const uint32_t* masks;
  const __half* X;  // [batch][ldx]
  int64_t ldx;
  __half* Y;        // [batch][ldy]
  int64_t ldy;
  float4* part;     // workspace: [blocks][2][32 lanes] fp32 partials of panels cut by blocks
  float4* part_sp;  // workspace (slices > 1): [slices][panels][32 lanes] whole slice-panels
  int* cnt;         // workspace: [panels] units counted so far of each cut panel
  int64_t rows;
  int64_t panels;   // ceil(rows / 16)
  int words;        // cols / 32, a multiple of 4
  int units;        // words / 4: 128-column units per panel
  int slices;       // column slices (x of a slice fits a block's shared memory)
  int cs;           // units per slice (the last slice may have fewer)
  int batch;        // 1..8
  int early_weights;
  int y_vec;        // Y 8-byte aligned and ldy % 4 == 0: 8-byte stores of 4 rows
  int bps = 0;      // set by the launcher: blocks per slice, and per slice
  int64_t bq = 0;   // panels * cs = bq * bps + br (bq_last, br_last: the last slice)
  int br = 0;
  int64_t bq_last = 0;
  int br_last = 0;
};

int spmm24_variant_count();
int spmm24_variant_warps(int variant);
int spmm24_slices(int units, size_t smem_optin);
size_t spmm24_workspace_bytes(int grid, int64_t panels, int slices);
cudaError_t launch_spmm24(const Spmm24Params& p, int variant, int grid, int flags,
                          cudaStream_t stream);

// ---- prefill-sized batches on the tensor cores -------------------------------
struct SpmmTcParams {
  const void* values;       // fp16 [rows][words*16], 16-byte aligned
  const uint32_t* masks;    // [rows][words]
  const void* X;            // fp16 [T][ldx], 16-byte aligned, ldx % 8 == 0
  int64_t ldx;
  __half* Y;                // fp16 [T][ldy]
  int64_t ldy;
  int64_t rows;
  int words;                // cols / 32
  int64_t T;                // tokens
  int slices = 1;           // K slices (> 1: fp32 partials in part, then a combine)
  int wslice = 0;           // mask words per slice (spmm_tc_slice_words)
  float* part = nullptr;    // fp32 [slices][T][rows] when slices > 1
  uint64_t wait_limit_ns = 0;  // bound of every in-kernel wait (0: the default)
  int stall_weights = 0;       // self-test: the weight producer issues nothing
};

int spmm_tc_variant_count();
int spmm_tc_default_variant(int64_t rows, int64_t T, int sms);
int spmm_tc_slice_words(int words, int splits);
int spmm_tc_slices(int words, int splits);
size_t spmm_tc_workspace_bytes(int64_t rows, int words, int64_t T, int splits);
void spmm_tc_default_plan(int64_t rows, int words, int64_t T, int sms, int variant, int splits,
                          int max_splits, int* variant_out, int* splits_out);
int spmm_tc_block_tokens(int variant);
cudaError_t launch_spmm_tc(const SpmmTcParams& p, int variant, cudaStream_t stream);
// Number of bounded mbarrier waits that gave up since the last reset.
cudaError_t read_wait_timeouts(unsigned long long* count, int reset);

// ---- format ----------------------------------------------------------------
cudaError_t launch_pack(const __half* W, int64_t rows, int64_t cols, int64_t ld, int M,
                        __half* values, uint32_t* masks, cudaStream_t stream);
cudaError_t launch_unpack(const __half* values, const uint32_t* masks, int64_t rows,
                          int64_t cols, __half* W, int64_t ld, cudaStream_t stream);
cudaError_t launch_check_masks(const uint32_t* masks, int64_t n_words,
                               unsigned long long* d_count, cudaStream_t stream);

// Launch flags (same values as NM_FLAG_* in nm_spmv.h).
constexpr int kFlagPdl = 1;

// Launch `kernel` with the programmatic-stream-serialization attribute when
// flags ask for it (the kernel may then start while the previous kernel on the
// stream finishes; it waits for it with griddepcontrol.wait).
template <typename Kernel, typename... Args>
inline cudaError_t launch_kernel(Kernel kernel, int grid, int block, size_t smem,
                                 cudaStream_t stream, int flags, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (flags & kFlagPdl) ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Sets the dynamic shared memory limit of `func` to the device maximum once
// per device.
cudaError_t ensure_max_smem(const void* func, int* done_flags, int max_devices);

}  // namespace nmk
