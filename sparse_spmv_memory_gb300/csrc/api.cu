// api.cu -- the extern "C" boundary: argument checks, launch plans, dispatch.
// Declarations and the contract of every entry point: include/nm_spmv.h.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include <atomic>

#include "../../include/nm_spmv.h"
#include "kernels.h"

namespace nmk {

// ---- per-device attributes, queried once ------------------------------------
struct DeviceInfo {
  int sms;
  int smem_optin;  // bytes of dynamic shared memory a block may opt into
};

static constexpr int kMaxDevices = 64;
static DeviceInfo g_info[kMaxDevices];
static std::atomic<int> g_info_ready[kMaxDevices];

static cudaError_t device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices && g_info_ready[dev].load(std::memory_order_acquire)) {
    *out = g_info[dev];
    return cudaSuccess;
  }
  DeviceInfo d{};
  e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices) {
    g_info[dev] = d;
    g_info_ready[dev].store(1, std::memory_order_release);
  }
  *out = d;
  return cudaSuccess;
}

cudaError_t ensure_max_smem(const void* func, int* done_flags, int max_devices) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < max_devices && __atomic_load_n(&done_flags[dev], __ATOMIC_ACQUIRE)) return cudaSuccess;
  DeviceInfo d;
  e = device_info(&d);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, d.smem_optin);
  if (e == cudaSuccess && dev < max_devices) __atomic_store_n(&done_flags[dev], 1, __ATOMIC_RELEASE);
  return e;
}

}  // namespace nmk

using namespace nmk;

namespace {

constexpr int64_t kMaxRows = (int64_t)1 << 31;
constexpr int64_t kMaxCols = (int64_t)1 << 31;  // words per row then fit an int
constexpr int kPrefillMaxSplits = 8;   // K slices the prefill plan considers
constexpr int kPrefillMaxSlices = 64;  // K slices a caller may ask for
constexpr int kMaxGrid24 = 65536;      // blocks an explicit 2:4 SpMM plan may ask for
constexpr int kDefaultVariant24 = 1;  // 20 warps x 1 unit, 4 accumulator chains

// nm_spmm24 indexes its 16-row x 128-column units in 32 bits.
bool spmm24_fits(int64_t rows, int64_t cols) {
  return (rows + 15) / 16 * (cols / 128) < ((int64_t)1 << 31);
}

// nm_spmm24's plan: variant, column slices (the fewest whose x fits a block's
// shared memory; cs units each, the last slice the rest) and a grid of whole
// slices (one block per SM by default, rounded down to a multiple of the
// slices; an explicit grid likewise).
struct Spmm24Plan {
  int variant, slices, cs, grid;
};

bool make_spmm24_plan(int64_t cols, int variant, int grid, const DeviceInfo& d, Spmm24Plan* pl) {
  const int units = (int)(cols / 128);
  int S = spmm24_slices(units, (size_t)d.smem_optin);
  if (S < 1) return false;
  const int cs = (units + S - 1) / S;
  S = (units + cs - 1) / cs;  // every slice non-empty
  if (grid <= 0) grid = d.sms;
  grid = grid / S * S;
  if (grid < S) grid = S;
  pl->variant = variant < 0 ? kDefaultVariant24 : variant;
  pl->slices = S;
  pl->cs = cs;
  pl->grid = grid;
  return true;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return na && nb && a0 < b0 + nb && b0 < a0 + na;
}

bool valid_pattern(int N, int M) {
  return (N == 2 && M == 4) || (N == 4 && M == 8) || (N == 8 && M == 16) || (N == 16 && M == 32);
}

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

int spmv_pitch(int64_t words) { return (int)round_up(words, 32); }

int64_t gemv_steps(int64_t cols) { return (cols + 511) / 512; }

// Measured on GB300 over the decode-layer shapes: the {20 warps, 3 steps in
// flight, fp16 x} variant streams large matrices fastest; below ~134M weight
// positions (where the launch's fixed start-up cost weighs more) the
// {24 warps, 2 steps, fp32 x} variant is ahead, and up to 4096x4096 (2^24)
// the {28 warps, 1 step, fp32 x} one.
int default_spmv_variant(int64_t rows = 0, int64_t cols = 0) {
  const int64_t n = rows * cols;
  return n >= ((int64_t)1 << 27) ? 1 : (n > ((int64_t)1 << 24) ? 0 : 6);
}

// The dense baseline's fastest variant on every decode-layer shape measured.
int default_gemv_variant() { return 0; }

// Builds the sparse launch plan; returns NM_OK or a status.
int make_spmv_plan(int64_t rows, int64_t cols, int variant, int grid, SpmvPlan* plan,
                   SpmvParams* p) {
  DeviceInfo d;
  if (device_info(&d) != cudaSuccess) return NM_ERR_CUDA;
  if (variant < 0) variant = default_spmv_variant(rows, cols);
  if (variant >= spmv_variant_count()) return NM_ERR_SHAPE;
  const int nw = spmv_variant_warps(variant);
  const int64_t words = cols / 32;
  const int pitch = spmv_pitch(words);
  const size_t smem = spmv_smem_bytes(pitch, nw);
  if (smem > (size_t)d.smem_optin) return NM_ERR_SHAPE;
  if (grid <= 0) grid = d.sms;  // one resident block per SM
  if (grid > rows) grid = (int)rows;
  plan->variant = variant;
  plan->grid = grid;
  plan->warps = nw;
  p->rows = rows;
  p->words = (int)words;
  p->steps = (int)((words + 31) / 32);
  p->pitch = pitch;
  return NM_OK;
}

int make_gemv_plan(int64_t rows, int64_t cols, int variant, int grid, GemvPlan* plan,
                   GemvParams* p) {
  DeviceInfo d;
  if (device_info(&d) != cudaSuccess) return NM_ERR_CUDA;
  if (variant < 0) variant = default_gemv_variant();
  if (variant >= gemv_variant_count()) return NM_ERR_SHAPE;
  const int nw = gemv_variant_warps(variant);
  const int64_t steps = gemv_steps(cols);
  if (gemv_smem_bytes((int)steps, nw) > (size_t)d.smem_optin) return NM_ERR_SHAPE;
  if (grid <= 0) grid = d.sms;
  if (grid > rows) grid = (int)rows;
  plan->variant = variant;
  plan->grid = grid;
  plan->warps = nw;
  p->rows = rows;
  p->cols = (int)cols;
  p->steps = (int)steps;
  return NM_OK;
}

// Sparse small-batch plan: padded batch, column slices so the x tile fits.
int make_spmm_plan(int64_t rows, int64_t cols, int batch, int variant, int grid, int slices,
                   SpmmPlan* plan, SpmmParams* p) {
  DeviceInfo d;
  if (device_info(&d) != cudaSuccess) return NM_ERR_CUDA;
  const int64_t words = cols / 32;
  const int64_t T = (words + 31) / 32;
  auto pitch_for = [&](int64_t S) { return (int)((T + S - 1) / S * 32); };
  if (variant < 0) {
    // measured on GB300 (8B/32B/70B layer shapes, whole-step kernel): 20
    // warps x 2 steps in flight with fp16 x slots when a whole row's x tile
    // fits (one column slice), 24 warps x 1 with the 12-byte slots of 5-6
    // tokens (0-2 % faster there); when the columns must be sliced, 16 warps
    // x 2 up to 6 tokens and 24 warps x 1 at 8 tokens (fewer registers per
    // thread for the slice walk; 2-6 % faster there).
    const int bp1 = spmm_padded_batch(batch, spmm_variant_xf(1));
    variant = bp1 == 6 ? 3 : 1;
    if (slices != 1 &&
        spmm_smem_bytes(pitch_for(1), spmm_variant_warps(variant), bp1, 0) >
            (size_t)d.smem_optin)
      variant = bp1 == 8 ? 3 : 0;
  }
  if (variant >= spmm_variant_count()) return NM_ERR_SHAPE;
  const int nw = spmm_variant_warps(variant);
  const int xf = spmm_variant_xf(variant);
  const int bp = spmm_padded_batch(batch, xf);
  if (slices <= 0) {
    int64_t S = 1;
    while (S < T && spmm_smem_bytes(pitch_for(S), nw, bp, xf) > (size_t)d.smem_optin) ++S;
    slices = (int)S;
  }
  if (slices > T || spmm_smem_bytes(pitch_for(slices), nw, bp, xf) > (size_t)d.smem_optin)
    return NM_ERR_SHAPE;
  if (grid <= 0) grid = d.sms;
  int64_t bps = grid / slices;
  if (bps < 1) bps = 1;
  if (bps > rows) bps = rows;
  plan->variant = variant;
  plan->grid = (int)(bps * slices);
  plan->bp = bp;
  plan->sms = d.sms;
  plan->warps = nw;
  p->rows = rows;
  p->words = (int)words;
  p->steps = (int)T;
  p->slices = slices;
  p->pitch = pitch_for(slices);
  p->batch = batch;
  return NM_OK;
}

size_t spmm_workspace_for(const SpmmParams& p) {
  return p.slices > 1 ? (size_t)p.slices * p.batch * p.rows * sizeof(float) : 0;
}

int check_spmv_args(const void* values, const uint32_t* masks, int64_t rows, int64_t cols,
                    const void* x, const void* y) {
  if (!values || !masks || !x || !y) return NM_ERR_NULL;
  if (rows < 0 || rows >= kMaxRows || cols <= 0 || cols >= kMaxCols ||
      cols % 32 != 0) return NM_ERR_SHAPE;
  if (!aligned(values, 32) || !aligned(masks, 4) || !aligned(x, 16) || !aligned(y, 2))
    return NM_ERR_ALIGN;
  const size_t yb = (size_t)rows * 2;
  if (overlap(y, yb, values, (size_t)rows * cols) || overlap(y, yb, masks, (size_t)rows * cols / 8) ||
      overlap(y, yb, x, (size_t)cols * 2))
    return NM_ERR_ALIAS;
  return NM_OK;
}

}  // namespace

extern "C" {

int64_t nm_spmv_max_cols(void);
size_t nm_spmm_workspace_bytes_ex(int64_t rows, int64_t cols, int batch, int variant, int slices);
int nm_spmm_ex(const void* values, const uint32_t* masks, int64_t rows, int64_t cols,
               const void* X, int64_t ldx, int batch, void* Y, int64_t ldy, void* workspace,
               size_t workspace_bytes, int variant, int grid, int slices, int flags, void* stream);
int nm_spmm_prefill_ws(const void* values, const uint32_t* masks, int64_t rows, int64_t cols,
                       const void* X, int64_t ldx, int64_t T, void* Y, int64_t ldy,
                       void* workspace, size_t workspace_bytes, void* stream);
size_t nm_spmm_prefill_workspace_bytes(int64_t rows, int64_t cols, int64_t T);

const char* nm_status_string(int status) {
  switch (status) {
    case NM_OK: return "NM_OK";
    case NM_ERR_NULL: return "NM_ERR_NULL: a required pointer is NULL";
    case NM_ERR_SHAPE: return "NM_ERR_SHAPE: unsupported shape (rows, cols % 32, ld, size limit)";
    case NM_ERR_PATTERN: return "NM_ERR_PATTERN: N:M must be 2:4, 4:8, 8:16 or 16:32";
    case NM_ERR_ALIGN: return "NM_ERR_ALIGN: misaligned pointer or leading dimension";
    case NM_ERR_WORKSPACE: return "NM_ERR_WORKSPACE: workspace missing or too small";
    case NM_ERR_CUDA: return "NM_ERR_CUDA: a CUDA call or kernel launch failed";
    case NM_ERR_ALIAS: return "NM_ERR_ALIAS: an output overlaps an input";
    default: return "unknown nm_status";
  }
}

size_t nm_values_bytes(int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 0 || cols % 32 != 0) return 0;
  return (size_t)rows * (size_t)(cols / 2) * 2;
}

size_t nm_masks_bytes(int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 0 || cols % 32 != 0) return 0;
  return (size_t)rows * (size_t)(cols / 32) * 4;
}

size_t nm_spmv_workspace_bytes(int64_t rows, int64_t cols) {
  if (rows <= 0 || rows >= kMaxRows || cols <= 0 || cols >= kMaxCols || cols % 32 != 0) return 0;
  const int64_t max_cols = nm_spmv_max_cols();
  if (max_cols < 0 || cols <= max_cols) return 0;  // the whole row's x tile fits
  // longer rows run as a one-token nm_spmm over column slices
  return nm_spmm_workspace_bytes_ex(rows, cols, 1, -1, 0);
}

int64_t nm_spmv_max_cols(void) {
  DeviceInfo d;
  if (device_info(&d) != cudaSuccess) return -NM_ERR_CUDA;
  int nw = 0;  // the most warps any default plan uses
  for (int64_t elems : {(int64_t)0, (int64_t)1 << 40}) {
    const int w = spmv_variant_warps(default_spmv_variant(elems, 1));
    nw = w > nw ? w : nw;
  }
  // largest multiple-of-32 pitch whose tile fits, times 32 columns per word
  int64_t pitch = ((int64_t)d.smem_optin / 4 - 6 * nw) / 34;
  pitch = pitch / 32 * 32;
  return pitch * 32;
}

int nm_pack(const void* W, int64_t rows, int64_t cols, int64_t ld, int N, int M, void* values,
            uint32_t* masks, void* stream) {
  if (!W || !values || !masks) return NM_ERR_NULL;
  if (rows < 0 || rows >= kMaxRows || cols <= 0 || cols >= kMaxCols ||
      cols % 32 != 0 || ld < cols) return NM_ERR_SHAPE;
  if (!valid_pattern(N, M)) return NM_ERR_PATTERN;
  if (!aligned(W, 2) || !aligned(values, 16) || !aligned(masks, 4)) return NM_ERR_ALIGN;
  const size_t wb = (size_t)((rows - 1) * ld + cols) * 2;
  if (rows && (overlap(values, (size_t)rows * cols, W, wb) ||
               overlap(masks, (size_t)rows * cols / 8, W, wb) ||
               overlap(values, (size_t)rows * cols, masks, (size_t)rows * cols / 8)))
    return NM_ERR_ALIAS;
  if (rows == 0) return NM_OK;
  cudaError_t e = launch_pack(static_cast<const __half*>(W), rows, cols, ld, M,
                              static_cast<__half*>(values), masks, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NM_OK : NM_ERR_CUDA;
}

int nm_unpack(const void* values, const uint32_t* masks, int64_t rows, int64_t cols, void* W_out,
              int64_t ld, void* stream) {
  if (!values || !masks || !W_out) return NM_ERR_NULL;
  if (rows < 0 || rows >= kMaxRows || cols <= 0 || cols >= kMaxCols ||
      cols % 32 != 0 || ld < cols) return NM_ERR_SHAPE;
  if (!aligned(values, 16) || !aligned(masks, 4) || !aligned(W_out, 2)) return NM_ERR_ALIGN;
  const size_t wb = (size_t)((rows - 1) * ld + cols) * 2;
  if (rows && (overlap(W_out, wb, values, (size_t)rows * cols) ||
               overlap(W_out, wb, masks, (size_t)rows * cols / 8)))
    return NM_ERR_ALIAS;
  if (rows == 0) return NM_OK;
  cudaError_t e = launch_unpack(static_cast<const __half*>(values), masks, rows, cols,
                                static_cast<__half*>(W_out), ld, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NM_OK : NM_ERR_CUDA;
}

int nm_spmv_ex(const void* values, const uint32_t* masks, int64_t rows, int64_t cols,
               const void* x, void* y, void* workspace, size_t workspace_bytes, int variant,
               int grid, int flags, void* stream) {
  int st = check_spmv_args(values, masks, rows, cols, x, y);
  if (st != NM_OK) return st;
  if (rows == 0) return NM_OK;
  const int64_t max_cols = nm_spmv_max_cols();
  if (max_cols > 0 && cols > max_cols && variant < 0) {
    // a row's x tile does not fit one block: one-token SpMM over column slices,
    // partial sums through the workspace (nm_spmv_workspace_bytes > 0)
    return nm_spmm_ex(values, masks, rows, cols, x, cols, 1, y, rows, workspace, workspace_bytes,
                      -1, grid, 0, flags, stream);
  }
  // single-block rows need no workspace; an explicit plan whose x tile does
  // not fit is refused by make_spmv_plan (NM_ERR_SHAPE)
  SpmvPlan plan;
  SpmvParams p;
  st = make_spmv_plan(rows, cols, variant, grid, &plan, &p);
  if (st != NM_OK) return st;
  p.values = static_cast<const uint32_t*>(values);
  p.masks = masks;
  p.x = static_cast<const __half*>(x);
  p.y = static_cast<__half*>(y);
  p.early_weights = (flags & NM_FLAG_WEIGHTS_CONST) ? 1 : 0;
  cudaError_t e = launch_spmv(p, plan, flags, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NM_OK : NM_ERR_CUDA;
}

int nm_spmv_swiglu_ex(const void* values, const uint32_t* masks, int64_t rows, int64_t cols,
                      const void* x, void* h, int variant, int grid, int flags, void* stream) {
  if (!values || !masks || !x || !h) return NM_ERR_NULL;
  if (rows < 0 || rows >= kMaxRows || rows % 2 != 0 || cols <= 0 || cols >= kMaxCols ||
      cols % 32 != 0)
    return NM_ERR_SHAPE;
  if (!aligned(values, 32) || !aligned(masks, 4) || !aligned(x, 16) || !aligned(h, 2))
    return NM_ERR_ALIGN;
  const size_t hb = (size_t)rows;  // rows/2 fp16
  if (overlap(h, hb, values, (size_t)rows * cols) || overlap(h, hb, masks, (size_t)rows * cols / 8) ||
      overlap(h, hb, x, (size_t)cols * 2))
    return NM_ERR_ALIAS;
  if (rows == 0) return NM_OK;
  SpmvPlan plan;
  SpmvParams p;
  int st = make_spmv_plan(rows, cols, variant, grid, &plan, &p);
  if (st != NM_OK) return st;
  // blocks own whole (gate, up) pairs; the rows' fp32 sums stay in shared memory
  if (plan.grid > rows / 2) plan.grid = (int)(rows / 2);
  DeviceInfo d;
  if (device_info(&d) != cudaSuccess) return NM_ERR_CUDA;
  const int64_t block_rows_max = 2 * ((rows / 2 + plan.grid - 1) / plan.grid);
  if (spmv_smem_bytes(p.pitch, plan.warps) + (size_t)block_rows_max * 4 > (size_t)d.smem_optin)
    return NM_ERR_SHAPE;
  p.values = static_cast<const uint32_t*>(values);
  p.masks = masks;
  p.x = static_cast<const __half*>(x);
  p.y = static_cast<__half*>(h);
  p.early_weights = (flags & NM_FLAG_WEIGHTS_CONST) ? 1 : 0;
  cudaError_t e = launch_spmv(p, plan, flags, static_cast<cudaStream_t>(stream), 1);
  return e == cudaSuccess ? NM_OK : NM_ERR_CUDA;
}

int nm_spmv_swiglu(const void* values, const uint32_t* masks, int64_t rows, int64_t cols,
                   const void* x, void* h, void* stream) {
  return nm_spmv_swiglu_ex(values, masks, rows, cols, x, h, -1, 0, NM_FLAG_PDL, stream);
}

int nm_spmv(const void* values, const uint32_t* masks, int64_t rows, int64_t cols, const void* x,
            void* y, void* workspace, size_t workspace_bytes, void* stream) {
  return nm_spmv_ex(values, masks, rows, cols, x, y, workspace, workspace_bytes, -1, 0,
                    NM_FLAG_PDL, stream);
}

int nm_spmv_plan(int64_t rows, int64_t cols, int* variant, int* grid, int* warps) {
  if (rows <= 0 || rows >= kMaxRows || cols <= 0 || cols >= kMaxCols ||
      cols % 32 != 0) return NM_ERR_SHAPE;
  SpmvPlan plan;
  SpmvParams p;
  int st = make_spmv_plan(rows, cols, -1, 0, &plan, &p);
  if (st != NM_OK) return st;
  if (variant) *variant = plan.variant;
  if (grid) *grid = plan.grid;
  if (warps) *warps = plan.warps;
  return NM_OK;
}

int nm_spmv_variant_count(void) { return spmv_variant_count(); }

int dense_gemv_variant_count(void) { return gemv_variant_count(); }

int dense_gemv_ex(const void* W, int64_t rows, int64_t cols, int64_t ld, const void* x, void* y,
                  int variant, int grid, int flags, void* stream) {
  if (!W || !x || !y) return NM_ERR_NULL;
  if (rows < 0 || rows >= kMaxRows || cols <= 0 || cols >= kMaxCols ||
      cols % 8 != 0 || ld < cols) return NM_ERR_SHAPE;
  if (!aligned(W, 16) || ld % 8 != 0 || !aligned(x, 16) || !aligned(y, 2)) return NM_ERR_ALIGN;
  const size_t yb = (size_t)rows * 2;
  if (rows && (overlap(y, yb, W, (size_t)((rows - 1) * ld + cols) * 2) ||
               overlap(y, yb, x, (size_t)cols * 2)))
    return NM_ERR_ALIAS;
  if (rows == 0) return NM_OK;
  GemvPlan plan;
  GemvParams p;
  int st = make_gemv_plan(rows, cols, variant, grid, &plan, &p);
  if (st != NM_OK) return st;
  p.W = static_cast<const __half*>(W);
  p.x = static_cast<const __half*>(x);
  p.y = static_cast<__half*>(y);
  p.ld = ld;
  p.early_weights = (flags & NM_FLAG_WEIGHTS_CONST) ? 1 : 0;
  cudaError_t e = launch_gemv(p, plan, flags, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NM_OK : NM_ERR_CUDA;
}

int dense_gemv(const void* W, int64_t rows, int64_t cols, int64_t ld, const void* x, void* y,
               void* stream) {
  return dense_gemv_ex(W, rows, cols, ld, x, y, -1, 0, NM_FLAG_PDL, stream);
}

size_t nm_spmm_workspace_bytes_ex(int64_t rows, int64_t cols, int batch, int variant,
                                  int slices) {
  if (rows <= 0 || rows >= kMaxRows || cols <= 0 || cols >= kMaxCols ||
      cols % 32 != 0 || batch < 1 || batch > 8)
    return 0;
  SpmmPlan plan;
  SpmmParams p;
  if (make_spmm_plan(rows, cols, batch, variant, 0, slices, &plan, &p) != NM_OK) return 0;
  return spmm_workspace_for(p);
}

size_t nm_spmm_workspace_bytes(int64_t rows, int64_t cols, int batch) {
  if (batch > 8) return nm_spmm_prefill_workspace_bytes(rows, cols, batch);
  return nm_spmm_workspace_bytes_ex(rows, cols, batch, -1, 0);
}

int nm_spmm_variant_count(void) { return spmm_variant_count(); }

int nm_spmm_ex(const void* values, const uint32_t* masks, int64_t rows, int64_t cols,
               const void* X, int64_t ldx, int batch, void* Y, int64_t ldy, void* workspace,
               size_t workspace_bytes, int variant, int grid, int slices, int flags,
               void* stream) {
  if (!values || !masks || !X || !Y) return NM_ERR_NULL;
  if (rows < 0 || rows >= kMaxRows || cols <= 0 || cols >= kMaxCols ||
      cols % 32 != 0 || batch < 1 || batch > 8 ||
      ldx < cols || ldy < rows)
    return NM_ERR_SHAPE;
  if (!aligned(values, 32) || !aligned(masks, 4) || !aligned(X, 16) || ldx % 8 != 0 ||
      !aligned(Y, 2) || (workspace && !aligned(workspace, 16)))
    return NM_ERR_ALIGN;
  if (rows == 0) return NM_OK;
  const size_t yb = (size_t)((batch - 1) * ldy + rows) * 2;
  const size_t xb = (size_t)((batch - 1) * ldx + cols) * 2;
  if (overlap(Y, yb, values, (size_t)rows * cols) || overlap(Y, yb, masks, (size_t)rows * cols / 8) ||
      overlap(Y, yb, X, xb) || overlap(Y, yb, workspace, workspace_bytes))
    return NM_ERR_ALIAS;
  SpmmPlan plan;
  SpmmParams p;
  int st = make_spmm_plan(rows, cols, batch, variant, grid, slices, &plan, &p);
  if (st != NM_OK) return st;
  const size_t need = spmm_workspace_for(p);
  if (need > 0 && (!workspace || workspace_bytes < need)) return NM_ERR_WORKSPACE;
  if (need > 0 && (overlap(workspace, need, values, (size_t)rows * cols) ||
                   overlap(workspace, need, masks, (size_t)rows * cols / 8) ||
                   overlap(workspace, need, X, xb)))
    return NM_ERR_ALIAS;
  p.values = static_cast<const uint32_t*>(values);
  p.masks = masks;
  p.X = static_cast<const __half*>(X);
  p.ldx = ldx;
  p.Y = static_cast<__half*>(Y);
  p.ldy = ldy;
  p.partial = static_cast<float*>(workspace);
  p.early_weights = (flags & NM_FLAG_WEIGHTS_CONST) ? 1 : 0;
  cudaError_t e = launch_spmm(p, plan, flags, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NM_OK : NM_ERR_CUDA;
}

int nm_spmm(const void* values, const uint32_t* masks, int64_t rows, int64_t cols, const void* X,
            int64_t ldx, int batch, void* Y, int64_t ldy, void* workspace, size_t workspace_bytes,
            void* stream) {
  if (batch > 8)  // beyond the CUDA-core kernel's batch: the tensor-core path
    return nm_spmm_prefill_ws(values, masks, rows, cols, X, ldx, batch, Y, ldy, workspace,
                              workspace_bytes, stream);
  return nm_spmm_ex(values, masks, rows, cols, X, ldx, batch, Y, ldy, workspace, workspace_bytes,
                    -1, 0, 0, NM_FLAG_PDL, stream);
}

int nm_spmm24_variant_count(void) { return spmm24_variant_count(); }

size_t nm_spmm24_workspace_bytes_ex(int64_t rows, int64_t cols, int batch, int variant,
                                    int grid) {
  if (rows <= 0 || rows >= kMaxRows || cols <= 0 || cols >= kMaxCols || cols % 128 != 0 ||
      batch < 1 || batch > 8 || variant >= spmm24_variant_count() || grid > kMaxGrid24 ||
      !spmm24_fits(rows, cols))
    return 0;
  DeviceInfo d;
  if (device_info(&d) != cudaSuccess) return 0;
  Spmm24Plan pl;
  if (!make_spmm24_plan(cols, variant, grid, d, &pl)) return 0;
  return spmm24_workspace_bytes(pl.grid, (rows + 15) / 16, pl.slices);
}

size_t nm_spmm24_workspace_bytes(int64_t rows, int64_t cols, int batch) {
  return nm_spmm24_workspace_bytes_ex(rows, cols, batch, -1, 0);
}

int nm_spmm24_ex(const void* values, const uint32_t* masks, int64_t rows, int64_t cols,
                 const void* X, int64_t ldx, int batch, void* Y, int64_t ldy, void* workspace,
                 size_t workspace_bytes, int variant, int grid, int flags, void* stream) {
  if (!values || !masks || !X || !Y) return NM_ERR_NULL;
  if (rows < 0 || rows >= kMaxRows || cols <= 0 || cols >= kMaxCols || cols % 128 != 0 ||
      batch < 1 || batch > 8 || ldx < cols || ldy < rows || variant >= spmm24_variant_count() ||
      grid > kMaxGrid24 || !spmm24_fits(rows, cols))
    return NM_ERR_SHAPE;
  if (!aligned(values, 32) || !aligned(masks, 4) || !aligned(X, 16) || ldx % 8 != 0 ||
      !aligned(Y, 2) || (workspace && !aligned(workspace, 16)))
    return NM_ERR_ALIGN;
  if (rows == 0) return NM_OK;
  const size_t yb = (size_t)((batch - 1) * ldy + rows) * 2;
  const size_t xb = (size_t)((batch - 1) * ldx + cols) * 2;
  if (overlap(Y, yb, values, (size_t)rows * cols) ||
      overlap(Y, yb, masks, (size_t)rows * cols / 8) || overlap(Y, yb, X, xb) ||
      overlap(Y, yb, workspace, workspace_bytes))
    return NM_ERR_ALIAS;
  DeviceInfo d;
  if (device_info(&d) != cudaSuccess) return NM_ERR_CUDA;
  Spmm24Plan pl;
  if (!make_spmm24_plan(cols, variant, grid, d, &pl)) return NM_ERR_SHAPE;
  const int64_t panels = (rows + 15) / 16;
  const size_t need = spmm24_workspace_bytes(pl.grid, panels, pl.slices);
  if (!workspace || workspace_bytes < need) return NM_ERR_WORKSPACE;
  if (overlap(workspace, need, values, (size_t)rows * cols) ||
      overlap(workspace, need, masks, (size_t)rows * cols / 8) || overlap(workspace, need, X, xb))
    return NM_ERR_ALIAS;
  Spmm24Params p;
  p.values = static_cast<const uint32_t*>(values);
  p.masks = masks;
  p.X = static_cast<const __half*>(X);
  p.ldx = ldx;
  p.Y = static_cast<__half*>(Y);
  p.ldy = ldy;
  p.part = static_cast<float4*>(workspace);
  p.part_sp = p.part + (size_t)pl.grid * 64;
  p.cnt = reinterpret_cast<int*>(p.part_sp + (pl.slices > 1 ? (size_t)pl.slices * panels * 32 : 0));
  p.rows = rows;
  p.panels = panels;
  p.words = (int)(cols / 32);
  p.units = p.words / 4;
  p.slices = pl.slices;
  p.cs = pl.cs;
  p.batch = batch;
  p.early_weights = (flags & NM_FLAG_WEIGHTS_CONST) ? 1 : 0;
  p.y_vec = (aligned(Y, 8) && ldy % 4 == 0) ? 1 : 0;
  cudaError_t e = launch_spmm24(p, pl.variant, pl.grid, flags, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NM_OK : NM_ERR_CUDA;
}

int nm_spmm24(const void* values, const uint32_t* masks, int64_t rows, int64_t cols,
              const void* X, int64_t ldx, int batch, void* Y, int64_t ldy, void* workspace,
              size_t workspace_bytes, void* stream) {
  return nm_spmm24_ex(values, masks, rows, cols, X, ldx, batch, Y, ldy, workspace,
                      workspace_bytes, -1, 0, NM_FLAG_PDL, stream);
}

int nm_spmm_prefill_variant_count(void) { return spmm_tc_variant_count(); }

// The prefill plan (variant, K slices) for a call; variant < 0 and splits
// <= 0 ask for the modelled choice.
static int prefill_plan(int64_t rows, int64_t cols, int64_t T, int variant, int splits,
                        int* v_out, int* z_out) {
  const int words = (int)(cols / 32);
  if (variant >= 0 && splits >= 1) {
    *v_out = variant;
    *z_out = splits;
    return NM_OK;
  }
  DeviceInfo d;
  if (device_info(&d) != cudaSuccess) return NM_ERR_CUDA;
  spmm_tc_default_plan(rows, words, T, d.sms, variant, splits, kPrefillMaxSplits, v_out, z_out);
  return NM_OK;
}

static bool prefill_shape_ok(int64_t rows, int64_t cols, int64_t T) {
  return rows >= 0 && rows < kMaxRows && (rows + 127) / 128 <= 65535 && cols > 0 &&
         cols < kMaxCols && cols % 32 == 0 && T >= 0 && T < kMaxRows;
}

size_t nm_spmm_prefill_workspace_bytes_ex(int64_t rows, int64_t cols, int64_t T, int variant,
                                          int splits) {
  if (!prefill_shape_ok(rows, cols, T) || rows == 0 || T == 0 ||
      variant >= spmm_tc_variant_count() || splits > kPrefillMaxSlices)
    return 0;
  int v, z;
  if (prefill_plan(rows, cols, T, variant, splits, &v, &z) != NM_OK) return 0;
  return spmm_tc_workspace_bytes(rows, (int)(cols / 32), T, z);
}

size_t nm_spmm_prefill_workspace_bytes(int64_t rows, int64_t cols, int64_t T) {
  return nm_spmm_prefill_workspace_bytes_ex(rows, cols, T, -1, 0);
}

int nm_spmm_prefill_plan(int64_t rows, int64_t cols, int64_t T, int sms, int* variant,
                         int* slices, int* tile_tokens) {
  if (!prefill_shape_ok(rows, cols, T) || rows == 0 || T == 0) return NM_ERR_SHAPE;
  if (sms <= 0) {
    DeviceInfo d;
    if (device_info(&d) != cudaSuccess) return NM_ERR_CUDA;
    sms = d.sms;
  }
  const int words = (int)(cols / 32);
  int v, z;
  spmm_tc_default_plan(rows, words, T, sms, -1, 0, kPrefillMaxSplits, &v, &z);
  if (variant) *variant = v;
  if (slices) *slices = spmm_tc_slices(words, z);
  if (tile_tokens) *tile_tokens = spmm_tc_block_tokens(v);
  return NM_OK;
}

int nm_spmm_prefill_ex(const void* values, const uint32_t* masks, int64_t rows, int64_t cols,
                       const void* X, int64_t ldx, int64_t T, void* Y, int64_t ldy, int variant,
                       int splits, void* workspace, size_t workspace_bytes, void* stream) {
  if (!values || !masks || !X || !Y) return NM_ERR_NULL;
  if (!prefill_shape_ok(rows, cols, T) || ldx < cols || ldy < rows)
    return NM_ERR_SHAPE;
  if (variant >= spmm_tc_variant_count() || splits > kPrefillMaxSlices) return NM_ERR_SHAPE;
  if (!aligned(values, 32) || !aligned(masks, 4) || !aligned(X, 16) || ldx % 8 != 0 ||
      !aligned(Y, 2) || (workspace && !aligned(workspace, 16)))
    return NM_ERR_ALIGN;
  if (rows == 0 || T == 0) return NM_OK;
  const size_t yb = (size_t)((T - 1) * ldy + rows) * 2;
  const size_t xb = (size_t)((T - 1) * ldx + cols) * 2;
  if (overlap(Y, yb, values, (size_t)rows * cols) || overlap(Y, yb, masks, (size_t)rows * cols / 8) ||
      overlap(Y, yb, X, xb))
    return NM_ERR_ALIAS;
  int v, z;
  const int st = prefill_plan(rows, cols, T, variant, splits, &v, &z);
  if (st != NM_OK) return st;
  const int words = (int)(cols / 32);
  const size_t need = spmm_tc_workspace_bytes(rows, words, T, z);
  if (need > 0 && (!workspace || workspace_bytes < need)) return NM_ERR_WORKSPACE;
  if (need > 0 && (overlap(workspace, need, values, (size_t)rows * cols) ||
                   overlap(workspace, need, masks, (size_t)rows * cols / 8) ||
                   overlap(workspace, need, X, xb) || overlap(workspace, need, Y, yb)))
    return NM_ERR_ALIAS;
  SpmmTcParams p;
  p.values = values;
  p.masks = masks;
  p.X = X;
  p.ldx = ldx;
  p.Y = static_cast<__half*>(Y);
  p.ldy = ldy;
  p.rows = rows;
  p.words = words;
  p.T = T;
  p.slices = spmm_tc_slices(words, z);
  p.wslice = spmm_tc_slice_words(words, z);
  p.part = static_cast<float*>(workspace);
  cudaError_t e = launch_spmm_tc(p, v, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NM_OK : NM_ERR_CUDA;
}

int nm_spmm_prefill_ws(const void* values, const uint32_t* masks, int64_t rows, int64_t cols,
                       const void* X, int64_t ldx, int64_t T, void* Y, int64_t ldy,
                       void* workspace, size_t workspace_bytes, void* stream) {
  return nm_spmm_prefill_ex(values, masks, rows, cols, X, ldx, T, Y, ldy, -1, 0, workspace,
                            workspace_bytes, stream);
}

int nm_spmm_prefill(const void* values, const uint32_t* masks, int64_t rows, int64_t cols,
                    const void* X, int64_t ldx, int64_t T, void* Y, int64_t ldy, void* stream) {
  return nm_spmm_prefill_ex(values, masks, rows, cols, X, ldx, T, Y, ldy, -1, 1, nullptr, 0,
                            stream);
}

int nm_prefill_stall_selftest(const void* values, const uint32_t* masks, int64_t rows,
                              int64_t cols, const void* X, int64_t ldx, int64_t T, void* Y,
                              int64_t ldy, int64_t wait_limit_us, void* stream) {
  if (!values || !masks || !X || !Y) return NM_ERR_NULL;
  if (rows <= 0 || rows >= kMaxRows || (rows + 127) / 128 > 65535 || cols <= 0 ||
      cols >= kMaxCols || cols % 32 != 0 || T <= 0 || T >= kMaxRows || ldx < cols ||
      ldy < rows || wait_limit_us <= 0 || wait_limit_us > 2000000)
    return NM_ERR_SHAPE;
  if (!aligned(values, 32) || !aligned(masks, 4) || !aligned(X, 16) || ldx % 8 != 0 ||
      !aligned(Y, 2))
    return NM_ERR_ALIGN;
  SpmmTcParams p;
  p.values = values;
  p.masks = masks;
  p.X = X;
  p.ldx = ldx;
  p.Y = static_cast<__half*>(Y);
  p.ldy = ldy;
  p.rows = rows;
  p.words = (int)(cols / 32);
  p.T = T;
  p.wait_limit_ns = (uint64_t)wait_limit_us * 1000u;
  p.stall_weights = 1;
  cudaError_t e = launch_spmm_tc(p, 3, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NM_OK : NM_ERR_CUDA;
}

int64_t nm_wait_timeouts(int reset) {
  unsigned long long n = 0;
  return read_wait_timeouts(&n, reset) == cudaSuccess ? (int64_t)n : -NM_ERR_CUDA;
}

int64_t nm_check_masks(const uint32_t* masks, int64_t rows, int64_t cols, void* stream) {
  if (!masks) return -NM_ERR_NULL;
  // the same row bound as the other entry points, and a column bound, so that
  // rows * cols / 32 cannot wrap
  if (rows < 0 || rows >= kMaxRows || cols <= 0 || cols >= kMaxCols || cols % 32 != 0)
    return -NM_ERR_SHAPE;
  if (!aligned(masks, 4)) return -NM_ERR_ALIGN;
  if (rows == 0) return 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned long long* d_count = nullptr;
  unsigned long long h_count = 0;
  if (cudaMallocAsync(reinterpret_cast<void**>(&d_count), sizeof(*d_count), s) != cudaSuccess)
    return -NM_ERR_CUDA;
  cudaError_t e = cudaMemsetAsync(d_count, 0, sizeof(*d_count), s);
  if (e == cudaSuccess) e = launch_check_masks(masks, rows * (cols / 32), d_count, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(&h_count, d_count, sizeof(h_count), cudaMemcpyDeviceToHost, s);
  cudaError_t ef = cudaFreeAsync(d_count, s);
  if (e == cudaSuccess) e = ef;
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? (int64_t)h_count : -NM_ERR_CUDA;
}

}  // extern "C"
