// spmm.cu -- small-batch N:M bitmask SpMM, Y = W X for 1..8 tokens (sm_103a):
// the launch dispatch, the column-slice combine and the plan's size
// queries.  The kernels and their design are in spmm_kernels.cuh, compiled
// once per x-slot width (spmm_b2.cu, spmm_b4.cu, spmm_b6.cu, spmm_b8.cu).
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device.cuh"
#include "kernels.h"
#include "spmm_variants.h"

namespace nmk {

// Y[j][r] = sum over slices s (in order) of partial[s][j][r], rounded to fp16.
__global__ void __launch_bounds__(256) spmm_combine_kernel(const float* __restrict__ partial,
                                                           int slices, int batch, int64_t rows,
                                                           __half* __restrict__ Y, int64_t ldy) {
  pdl_launch_dependents();
  pdl_wait_previous();
  for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < rows;
       r += (int64_t)gridDim.x * blockDim.x) {
    for (int j = 0; j < batch; ++j) {
      float s = 0.f;
      for (int k = 0; k < slices; ++k) s += partial[((int64_t)k * batch + j) * rows + r];
      Y[j * ldy + r] = __float2half_rn(s);
    }
  }
}

size_t spmm_smem_bytes(int pitch, int nw, int bp, int xf) {
  return (size_t)34 * pitch * bp * ((xf == 1 || xf == 2) ? 4 : 2) +
         2 * (size_t)nw * bp * sizeof(float) +
         4 * (size_t)nw * sizeof(int);
}

// Tokens per x slot: 2, 4, 8, and 6 for 5-6 tokens with fp16 slots (12-byte
// slots: three 4-byte gathers per nonzero, 3 shared-memory wavefronts per
// warp instead of the 4 of a 16-byte slot; the 8-token kernel is bound by
// those wavefronts).
int spmm_padded_batch(int batch, int xf) {
  if (batch <= 2) return 2;
  if (batch <= 4) return 4;
  return (batch <= 6 && xf == 0) ? 6 : 8;
}

int spmm_variant_count() { return kSpmmVariantCount; }

int spmm_variant_warps(int variant) {
  return (variant >= 0 && variant < spmm_variant_count()) ? kSpmmVariants[variant][0] : 0;
}

int spmm_variant_xf(int variant) {
  return (variant >= 0 && variant < spmm_variant_count()) ? kSpmmVariants[variant][2] : 0;
}

cudaError_t launch_spmm(const SpmmParams& p0, const SpmmPlan& plan, int flags,
                        cudaStream_t stream) {
  SpmmParams p = p0;
  p.bps = plan.grid / p.slices;  // the plan's grid is a whole number of blocks per slice
  p.rows_q = p.rows / p.bps;
  p.rows_r = (int)(p.rows % p.bps);
  p.steps_q = p.steps / p.slices;
  p.steps_r = p.steps % p.slices;
  cudaError_t e;
  switch (plan.bp) {
    case 2: e = launch_spmm_variant<2>(p, plan.variant, plan.grid, flags, stream); break;
    case 4: e = launch_spmm_variant<4>(p, plan.variant, plan.grid, flags, stream); break;
    case 6: e = launch_spmm_variant<6>(p, plan.variant, plan.grid, flags, stream); break;
    case 8: e = launch_spmm_variant<8>(p, plan.variant, plan.grid, flags, stream); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess || p.slices == 1) return e;
  const int64_t n = (int64_t)p.batch * p.rows;
  int blocks = (int)((n + 255) / 256);
  if (blocks > 4 * plan.sms) blocks = 4 * plan.sms;
  return launch_kernel(spmm_combine_kernel, blocks > 0 ? blocks : 1, 256, 0, stream, flags,
                       p.partial, p.slices, p.batch, p.rows, p.Y, p.ldy);
}

}  // namespace nmk
