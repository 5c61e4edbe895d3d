// gemv.cu -- dense fp16 GEMV baseline, y = W x, for sm_103a.
//
// The pages state the sparse kernel's speedup against dense decoding
// (aimodeling.com article, "The Kernel Is the Other Half of the Answer"), so
// the library carries its own dense kernel, built the same way, as the
// comparison point: persistent blocks over balanced row ranges, the row-steps
// split evenly across warps (split.cuh), x staged once per block in shared
// memory (fp16, natural order), and 128-bit streaming loads of W.  A step is
// 512 columns of one row: lane l reads columns 512t + 8l and 512t + 256 + 8l
// (two 16-byte loads, each warp instruction covering 512 contiguous bytes)
// and the matching 16 bytes of x from shared memory (conflict-free).
// Products and sums are fp32 (one mixed-precision fp16*fp16+fp32 FMA per
// weight, which rounds exactly like converting both operands to fp32 and
// using fmaf); y is rounded to fp16 with round-to-nearest-even.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device.cuh"
#include "kernels.h"
#include "split.cuh"

namespace nmk {

template <int U>
struct GemvBatch {
  uint4 w[U][2];
};

struct GemvCursor {
  int64_t s;
  int64_t row;
  int t;
};

__device__ __forceinline__ void advance(GemvCursor& c, int T) {
  ++c.s;
  if (++c.t == T) {
    c.t = 0;
    ++c.row;
  }
}

template <int U>
__device__ __forceinline__ void gemv_load(GemvBatch<U>& bt, GemvCursor& c, int64_t se, int T,
                                          const GemvParams& p, int64_t r0, int lane) {
#pragma unroll
  for (int i = 0; i < U; ++i) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int col = c.t * 512 + j * 256 + lane * 8;
      if (c.s < se && col < p.cols) {
        bt.w[i][j] = ld_stream_v4(p.W + (r0 + c.row) * p.ld + col);
      } else {
        bt.w[i][j] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    if (c.s < se) advance(c, T);
  }
}

__device__ __forceinline__ void fma8(const uint4& w, const uint4& x, float& a0, float& a1) {
  const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
  const uint32_t xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    a0 = fma_f16f16_f32((uint16_t)(wv[j] & 0xFFFFu), (uint16_t)(xv[j] & 0xFFFFu), a0);
    a1 = fma_f16f16_f32((uint16_t)(wv[j] >> 16), (uint16_t)(xv[j] >> 16), a1);
  }
}

template <int NW, int U>
__global__ void __launch_bounds__(NW * 32, 1) nm_dense_matvec_kernel(const GemvParams p) {
  extern __shared__ __align__(16) uint4 gsmem[];
  const int T = p.steps;
  uint4* xs = gsmem;                                     // [T*64] x as fp16, zero padded
  float* pf = reinterpret_cast<float*>(gsmem + T * 64);  // [NW]
  float* pl = pf + NW;                                   // [NW]
  int* rinfo = reinterpret_cast<int*>(pl + NW);          // [NW][4]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BlockRows br = block_rows(p.rows_q, p.rows_r);
  const int64_t F = (br.r1 - br.r0) * T;
  const WarpRange wr = warp_range<NW>(F, warp);
  const int64_t row0 = div_steps(wr.sb, T);
  const int t0 = (int)(wr.sb - row0 * T);

  GemvCursor lc{wr.sb, row0, t0};
  GemvBatch<U> A, B;
  pdl_launch_dependents();
  if (!p.early_weights) pdl_wait_previous();
  gemv_load<U>(A, lc, wr.se, T, p, br.r0, lane);
  if (p.early_weights) pdl_wait_previous();  // x (and y) may come from the previous kernel

  for (int i = threadIdx.x; i < T * 64; i += NW * 32) {
    xs[i] = (i * 8 < p.cols) ? ld_keep_v4(p.x + (int64_t)i * 8) : make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();

  auto store = [&](int row, float v) { p.y[br.r0 + row] = __float2half_rn(v); };
  GemvCursor cc{wr.sb, row0, t0};
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;

  auto compute = [&](GemvBatch<U>& bt) {
#pragma unroll
    for (int i = 0; i < U; ++i) {
      if (cc.s < wr.se) {
        const uint4 x0 = xs[cc.t * 64 + lane];
        const uint4 x1 = xs[cc.t * 64 + 32 + lane];
        fma8(bt.w[i][0], x0, a0, a1);
        fma8(bt.w[i][1], x1, a2, a3);
        if (cc.t == T - 1 || cc.s == wr.se - 1) {
          const float v = warp_sum((a0 + a1) + (a2 + a3));
          const bool whole = cc.t == T - 1 && (cc.row != row0 || t0 == 0);
          finish_row((int)cc.row, v, whole, (int)row0, warp, lane, pf, pl, store);
          a0 = a1 = a2 = a3 = 0.f;
        }
        advance(cc, T);
      }
    }
  };

  while (cc.s < wr.se) {
    gemv_load<U>(B, lc, wr.se, T, p, br.r0, lane);
    compute(A);
    if (cc.s >= wr.se) break;
    gemv_load<U>(A, lc, wr.se, T, p, br.r0, lane);
    compute(B);
  }
  note_range(rinfo, warp, lane, wr.se > wr.sb ? (int)row0 : -1, t0 != 0,
             (int)(cc.t != 0 ? cc.row : cc.row - 1), cc.t != 0);

  __syncthreads();
  combine_cut_rows<NW>(rinfo, pf, pl, store);
}

size_t gemv_smem_bytes(int steps, int nw) {
  return (size_t)steps * 64 * sizeof(uint4) + 6 * (size_t)nw * sizeof(float);
}

template <int NW, int U>
static cudaError_t launch_gemv_t(const GemvParams& p0, int grid, int flags, cudaStream_t stream) {
  static int smem_set[64] = {0};
  GemvParams p = p0;
  p.rows_q = p.rows / grid;
  p.rows_r = (int)(p.rows % grid);
  auto* k = nm_dense_matvec_kernel<NW, U>;
  cudaError_t e = ensure_max_smem(reinterpret_cast<const void*>(k), smem_set, 64);
  if (e != cudaSuccess) return e;
  return launch_kernel(k, grid, NW * 32, gemv_smem_bytes(p.steps, NW), stream, flags, p);
}

// (warps per block, steps in flight per warp), one block per SM.  Variant 0
// was the fastest on every decode-layer shape measured on GB300.
static const int kGemvVariants[][2] = {{24, 2}, {16, 4}, {16, 2}};

int gemv_variant_count() { return (int)(sizeof(kGemvVariants) / sizeof(kGemvVariants[0])); }

int gemv_variant_warps(int variant) {
  return (variant >= 0 && variant < gemv_variant_count()) ? kGemvVariants[variant][0] : 0;
}

cudaError_t launch_gemv(const GemvParams& p, const GemvPlan& plan, int flags,
                        cudaStream_t stream) {
  switch (plan.variant) {
#define NM_GEMV_CASE(i)                                                                 \
  case i:                                                                              \
    return launch_gemv_t<kGemvVariants[i][0], kGemvVariants[i][1]>(p, plan.grid, flags, stream);
    NM_GEMV_CASE(0) NM_GEMV_CASE(1) NM_GEMV_CASE(2)
#undef NM_GEMV_CASE
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nmk
