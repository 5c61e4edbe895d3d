// spmv.cu -- batch-one N:M bitmask SpMV, y = W x, for sm_103a.
//
// What it computes: aimodeling.com article, "The Kernel Is the Other Half of
// the Answer" -- W is stored as compact fp16 values plus one 32-bit mask word
// per 32 input columns with exactly 16 set bits; the kernel walks each word
// with a fixed-step loop (16 nonzeros per word, so the values of word w sit at
// the fixed offset 16*w of the row and the inner loop has exactly 16 trips).
// weekinpapers.com, Abstract: "bitmask indexing and fixed-step traversal".
//
// GB300 design (the pages' A100 kernel is not described beyond those two
// sentences; everything below is this library's own):
//  * Persistent grid: one block per SM, each owning a balanced contiguous row
//    range; inside the block the row-steps are split evenly over the warps
//    (split.cuh), so every warp streams the same number of bytes.
//  * A step is 32 consecutive mask words of one row: lane l takes word
//    32*t + l, reads its 16 values with one 256-bit load and its mask with one
//    32-bit load.  A warp's step is 1 KiB of values + 128 B of masks, fully
//    contiguous.  U steps are in flight per warp, double-buffered in registers.
//  * x is staged once per block in shared memory as fp32, TRANSPOSED:
//    xs[b][w] = x[32*w + b].  Lanes of a warp always work on 32 consecutive
//    words, so whatever bit b each lane is at, the 32 reads fall in 32
//    distinct banks: the gather never has a bank conflict, for any pattern.
//    A zero pad row sits at b = -1; bfind() of an exhausted (or corrupt) mask
//    returns -1, so every read stays inside the array without a branch.
//  * Decode: most-significant set bit first (bfind), so nonzero k = 15..0 is
//    matched with value k; fp32 FMA into two accumulators; warp butterfly;
//    rows cut between warps are summed in warp order (deterministic).
//  * No tensor cores: batch-one SpMV does ~0.9 flop per byte, far below the
//    tensor roofline; the bound is HBM bandwidth.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device.cuh"
#include "kernels.h"
#include "split.cuh"

namespace nmk {

template <int U>
struct SpmvBatch {
  uint32_t m[U];
  uint32_t v[U][8];
};

struct SpmvCursor {
  int64_t s;    // next flattened step
  int64_t row;  // its local row
  int t;        // its step within the row
};

__device__ __forceinline__ void advance(SpmvCursor& c, int T) {
  ++c.s;
  if (++c.t == T) {
    c.t = 0;
    ++c.row;
  }
}

template <int U>
__device__ __forceinline__ void spmv_load(SpmvBatch<U>& bt, SpmvCursor& c, int64_t se, int T,
                                          const SpmvParams& p, int64_t r0, int lane) {
#pragma unroll
  for (int i = 0; i < U; ++i) {
    const int w = c.t * 32 + lane;
    const bool valid = (c.s < se) && (w < p.words);
    if (valid) {
      const int64_t word = (r0 + c.row) * (int64_t)p.words + w;
      bt.m[i] = ld_stream_u32(p.masks + word);
      ld_stream_v8(p.values + word * 8, bt.v[i]);
    } else {
      bt.m[i] = 0u;  // decodes to the zero pad row
#pragma unroll
      for (int j = 0; j < 8; ++j) bt.v[i][j] = 0u;
    }
    if (c.s < se) advance(c, T);
  }
}

// The fixed-step traversal of one mask word: 16 trips, unrolled.
__device__ __forceinline__ void spmv_word(uint32_t m, const uint32_t (&v)[8], uint32_t col_addr,
                                          uint32_t row_bytes, float& a0, float& a1) {
#pragma unroll
  for (int k = 15; k >= 0; --k) {
    const uint32_t b = msb_index(m);                 // column within the word, or ~0u
    const float xv = lds_f32(col_addr + b * row_bytes);
    m ^= bit_at(b);
    const float2 w2 = half2_bits_to_float2(v[k >> 1]);
    if (k & 1)
      a1 = fmaf(w2.y, xv, a1);
    else
      a0 = fmaf(w2.x, xv, a0);
  }
}

template <int NW, int U>
__global__ void __launch_bounds__(NW * 32, 1) spmv_kernel(const SpmvParams p) {
  extern __shared__ __align__(16) float smem[];
  const int P = p.pitch;
  float* xs = smem;             // [33][P]: pad row, then b = 0..31
  float* pf = smem + 33 * P;    // [NW] first-row partials
  float* pl = pf + NW;          // [NW] last-row partials

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.steps;
  const BlockRows br = block_rows(p.rows);
  const int64_t F = (br.r1 - br.r0) * T;
  const WarpRange wr = warp_range<NW>(F, warp);

  SpmvCursor lc{wr.sb, wr.sb / T, (int)(wr.sb % T)};
  SpmvBatch<U> A, B;
  // Start the first weight loads before staging x so both latencies overlap.
  spmv_load<U>(A, lc, wr.se, T, p, br.r0, lane);

  // Stage x transposed: xs[1 + b][w] = x[32 w + b]; row 0 is zero.
  for (int i = threadIdx.x; i < P; i += NW * 32) xs[i] = 0.f;
  for (int c = warp; c * 32 < p.words; c += NW) {
    const int w = c * 32 + lane;
    if (w < p.words) {
      const uint4* src = reinterpret_cast<const uint4*>(p.x) + (int64_t)w * 4;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 h = ld_keep_v4(src + q);
        const uint32_t hw[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = half2_bits_to_float2(hw[j]);
          const int b = q * 8 + j * 2;
          xs[(1 + b) * P + w] = f.x;
          xs[(2 + b) * P + w] = f.y;
        }
      }
    }
  }
  __syncthreads();

  const uint32_t xs_base = smem_addr(xs);
  const uint32_t row_bytes = 4u * (uint32_t)P;
  auto store = [&](int64_t row, float v) { p.y[br.r0 + row] = __float2half_rn(v); };

  SpmvCursor cc{wr.sb, wr.sb / T, (int)(wr.sb % T)};
  float a0 = 0.f, a1 = 0.f;

  auto compute = [&](SpmvBatch<U>& bt) {
#pragma unroll
    for (int i = 0; i < U; ++i) {
      if (cc.s < wr.se) {
        const uint32_t col_addr = xs_base + row_bytes + 4u * (uint32_t)(cc.t * 32 + lane);
        spmv_word(bt.m[i], bt.v[i], col_addr, row_bytes, a0, a1);
        if (cc.t == T - 1 || cc.s == wr.se - 1) {
          const float v = warp_sum(a0 + a1);
          finish_row(cc.row, v, wr, T, warp, lane, pf, pl, store);
          a0 = 0.f;
          a1 = 0.f;
        }
        advance(cc, T);
      }
    }
  };

  while (cc.s < wr.se) {
    spmv_load<U>(B, lc, wr.se, T, p, br.r0, lane);
    compute(A);
    if (cc.s >= wr.se) break;
    spmv_load<U>(A, lc, wr.se, T, p, br.r0, lane);
    compute(B);
  }

  __syncthreads();
  combine_cut_rows<NW>(F, T, pf, pl, store);
}

template <int NW, int U>
static cudaError_t launch_spmv_t(const SpmvParams& p, int grid, cudaStream_t stream) {
  static int smem_set[64] = {0};
  auto* k = spmv_kernel<NW, U>;
  cudaError_t e = ensure_max_smem(reinterpret_cast<const void*>(k), smem_set, 64);
  if (e != cudaSuccess) return e;
  k<<<grid, NW * 32, spmv_smem_bytes(p.pitch, NW), stream>>>(p);
  return cudaGetLastError();
}

size_t spmv_smem_bytes(int pitch, int nw) {
  return (size_t)(33 * pitch + 2 * nw) * sizeof(float);
}

// (warps per block, steps in flight per warp)
static const int kSpmvVariants[][2] = {{16, 4}, {24, 2}, {16, 2}, {8, 4}, {8, 8}};

int spmv_variant_count() { return (int)(sizeof(kSpmvVariants) / sizeof(kSpmvVariants[0])); }

int spmv_variant_warps(int variant) {
  return (variant >= 0 && variant < spmv_variant_count()) ? kSpmvVariants[variant][0] : 0;
}

cudaError_t launch_spmv(const SpmvParams& p, const SpmvPlan& plan, cudaStream_t stream) {
  switch (plan.variant) {
    case 0: return launch_spmv_t<16, 4>(p, plan.grid, stream);
    case 1: return launch_spmv_t<24, 2>(p, plan.grid, stream);
    case 2: return launch_spmv_t<16, 2>(p, plan.grid, stream);
    case 3: return launch_spmv_t<8, 4>(p, plan.grid, stream);
    case 4: return launch_spmv_t<8, 8>(p, plan.grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nmk
