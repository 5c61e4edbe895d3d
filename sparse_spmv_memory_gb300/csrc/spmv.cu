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
//  * Two kernels share the decode: spmv_full_kernel for rows whose mask words
//    fill whole steps (cols % 1024 == 0, every decode-layer shape), where a
//    warp's steps are one contiguous stretch of memory walked by pointer
//    increments with no per-lane predication; spmv_kernel for any other cols
//    (ragged last step, lanes past the row end load nothing).
//  * x is staged once per block in shared memory, one 32-bit slot per column
//    (fp32, or the fp16 bits in the slot's low half), TRANSPOSED:
//    xs[b][w] = x[32*w + b].  Lanes of a warp always work on 32 consecutive
//    words, so whatever bit b each lane is at, the 32 reads fall in 32
//    distinct banks: the gather never has a bank conflict, for any pattern.
//  * Decode: the 16 trips of a word run as two independent chains of 8 -- the
//    upper values 15..8 scan the mask from its most significant bit (bfind),
//    the lower values 0..7 scan the bit-reversed mask the same way (so from the
//    least significant bit) -- which halves the serial bit-scan latency.  Zero
//    pad rows sit at b = -1 and b = 32 of the x tile; an exhausted (or
//    corrupt) mask makes bfind return -1, which lands in a pad row, so every
//    read stays inside the tile without a branch.  fp32 FMA (or, with x kept as
//    fp16, one mixed fp16*fp16+fp32 FMA), warp butterfly, and rows cut between
//    warps summed in warp order (deterministic).
//  * Programmatic dependent launch (NM_FLAG_PDL): a block signals its
//    dependents as soon as it starts and waits for the previous kernel on the
//    stream only before it reads x or writes y, so in a chain of projections
//    the next launch ramps up under the tail of the current one.  With
//    NM_FLAG_WEIGHTS_CONST the first weight loads are issued before that wait.
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

// x tile layout in shared memory: rows of P 32-bit slots; row 0 and row 33 are
// zero pad rows, row 1 + b holds column b of every mask word.  DEC 1 keeps x as
// fp32, DEC 2/3 keep its fp16 bits in the low half of each slot.
// Short x (at most nthreads / 4 words, up to 6-7K columns; the whole-step
// kernel's SX instances): half a word (16 columns, 32 bytes) per thread,
// consecutive threads consecutive halves, so every warp reads 1 KiB of x
// contiguously with one 256-bit load per lane (two 128-bit loads when x is
// only 16-byte aligned) and twice as many threads share the stores (two
// lanes per word: a 2-way bank conflict).  On GB300 this staged a
// 4096-column x ~0.2 us faster per call.  It is a separate kernel instance:
// adding the branch to the long-x kernels made them 0.1-0.4 us slower.
template <int DEC>
__device__ __forceinline__ void stage_x_halves(float* xs, const __half* x, int words, int P,
                                               int nthreads) {
  for (int i = threadIdx.x; i < P; i += nthreads) {
    xs[i] = 0.f;
    xs[33 * P + i] = 0.f;
  }
  const int c = threadIdx.x;
  if (c >= 2 * words) return;
  const int w = c >> 1, hf = c & 1;  // columns 16 hf .. 16 hf + 15 of word w
  const uint32_t* x32 = reinterpret_cast<const uint32_t*>(x) + (int64_t)c * 8;
  uint32_t hw[8];
  if ((reinterpret_cast<uintptr_t>(x) & 31u) == 0) {
    ld_keep_v8(x32, hw);
  } else {
    const uint4 h0 = ld_keep_v4(x32), h1 = ld_keep_v4(x32 + 4);
    hw[0] = h0.x; hw[1] = h0.y; hw[2] = h0.z; hw[3] = h0.w;
    hw[4] = h1.x; hw[5] = h1.y; hw[6] = h1.z; hw[7] = h1.w;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int b = 16 * hf + 2 * j;
    if (DEC == 1) {
      const float2 f = half2_bits_to_float2(hw[j]);
      xs[(1 + b) * P + w] = f.x;
      xs[(2 + b) * P + w] = f.y;
    } else {
      reinterpret_cast<uint32_t*>(xs)[(1 + b) * P + w] = hw[j] & 0xFFFFu;
      reinterpret_cast<uint32_t*>(xs)[(2 + b) * P + w] = hw[j] >> 16;
    }
  }
}

template <int DEC>
__device__ __forceinline__ void stage_x(float* xs, const __half* x, int words, int P, int nthreads) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < P; i += nthreads) {
    xs[i] = 0.f;
    xs[33 * P + i] = 0.f;
  }
  for (int c = warp; c * 32 < words; c += nthreads / 32) {
    const int w = c * 32 + lane;
    if (w < words) {
      const uint4* src = reinterpret_cast<const uint4*>(x) + (int64_t)w * 4;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 h = ld_keep_v4(src + q);
        const uint32_t hw[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int b = q * 8 + j * 2;
          if (DEC == 1) {
            const float2 f = half2_bits_to_float2(hw[j]);
            xs[(1 + b) * P + w] = f.x;
            xs[(2 + b) * P + w] = f.y;
          } else {
            reinterpret_cast<uint32_t*>(xs)[(1 + b) * P + w] = hw[j] & 0xFFFFu;
            reinterpret_cast<uint32_t*>(xs)[(2 + b) * P + w] = hw[j] >> 16;
          }
        }
      }
    }
  }
}

// The fixed-step traversal of one mask word: 16 trips as two independent
// chains of 8.  The upper chain scans the mask from its most significant bit
// (bfind gives the column b directly) and pairs it with values 15..8; the
// lower chain scans the bit-reversed mask the same way (bfind gives 31 - b)
// and pairs it with values 0..7.  col_addr is the shared address of (b = 0,
// this word); an exhausted chain gets bfind = ~0u and reads a zero pad row.
// DEC 1: fp32 x, fp16 -> fp32 convert + fp32 FMA.
// DEC 2: fp16 x, one mixed fp16*fp16+fp32 FMA; clears the scanned bit by xor.
// DEC 3: as 2, clearing the scanned bit and all above it with bmsk.
template <int DEC>
__device__ __forceinline__ void decode_word(uint32_t m, const uint32_t (&v)[8], uint32_t col_addr,
                                            uint32_t row_bytes, float& a0, float& a1) {
  uint32_t mh = m;
  uint32_t ml = bit_reverse(m);
  const uint32_t top = col_addr + 31u * row_bytes;
  const uint32_t neg_row = 0u - row_bytes;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t bh = msb_index(mh);
    const uint32_t bl = msb_index(ml);
    const uint32_t ah = col_addr + bh * row_bytes;  // bh = ~0u -> pad row 0
    const uint32_t al = top + bl * neg_row;         // bl = ~0u -> pad row 33
    if (DEC == 3) {
      mh &= low_bits(bh);
      ml &= low_bits(bl);
    } else {
      mh ^= bit_at(bh);
      ml ^= bit_at(bl);
    }
    const int kh = 15 - k, kl = k;
    if (DEC == 1) {
      const float xh = lds_f32(ah), xl = lds_f32(al);
      const float2 wh = half2_bits_to_float2(v[kh >> 1]);
      const float2 wl = half2_bits_to_float2(v[kl >> 1]);
      a1 = fmaf((kh & 1) ? wh.y : wh.x, xh, a1);
      a0 = fmaf((kl & 1) ? wl.y : wl.x, xl, a0);
    } else {
      const uint16_t xh = lds_u16(ah), xl = lds_u16(al);
      const uint16_t wh = (kh & 1) ? (uint16_t)(v[kh >> 1] >> 16) : (uint16_t)(v[kh >> 1] & 0xFFFFu);
      const uint16_t wl = (kl & 1) ? (uint16_t)(v[kl >> 1] >> 16) : (uint16_t)(v[kl >> 1] & 0xFFFFu);
      a1 = fma_f16f16_f32(wh, xh, a1);
      a0 = fma_f16f16_f32(wl, xl, a0);
    }
  }
}

// ---------------------------------------------------------------------------
// General kernel: any cols (cols % 32 == 0).  Lanes whose word lies past the
// row end, and steps past the warp's range, load nothing (mask 0, values 0).
// ---------------------------------------------------------------------------
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
      bt.m[i] = 0u;  // decodes to the zero pad rows
#pragma unroll
      for (int j = 0; j < 8; ++j) bt.v[i][j] = 0u;
    }
    if (c.s < se) advance(c, T);
  }
}

// Epilogue EPI 1 (SwiGLU): rows are interleaved (gate, up) pairs; each block
// owns whole pairs, keeps its rows' fp32 sums in shared memory and writes
// h[i] = silu(gate_i) * up_i (fp16) for its pairs after the cut-row combine.
template <int NW>
__device__ __forceinline__ void swiglu_epilogue(const float* ysm, int64_t r0, int64_t r1,
                                                __half* h) {
  __syncthreads();
  for (int64_t k = threadIdx.x; 2 * k < r1 - r0; k += NW * 32) {
    const float g = ysm[2 * k], u = ysm[2 * k + 1];
    h[r0 / 2 + k] = __float2half_rn(g / (1.0f + expf(-g)) * u);
  }
}

template <int NW, int U, int DEC, int EPI>
__global__ void __launch_bounds__(NW * 32, 1) spmv_kernel(const SpmvParams p) {
  extern __shared__ __align__(16) float smem[];
  const int P = p.pitch;
  float* xs = smem;                                    // [34][P]
  float* pf = smem + 34 * P;                           // [NW] first-row partials
  float* pl = pf + NW;                                 // [NW] last-row partials
  int* rinfo = reinterpret_cast<int*>(pl + NW);        // [NW][4] rows each warp touches
  float* ysm = reinterpret_cast<float*>(rinfo + 4 * NW);  // EPI 1: fp32 sums of the block's rows

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.steps;
  const BlockRows br = EPI ? block_row_pairs(p.rows_q, p.rows_r) : block_rows(p.rows_q, p.rows_r);
  const int64_t F = (br.r1 - br.r0) * T;
  const WarpRange wr = warp_range<NW>(F, warp);
  const int64_t row0 = div_steps(wr.sb, T);
  const int t0 = (int)(wr.sb - row0 * T);

  SpmvCursor lc{wr.sb, row0, t0};
  SpmvBatch<U> A, B;
  pdl_launch_dependents();
  if (!p.early_weights) pdl_wait_previous();
  // Start the first weight loads before staging x so both latencies overlap.
  spmv_load<U>(A, lc, wr.se, T, p, br.r0, lane);
  if (p.early_weights) pdl_wait_previous();  // x (and y) may come from the previous kernel
  stage_x<DEC>(xs, p.x, p.words, P, NW * 32);
  __syncthreads();

  const uint32_t xs_base = smem_addr(xs);
  const uint32_t row_bytes = 4u * (uint32_t)P;
  auto store = [&](int row, float v) {
    if (EPI)
      ysm[row] = v;
    else
      p.y[br.r0 + row] = __float2half_rn(v);
  };

  SpmvCursor cc{wr.sb, row0, t0};
  float a0 = 0.f, a1 = 0.f;

  auto compute = [&](SpmvBatch<U>& bt) {
#pragma unroll
    for (int i = 0; i < U; ++i) {
      if (cc.s < wr.se) {
        const uint32_t col_addr = xs_base + row_bytes + 4u * (uint32_t)(cc.t * 32 + lane);
        decode_word<DEC>(bt.m[i], bt.v[i], col_addr, row_bytes, a0, a1);
        if (cc.t == T - 1 || cc.s == wr.se - 1) {
          const float v = warp_sum(a0 + a1);
          const bool whole = cc.t == T - 1 && (cc.row != row0 || t0 == 0);
          finish_row((int)cc.row, v, whole, (int)row0, warp, lane, pf, pl, store);
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
  // cc now points just past the range: a nonzero step means the range ends inside a row
  note_range(rinfo, warp, lane, wr.se > wr.sb ? (int)row0 : -1, t0 != 0,
             (int)(cc.t != 0 ? cc.row : cc.row - 1), cc.t != 0);

  __syncthreads();
  combine_cut_rows<NW>(rinfo, pf, pl, store);
  if (EPI) swiglu_epilogue<NW>(ysm, br.r0, br.r1, p.y);
}

// ---------------------------------------------------------------------------
// Whole-step kernel: cols % 1024 == 0, so every lane of every step has a word
// and a warp's steps are one contiguous stretch of the values and masks
// arrays.  Loads walk two pointers; full batches of U steps run without any
// predication; at most U - 1 trailing steps run one at a time.  A block's
// step count must fit in int (checked on the host).
// ---------------------------------------------------------------------------
template <int U>
__device__ __forceinline__ void load_steps(SpmvBatch<U>& bt, const uint32_t*& vp,
                                           const uint32_t*& mp) {
#pragma unroll
  for (int i = 0; i < U; ++i) {
    bt.m[i] = ld_stream_u32(mp);
    ld_stream_v8(vp, bt.v[i]);
    mp += 32;   // 32 mask words per step
    vp += 256;  // 32 words x 16 fp16 values per step
  }
}

template <int NW, int U, int DEC, int EPI, bool SX>
__global__ void __launch_bounds__(NW * 32, 1) spmv_full_kernel(const SpmvParams p) {
  extern __shared__ __align__(16) float smem[];
  const int P = p.pitch;  // == words
  float* xs = smem;
  float* pf = smem + 34 * P;
  float* pl = pf + NW;
  int* rinfo = reinterpret_cast<int*>(pl + NW);
  float* ysm = reinterpret_cast<float*>(rinfo + 4 * NW);  // EPI 1

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.steps;
  const BlockRows br = EPI ? block_row_pairs(p.rows_q, p.rows_r) : block_rows(p.rows_q, p.rows_r);
  const int F = (int)((br.r1 - br.r0) * T);
  const WarpRange wr = warp_range<NW>(F, warp);
  const int sb = (int)wr.sb, se = (int)wr.se;
  const int nfull = (se - sb) / U;

  const int64_t g = br.r0 * T + sb;  // global index of the warp's first step
  const uint32_t* mp = p.masks + g * 32 + lane;
  const uint32_t* vp = p.values + (g * 32 + lane) * 8;

  SpmvBatch<U> A, B;
  pdl_launch_dependents();
  if (!p.early_weights) pdl_wait_previous();
  if (nfull > 0) load_steps<U>(A, vp, mp);
  if (p.early_weights) pdl_wait_previous();  // x (and y) may come from the previous kernel
  if (SX)
    stage_x_halves<DEC>(xs, p.x, p.words, P, NW * 32);
  else
    stage_x<DEC>(xs, p.x, p.words, P, NW * 32);
  __syncthreads();

  const uint32_t row_bytes = 4u * (uint32_t)P;
  const uint32_t lane_col = smem_addr(xs) + row_bytes + 4u * (uint32_t)lane;
  auto store = [&](int row, float v) {
    if (EPI)
      ysm[row] = v;
    else
      p.y[br.r0 + row] = __float2half_rn(v);
  };

  const int row0 = sb / T, t0 = sb - row0 * T;
  int row = row0, t = t0;
  uint32_t col_addr = lane_col + 128u * (uint32_t)t;
  float a0 = 0.f, a1 = 0.f;

  auto step = [&](uint32_t m, const uint32_t (&v)[8]) {
    decode_word<DEC>(m, v, col_addr, row_bytes, a0, a1);
    col_addr += 128u;
    if (++t == T) {  // row complete
      finish_row(row, warp_sum(a0 + a1), row != row0 || t0 == 0, row0, warp, lane, pf, pl, store);
      a0 = 0.f;
      a1 = 0.f;
      t = 0;
      ++row;
      col_addr = lane_col;
    }
  };

  for (int i = 0; i < nfull; i += 2) {
    if (i + 1 < nfull) load_steps<U>(B, vp, mp);
#pragma unroll
    for (int u = 0; u < U; ++u) step(A.m[u], A.v[u]);
    if (i + 1 >= nfull) break;
    if (i + 2 < nfull) load_steps<U>(A, vp, mp);
#pragma unroll
    for (int u = 0; u < U; ++u) step(B.m[u], B.v[u]);
  }
  for (int s = sb + nfull * U; s < se; ++s) {
    SpmvBatch<1> one;
    load_steps<1>(one, vp, mp);
    step(one.m[0], one.v[0]);
  }
  if (se > sb && t != 0)  // the warp's range ends inside a row
    finish_row(row, warp_sum(a0 + a1), false, row0, warp, lane, pf, pl, store);
  note_range(rinfo, warp, lane, se > sb ? row0 : -1, t0 != 0, t != 0 ? row : row - 1, t != 0);

  __syncthreads();
  combine_cut_rows<NW>(rinfo, pf, pl, store);
  if (EPI) swiglu_epilogue<NW>(ysm, br.r0, br.r1, p.y);
}

size_t spmv_smem_bytes(int pitch, int nw) {
  return (size_t)(34 * pitch + 6 * nw) * sizeof(float);  // x tile, pf, pl, rinfo
}

template <int NW, int U, int DEC, int EPI>
static cudaError_t launch_spmv_e(const SpmvParams& p0, int grid, int flags, cudaStream_t stream) {
  static int smem_full[64] = {0}, smem_short[64] = {0}, smem_gen[64] = {0};
  SpmvParams p = p0;
  const int64_t units = EPI ? p.rows / 2 : p.rows;  // rows, or (gate, up) pairs
  p.rows_q = units / grid;
  p.rows_r = (int)(units % grid);
  const int64_t block_rows_max = EPI ? 2 * ((p.rows / 2 + grid - 1) / grid) : 0;
  const size_t smem = spmv_smem_bytes(p.pitch, NW) + (size_t)block_rows_max * sizeof(float);
  const int64_t block_steps = ((p.rows + grid - 1) / grid + 2) * p.steps;
  if (p.words % 32 == 0 && block_steps < (int64_t)0x7FFFFFFF) {
    const bool sx = 4 * p.words <= NW * 32;  // short x: the half-word staging instance
    auto* k = sx ? spmv_full_kernel<NW, U, DEC, EPI, true> : spmv_full_kernel<NW, U, DEC, EPI, false>;
    cudaError_t e = ensure_max_smem(reinterpret_cast<const void*>(k), sx ? smem_short : smem_full, 64);
    if (e != cudaSuccess) return e;
    return launch_kernel(k, grid, NW * 32, smem, stream, flags, p);
  }
  auto* k = spmv_kernel<NW, U, DEC, EPI>;
  cudaError_t e = ensure_max_smem(reinterpret_cast<const void*>(k), smem_gen, 64);
  if (e != cudaSuccess) return e;
  return launch_kernel(k, grid, NW * 32, smem, stream, flags, p);
}

template <int NW, int U, int DEC>
static cudaError_t launch_spmv_t(const SpmvParams& p, int grid, int epi, int flags,
                                 cudaStream_t stream) {
  return epi ? launch_spmv_e<NW, U, DEC, 1>(p, grid, flags, stream)
             : launch_spmv_e<NW, U, DEC, 0>(p, grid, flags, stream);
}

// (warps per block, steps in flight per warp, decode).  Every variant runs
// one resident block per SM.  Sweeps on GB300 over the decode-layer shapes put
// variant 6 ahead below ~33M weight positions (more warps hide the decode's
// latencies when each warp has only a few steps), variant 0 up to ~134M and
// variant 1 above; the others stay for tuning and so the tests cover more
// block shapes.  (Blocks sized for two per SM, one or two launched per SM,
// were slower on every shape.)
static const int kSpmvVariants[][3] = {{24, 2, 1}, {20, 3, 2}, {16, 4, 2}, {24, 2, 2},
                                       {24, 2, 3}, {16, 2, 1}, {28, 1, 1}};

int spmv_variant_count() { return (int)(sizeof(kSpmvVariants) / sizeof(kSpmvVariants[0])); }

int spmv_variant_warps(int variant) {
  return (variant >= 0 && variant < spmv_variant_count()) ? kSpmvVariants[variant][0] : 0;
}

cudaError_t launch_spmv(const SpmvParams& p, const SpmvPlan& plan, int flags,
                        cudaStream_t stream, int epilogue) {
  switch (plan.variant) {
#define NM_SPMV_CASE(i)                                                                 \
  case i:                                                                              \
    return launch_spmv_t<kSpmvVariants[i][0], kSpmvVariants[i][1], kSpmvVariants[i][2]>( \
        p, plan.grid, epilogue, flags, stream);
    NM_SPMV_CASE(0) NM_SPMV_CASE(1) NM_SPMV_CASE(2) NM_SPMV_CASE(3) NM_SPMV_CASE(4)
    NM_SPMV_CASE(5) NM_SPMV_CASE(6)
#undef NM_SPMV_CASE
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nmk
