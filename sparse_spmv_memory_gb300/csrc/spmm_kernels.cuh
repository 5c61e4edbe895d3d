// spmm_kernels.cuh -- the small-batch N:M bitmask SpMM kernels, Y = W X for
// 1..8 tokens (sm_103a); compiled once per x-slot width (spmm_b2.cu ...
// spmm_b8.cu, in parallel), dispatched from spmm.cu.
//
// Decoding several tokens at once (small-batch serving, speculative decoding)
// turns the batch-one product of the SparseDecoding pages (aimodeling.com
// article, "The Kernel Is the Other Half of the Answer"; news.bitwarelabs.com
// summary, "What's new": decoding is SpMV-bound, prefill SpMM-bound) into a
// product with a handful of right-hand sides.  The weights still dominate the
// traffic, so the kernel streams them exactly as nm_spmv does and decodes each
// mask word once for the whole batch:
//  * the x tile holds, for every (bit b, mask word w), one slot of BP fp16
//    values -- the BP tokens' x at column 32w + b (BP = 2, 4, 6 or 8; tokens
//    past the batch are zero).  Lanes of a warp hold consecutive words, so one
//    4/8/16-byte shared load (three 4-byte loads for a 12-byte slot) per
//    nonzero feeds all BP FMAs without a bank conflict;
//  * the same two-chain bfind scan as nm_spmv (values 15..8 from the top bit,
//    0..7 from the bit-reversed mask; exhausted chains read zero pad rows);
//  * per nonzero either one mixed-precision fp16*fp16+fp32 FMA per token
//    (XF 0: fp16 slots; XF 3: the same with the slot split into 16-bit
//    registers inside the PTX) or one fp16->fp32 convert of the weight and one
//    packed fp32x2 FMA per two tokens (XF 1: fp32 slots, twice the shared
//    memory, half the FMA instructions at batch 4-8);
//  * rows split over blocks and row-steps over warps as in nm_spmv
//    (split.cuh), with BP sums per row.
// When the tile of a whole row does not fit in shared memory (long rows with
// a large batch), the columns are cut into S slices of whole warp-steps, the
// grid is shared among the slices, each block writes fp32 partial sums for
// its slice to the caller's workspace, and a second kernel adds the S
// partials in slice order (deterministic) and rounds to fp16.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device.cuh"
#include "kernels.h"
#include "spmm_variants.h"
#include "split.cuh"

namespace nmk {

template <int BP>
__device__ __forceinline__ void lds_slot(uint32_t addr, uint32_t (&r)[BP / 2]) {
  if constexpr (BP == 2) {
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(r[0]) : "r"(addr));
  } else if constexpr (BP == 6) {  // 12-byte slots: three 4-byte loads
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(r[0]) : "r"(addr));
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(r[1]) : "r"(addr + 4u));
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(r[2]) : "r"(addr + 8u));
  } else if constexpr (BP == 4) {
    asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
  } else {
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
  }
}

// fp32 slot loads: BP floats as BP/2 packed pairs.  A 32-byte slot (BP 8) is
// read as two 16-byte halves; word w keeps its halves swapped when bit 2 of w
// is set (swz = 16), so the 8 lanes of a quarter-warp hit disjoint banks.
template <int BP>
__device__ __forceinline__ void lds_slot_f32(uint32_t addr, uint32_t swz,
                                             unsigned long long (&r)[BP / 2]) {
  if constexpr (BP == 2) {
    asm volatile("ld.shared.b64 %0, [%1];" : "=l"(r[0]) : "r"(addr));
  } else if constexpr (BP == 4) {
    asm volatile("ld.shared.v2.b64 {%0,%1}, [%2];" : "=l"(r[0]), "=l"(r[1]) : "r"(addr));
  } else {
    asm volatile("ld.shared.v2.b64 {%0,%1}, [%2];" : "=l"(r[0]), "=l"(r[1]) : "r"(addr + swz));
    asm volatile("ld.shared.v2.b64 {%0,%1}, [%2];"
                 : "=l"(r[2]), "=l"(r[3])
                 : "r"(addr + (16u - swz)));
  }
}

__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b,
                                                    unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ unsigned long long splat2(float v) {
  const unsigned long long u = __float_as_uint(v);
  return (u << 32) | u;
}

__device__ __forceinline__ float pair_lo(unsigned long long p) { return __uint_as_float((uint32_t)p); }
__device__ __forceinline__ float pair_hi(unsigned long long p) {
  return __uint_as_float((uint32_t)(p >> 32));
}

__device__ __forceinline__ uint16_t half_of(uint32_t pair, int hi) {
  return hi ? (uint16_t)(pair >> 16) : (uint16_t)(pair & 0xFFFFu);
}

// One mask word, all BP tokens: 16 trips as two chains of 8.
template <int BP>
__device__ __forceinline__ void decode_word_batch(uint32_t m, const uint32_t (&v)[8],
                                                  uint32_t col_addr, uint32_t row_bytes,
                                                  float (&a)[2][BP]) {
  uint32_t mh = m;
  uint32_t ml = bit_reverse(m);
  const uint32_t top = col_addr + 31u * row_bytes;
  const uint32_t neg_row = 0u - row_bytes;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t bh = msb_index(mh);
    const uint32_t bl = msb_index(ml);
    const uint32_t ah = col_addr + bh * row_bytes;  // ~0u -> pad row 0
    const uint32_t al = top + bl * neg_row;         // ~0u -> pad row 33
    mh ^= bit_at(bh);
    ml ^= bit_at(bl);
    uint32_t xh[BP / 2], xl[BP / 2];
    lds_slot<BP>(ah, xh);
    lds_slot<BP>(al, xl);
    const int kh = 15 - k, kl = k;
    const uint16_t wh = half_of(v[kh >> 1], kh & 1);
    const uint16_t wl = half_of(v[kl >> 1], kl & 1);
#pragma unroll
    for (int j = 0; j < BP; ++j) {
      a[1][j] = fma_f16f16_f32(wh, half_of(xh[j >> 1], j & 1), a[1][j]);
      a[0][j] = fma_f16f16_f32(wl, half_of(xl[j >> 1], j & 1), a[0][j]);
    }
  }
}

// As decode_word_batch, with fp32 slots: a[c][q] packs tokens 2q, 2q+1.
template <int BP>
__device__ __forceinline__ void decode_word_batch_f32(uint32_t m, const uint32_t (&v)[8],
                                                      uint32_t col_addr, uint32_t row_bytes,
                                                      uint32_t swz,
                                                      unsigned long long (&a)[2][BP / 2]) {
  uint32_t mh = m;
  uint32_t ml = bit_reverse(m);
  const uint32_t top = col_addr + 31u * row_bytes;
  const uint32_t neg_row = 0u - row_bytes;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t bh = msb_index(mh);
    const uint32_t bl = msb_index(ml);
    const uint32_t ah = col_addr + bh * row_bytes;
    const uint32_t al = top + bl * neg_row;
    mh ^= bit_at(bh);
    ml ^= bit_at(bl);
    unsigned long long xh[BP / 2], xl[BP / 2];
    lds_slot_f32<BP>(ah, swz, xh);
    lds_slot_f32<BP>(al, swz, xl);
    const int kh = 15 - k, kl = k;
    const float2 fh = half2_bits_to_float2(v[kh >> 1]);
    const float2 fl = half2_bits_to_float2(v[kl >> 1]);
    const unsigned long long wh = splat2((kh & 1) ? fh.y : fh.x);
    const unsigned long long wl = splat2((kl & 1) ? fl.y : fl.x);
#pragma unroll
    for (int q = 0; q < BP / 2; ++q) {
      a[1][q] = ffma2(wh, xh[q], a[1][q]);
      a[0][q] = ffma2(wl, xl[q], a[0][q]);
    }
  }
}

// fp32 slots with scalar FMAs (XF 2): one convert of the weight and one fp32
// FMA per token, no half extraction.
template <int BP>
__device__ __forceinline__ void decode_word_batch_f32s(uint32_t m, const uint32_t (&v)[8],
                                                       uint32_t col_addr, uint32_t row_bytes,
                                                       uint32_t swz, float (&a)[2][BP]) {
  uint32_t mh = m;
  uint32_t ml = bit_reverse(m);
  const uint32_t top = col_addr + 31u * row_bytes;
  const uint32_t neg_row = 0u - row_bytes;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t bh = msb_index(mh);
    const uint32_t bl = msb_index(ml);
    const uint32_t ah = col_addr + bh * row_bytes;
    const uint32_t al = top + bl * neg_row;
    mh ^= bit_at(bh);
    ml ^= bit_at(bl);
    unsigned long long xh[BP / 2], xl[BP / 2];
    lds_slot_f32<BP>(ah, swz, xh);
    lds_slot_f32<BP>(al, swz, xl);
    const int kh = 15 - k, kl = k;
    const float2 fh = half2_bits_to_float2(v[kh >> 1]);
    const float2 fl = half2_bits_to_float2(v[kl >> 1]);
    const float wh = (kh & 1) ? fh.y : fh.x;
    const float wl = (kl & 1) ? fl.y : fl.x;
#pragma unroll
    for (int j = 0; j < BP; ++j) {
      const float xhj = (j & 1) ? pair_hi(xh[j >> 1]) : pair_lo(xh[j >> 1]);
      const float xlj = (j & 1) ? pair_hi(xl[j >> 1]) : pair_lo(xl[j >> 1]);
      a[1][j] = fmaf(wh, xhj, a[1][j]);
      a[0][j] = fmaf(wl, xlj, a[0][j]);
    }
  }
}

// The x slot's BP fp16 values unpacked into 16-bit registers inside the PTX
// (mov.b32 {lo, hi} names the halves of a 32-bit register, so the mixed
// fp16*fp16+fp32 FMAs take them without separate extraction instructions).
// XF 3: one 4/8/16-byte shared load per nonzero, as XF 0.
template <int BP>
__device__ __forceinline__ void fma_slot_u32(uint32_t addr, uint16_t w, float (&a)[BP]) {
  if constexpr (BP == 2) {
    asm volatile(
        "{.reg .b32 r0; .reg .b16 x0, x1;\n\t"
        "ld.shared.b32 r0, [%2];\n\t"
        "mov.b32 {x0, x1}, r0;\n\t"
        "fma.rn.f32.f16 %0, %3, x0, %0;\n\t"
        "fma.rn.f32.f16 %1, %3, x1, %1;}"
        : "+f"(a[0]), "+f"(a[1])
        : "r"(addr), "h"(w));
  } else if constexpr (BP == 4) {
    asm volatile(
        "{.reg .b32 r0, r1; .reg .b16 x0, x1, x2, x3;\n\t"
        "ld.shared.v2.b32 {r0, r1}, [%4];\n\t"
        "mov.b32 {x0, x1}, r0;\n\t"
        "mov.b32 {x2, x3}, r1;\n\t"
        "fma.rn.f32.f16 %0, %5, x0, %0;\n\t"
        "fma.rn.f32.f16 %1, %5, x1, %1;\n\t"
        "fma.rn.f32.f16 %2, %5, x2, %2;\n\t"
        "fma.rn.f32.f16 %3, %5, x3, %3;}"
        : "+f"(a[0]), "+f"(a[1]), "+f"(a[2]), "+f"(a[3])
        : "r"(addr), "h"(w));
  } else {
    asm volatile(
        "{.reg .b32 r0, r1, r2, r3; .reg .b16 x0, x1, x2, x3, x4, x5, x6, x7;\n\t"
        "ld.shared.v4.b32 {r0, r1, r2, r3}, [%8];\n\t"
        "mov.b32 {x0, x1}, r0;\n\t"
        "mov.b32 {x2, x3}, r1;\n\t"
        "mov.b32 {x4, x5}, r2;\n\t"
        "mov.b32 {x6, x7}, r3;\n\t"
        "fma.rn.f32.f16 %0, %9, x0, %0;\n\t"
        "fma.rn.f32.f16 %1, %9, x1, %1;\n\t"
        "fma.rn.f32.f16 %2, %9, x2, %2;\n\t"
        "fma.rn.f32.f16 %3, %9, x3, %3;\n\t"
        "fma.rn.f32.f16 %4, %9, x4, %4;\n\t"
        "fma.rn.f32.f16 %5, %9, x5, %5;\n\t"
        "fma.rn.f32.f16 %6, %9, x6, %6;\n\t"
        "fma.rn.f32.f16 %7, %9, x7, %7;}"
        : "+f"(a[0]), "+f"(a[1]), "+f"(a[2]), "+f"(a[3]), "+f"(a[4]), "+f"(a[5]), "+f"(a[6]),
          "+f"(a[7])
        : "r"(addr), "h"(w));
  }
}

// XF 3 decode: as decode_word_batch, the x slot unpacked inside the PTX.
template <int BP>
__device__ __forceinline__ void decode_word_batch_u(uint32_t m, const uint32_t (&v)[8],
                                                    uint32_t col_addr, uint32_t row_bytes,
                                                    float (&a)[2][BP]) {
  uint32_t mh = m;
  uint32_t ml = bit_reverse(m);
  const uint32_t top = col_addr + 31u * row_bytes;
  const uint32_t neg_row = 0u - row_bytes;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t bh = msb_index(mh);
    const uint32_t bl = msb_index(ml);
    const uint32_t ah = col_addr + bh * row_bytes;  // ~0u -> pad row 0
    const uint32_t al = top + bl * neg_row;         // ~0u -> pad row 33
    mh ^= bit_at(bh);
    ml ^= bit_at(bl);
    const int kh = 15 - k, kl = k;
    fma_slot_u32<BP>(ah, half_of(v[kh >> 1], kh & 1), a[1]);
    fma_slot_u32<BP>(al, half_of(v[kl >> 1], kl & 1), a[0]);
  }
}

template <int U>
struct SpmmBatch {
  uint32_t m[U];
  uint32_t v[U][8];
};

struct SpmmCursor {
  int64_t s;    // next step of the block's flattened (row, step) range
  int64_t row;  // its local row
  int t;        // its step within the slice's part of the row
};

__device__ __forceinline__ void advance(SpmmCursor& c, int T) {
  ++c.s;
  if (++c.t == T) {
    c.t = 0;
    ++c.row;
  }
}

template <int U>
__device__ __forceinline__ void spmm_load(SpmmBatch<U>& bt, SpmmCursor& c, int64_t se, int T,
                                          const SpmmParams& p, int64_t r0, int w0, int wend,
                                          int lane) {
#pragma unroll
  for (int i = 0; i < U; ++i) {
    const int w = w0 + c.t * 32 + lane;
    if (c.s < se && w < wend) {
      const int64_t word = (r0 + c.row) * (int64_t)p.words + w;
      bt.m[i] = ld_stream_u32(p.masks + word);
      ld_stream_v8(p.values + word * 8, bt.v[i]);
    } else {
      bt.m[i] = 0u;
#pragma unroll
      for (int j = 0; j < 8; ++j) bt.v[i][j] = 0u;
    }
    if (c.s < se) advance(c, T);
  }
}

// fp16 slots of one column slice: task (q, wl) reads columns 8q .. 8q + 7 of
// local word wl for up to four tokens at a time (one 16-byte load per token),
// transposes those 4 x 8 halves in registers (one byte permute per pair of
// tokens and column) and writes each column's part of its slot whole (one
// 4- or 8-byte store).  Tasks are q-major, so the lanes of a warp write
// consecutive slots of one tile row: no bank conflicts, and the tile is
// written in as many shared-memory wavefronts as it has 128-byte lines.
template <int BP>
__device__ __forceinline__ void stage_x_slice_f16(uint32_t* tile32, const SpmmParams& p, int P,
                                                  int w0, int wend, int nthreads) {
  constexpr int kSlotWords = BP / 2;
  // tokens per pass: 12-byte slots (BP 6) are only 4-byte aligned, so they
  // are written one 4-byte word (two tokens) at a time
  constexpr int G = BP < 4 ? BP : (BP == 6 ? 2 : 4);
  for (int i = threadIdx.x; i < P * kSlotWords; i += nthreads) {
    tile32[i] = 0u;
    tile32[33 * P * kSlotWords + i] = 0u;
  }
  const uint32_t tile_addr = smem_addr(tile32);
  for (int task = threadIdx.x; task < 4 * P; task += nthreads) {
    const int q = task / P, wl = task - q * P;
    const int w = w0 + wl;
#pragma unroll
    for (int g = 0; g < BP; g += G) {
      uint4 h[G];
#pragma unroll
      for (int j = 0; j < G; ++j) {
        h[j] = make_uint4(0u, 0u, 0u, 0u);
        if (w < wend && g + j < p.batch)
          h[j] = ld_keep_v4(p.X + (int64_t)(g + j) * p.ldx + (int64_t)w * 32 + q * 8);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {  // column b = 8q + i
        uint32_t part[G / 2];
#pragma unroll
        for (int k = 0; k < G / 2; ++k) {
          const uint4 a = h[2 * k], b = h[2 * k + 1];
          const int r = i >> 1;
          const uint32_t ra = r == 0 ? a.x : r == 1 ? a.y : r == 2 ? a.z : a.w;
          const uint32_t rb = r == 0 ? b.x : r == 1 ? b.y : r == 2 ? b.z : b.w;
          part[k] = __byte_perm(ra, rb, (i & 1) ? 0x7632u : 0x5410u);  // tokens g+2k, g+2k+1
        }
        const uint32_t at =
            tile_addr + (uint32_t)(((1 + 8 * q + i) * P + wl) * kSlotWords + g / 2) * 4u;
        if constexpr (G == 2)
          asm volatile("st.shared.b32 [%0], %1;" ::"r"(at), "r"(part[0]));
        else
          asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(at), "r"(part[0]), "r"(part[1]));
      }
    }
  }
}

// Stage one column slice of X in shared memory: tile[1 + b][wl][j] =
// X[j][32 (w0 + wl) + b] for the slice's words w0 + wl < wend (fp16, or fp32
// with the two 16-byte halves of a 32-byte slot swapped for odd word groups),
// zero pad rows 0 and 33, tokens past the batch zero.
template <int BP, bool F32>
__device__ __forceinline__ void stage_x_slice(float* smem, const SpmmParams& p, int P, int w0,
                                              int wend, int nthreads) {
  if constexpr (!F32) {
    stage_x_slice_f16<BP>(reinterpret_cast<uint32_t*>(smem), p, P, w0, wend, nthreads);
    return;
  }
  constexpr int kSlotWords = F32 ? BP : BP / 2;
  uint16_t* tile = reinterpret_cast<uint16_t*>(smem);
  float* tile_f = smem;
  uint32_t* tile32 = reinterpret_cast<uint32_t*>(smem);
  for (int i = threadIdx.x; i < P * kSlotWords; i += nthreads) {
    tile32[i] = 0u;
    tile32[33 * P * kSlotWords + i] = 0u;
  }
  for (int task = threadIdx.x; task < P * BP; task += nthreads) {
    const int j = task / P, wl = task - j * P;
    const int w = w0 + wl;
    uint32_t h[16];
    if (w < wend && j < p.batch) {
      const uint4* src = reinterpret_cast<const uint4*>(p.X + (int64_t)j * p.ldx) + (int64_t)w * 4;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 u = ld_keep_v4(src + q);
        h[4 * q] = u.x;
        h[4 * q + 1] = u.y;
        h[4 * q + 2] = u.z;
        h[4 * q + 3] = u.w;
      }
    } else {
#pragma unroll
      for (int q = 0; q < 16; ++q) h[q] = 0u;
    }
#pragma unroll
    for (int b = 0; b < 32; ++b) {
      const int jp = (F32 && BP == 8) ? (((j >> 2) ^ ((wl >> 2) & 1)) << 2) | (j & 3) : j;
      const int64_t at = ((int64_t)(1 + b) * P + wl) * BP + jp;
      if (F32) {
        const float2 f = half2_bits_to_float2(h[b >> 1]);
        tile_f[at] = (b & 1) ? f.y : f.x;
      } else {
        tile[at] = half_of(h[b >> 1], b & 1);
      }
    }
  }
}

// Warp sums of BP per-lane values (one per token) in five xor levels: first
// log2(BP) split levels (xor 16, 8, ...) where each lane keeps half of its
// remaining values and adds its partner's copy of that half, then plain
// butterfly levels on the one value left.  Lane L ends with the total of
// token L / (32 / BP) -- BP - 1 + log2(32 / BP) shuffles instead of 5 BP,
// and every total is bit for bit that of a butterfly per token (each level
// adds the same two partial sums, and fp32 addition commutes).
template <int BP>
__device__ __forceinline__ float warp_sum_tokens(float (&v)[BP], int lane) {
#pragma unroll
  for (int half = BP / 2, off = 16; half >= 1; half /= 2, off /= 2) {
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? v[i] : v[half + i];
      const float keep = up ? v[half + i] : v[i];
      v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
    }
  }
  float t = v[0];
#pragma unroll
  for (int off = 16 / BP; off > 0; off >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, off);
  return t;
}

template <int NW, int U, int BP, int XF>
__global__ void __launch_bounds__(NW * 32, 1) spmm_kernel(const SpmmParams p) {
  extern __shared__ __align__(16) float smem[];
  const int P = p.pitch;
  constexpr bool kF32 = XF == 1 || XF == 2;             // fp32 slots
  constexpr int kSlotWords = kF32 ? BP : BP / 2;        // 32-bit words per slot
  uint16_t* tile = reinterpret_cast<uint16_t*>(smem);   // [34][P][BP] slots
  float* pf = smem + 34 * P * kSlotWords;               // [NW][BP]
  float* pl = pf + NW * BP;                             // [NW][BP]
  int* rinfo = reinterpret_cast<int*>(pl + NW * BP);    // [NW][4]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sl = (int)(blockIdx.x / (unsigned)p.bps), c = blockIdx.x - sl * p.bps;  // slice, block in it
  const BlockRows br = split_part(c, p.rows_q, p.rows_r, p.bps);
  const int64_t r0 = br.r0, r1 = br.r1;
  const BlockRows sr = split_part(sl, p.steps_q, p.steps_r, p.slices);
  const int ts0 = (int)sr.r0, ts1 = (int)sr.r1;
  const int T = ts1 - ts0;              // warp-steps per row in this slice
  const int w0 = ts0 * 32;              // first mask word of the slice
  const int wend = min(ts1 * 32, p.words);
  const int64_t F = (r1 - r0) * T;
  const WarpRange wr = warp_range<NW>(F, warp);
  const int64_t row0 = div_steps(wr.sb, T);
  const int t0 = (int)(wr.sb - row0 * T);

  SpmmCursor lc{wr.sb, row0, t0};
  SpmmBatch<U> A, B;
  pdl_launch_dependents();
  if (!p.early_weights) pdl_wait_previous();
  spmm_load<U>(A, lc, wr.se, T, p, r0, w0, wend, lane);
  if (p.early_weights) pdl_wait_previous();  // X (and Y, the workspace) may be the previous kernel's

  stage_x_slice<BP, kF32>(smem, p, P, w0, wend, NW * 32);
  __syncthreads();

  const uint32_t row_bytes = (uint32_t)P * kSlotWords * 4u;
  const uint32_t swz = ((lane >> 2) & 1) ? 16u : 0u;  // local word bit 2 == lane bit 2
  const uint32_t tile_base = smem_addr(tile) + row_bytes;  // row b = 0
  auto store = [&](int row, const float (&v)[BP]) {
    const int64_t gr = r0 + row;
    if (p.slices == 1) {
#pragma unroll
      for (int j = 0; j < BP; ++j)
        if (j < p.batch) p.Y[(int64_t)j * p.ldy + gr] = __float2half_rn(v[j]);
    } else {
#pragma unroll
      for (int j = 0; j < BP; ++j)
        if (j < p.batch) p.partial[((int64_t)sl * p.batch + j) * p.rows + gr] = v[j];
    }
  };

  SpmmCursor cc{wr.sb, row0, t0};
  float a[2][BP];                   // XF 0
  unsigned long long a2[2][BP / 2];  // XF 1: packed pairs of tokens
#pragma unroll
  for (int j = 0; j < BP; ++j) a[0][j] = a[1][j] = 0.f;
#pragma unroll
  for (int q = 0; q < BP / 2; ++q) a2[0][q] = a2[1][q] = 0ull;

  auto compute = [&](SpmmBatch<U>& bt) {
#pragma unroll
    for (int i = 0; i < U; ++i) {
      if (cc.s < wr.se) {
        const uint32_t col_addr = tile_base + (uint32_t)(cc.t * 32 + lane) * (kSlotWords * 4u);
        if constexpr (XF == 1)
          decode_word_batch_f32<BP>(bt.m[i], bt.v[i], col_addr, row_bytes, swz, a2);
        else if constexpr (XF == 3)
          decode_word_batch_u<BP>(bt.m[i], bt.v[i], col_addr, row_bytes, a);
        else if constexpr (XF == 2)
          decode_word_batch_f32s<BP>(bt.m[i], bt.v[i], col_addr, row_bytes, swz, a);
        else
          decode_word_batch<BP>(bt.m[i], bt.v[i], col_addr, row_bytes, a);
        if (cc.t == T - 1 || cc.s == wr.se - 1) {
          float v[BP];
#pragma unroll
          for (int j = 0; j < BP; ++j) {
            const float part = XF == 1
                                   ? ((j & 1) ? pair_hi(a2[0][j >> 1]) + pair_hi(a2[1][j >> 1])
                                              : pair_lo(a2[0][j >> 1]) + pair_lo(a2[1][j >> 1]))
                                   : a[0][j] + a[1][j];
            v[j] = warp_sum(part);
            a[0][j] = a[1][j] = 0.f;
          }
#pragma unroll
          for (int q = 0; q < BP / 2; ++q) a2[0][q] = a2[1][q] = 0ull;
          const bool whole = cc.t == T - 1 && (cc.row != row0 || t0 == 0);
          finish_row_n<BP>((int)cc.row, v, whole, (int)row0, warp, lane, pf, pl, store);
        }
        advance(cc, T);
      }
    }
  };

  while (cc.s < wr.se) {
    spmm_load<U>(B, lc, wr.se, T, p, r0, w0, wend, lane);
    compute(A);
    if (cc.s >= wr.se) break;
    spmm_load<U>(A, lc, wr.se, T, p, r0, w0, wend, lane);
    compute(B);
  }

  note_range(rinfo, warp, lane, wr.se > wr.sb ? (int)row0 : -1, t0 != 0,
             (int)(cc.t != 0 ? cc.row : cc.row - 1), cc.t != 0);

  __syncthreads();
  combine_cut_rows_n<NW, BP>(rinfo, pf, pl, store);
}

// Whole-step kernel (cols % 1024 == 0, so every step of every slice is 32
// whole mask words): as spmm_kernel, but a warp's steps are walked by pointer
// increments with no per-step predication (as in spmv_full_kernel) -- one
// contiguous stretch per row slice, a fixed jump over the other slices' steps
// at each row change -- and a row's BP sums are reduced by warp_sum_tokens,
// each token's total then held (and stored) by its own lane.  SLICED is
// false for a single column slice: the block's steps are then one contiguous
// stretch and the sums go straight to Y, with no slice bookkeeping at all
// (it cost 2-5 % at 2-4 tokens when kept as run-time checks).
template <int U, bool SLICED>
__device__ __forceinline__ void load_steps_batch(SpmmBatch<U>& bt, const uint32_t*& vp,
                                                 const uint32_t*& mp, int& lt, int Ts,
                                                 int skip) {
#pragma unroll
  for (int i = 0; i < U; ++i) {
    bt.m[i] = ld_stream_u32(mp);
    ld_stream_v8(vp, bt.v[i]);
    mp += 32;
    vp += 256;
    if (SLICED && ++lt == Ts) {  // next row: jump over the other slices' steps
      lt = 0;
      mp += 32 * skip;
      vp += 256 * skip;
    }
  }
}

template <int NW, int U, int BP, int XF, bool SLICED>
__global__ void __launch_bounds__(NW * 32, 1) spmm_full_kernel(const SpmmParams p) {
  extern __shared__ __align__(16) float smem[];
  const int P = p.pitch;
  constexpr bool kF32 = XF == 1 || XF == 2;
  constexpr int kSlotWords = kF32 ? BP : BP / 2;
  constexpr int BR = BP == 6 ? 8 : BP;  // tokens in the reduction (BP 6: two zero)
  constexpr int kLanesPerToken = 32 / BR;
  uint16_t* tile = reinterpret_cast<uint16_t*>(smem);
  float* pf = smem + 34 * P * kSlotWords;               // [NW][BP]
  float* pl = pf + NW * BP;                             // [NW][BP]
  int* rinfo = reinterpret_cast<int*>(pl + NW * BP);    // [NW][4]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int sl = 0, ts0 = 0, Ts = p.steps;  // slice, its first step and steps of a row
  BlockRows br;
  if (SLICED) {
    sl = (int)(blockIdx.x / (unsigned)p.bps);
    const int c = blockIdx.x - sl * p.bps;  // block within the slice
    br = split_part(c, p.rows_q, p.rows_r, p.bps);
    const BlockRows sr = split_part(sl, p.steps_q, p.steps_r, p.slices);
    ts0 = (int)sr.r0;
    Ts = (int)(sr.r1 - sr.r0);
  } else {
    br = block_rows(p.rows_q, p.rows_r);
  }
  const int skip = p.steps - Ts;  // the other slices' steps
  const int F = (int)((br.r1 - br.r0) * Ts);
  const WarpRange wr = warp_range<NW>(F, warp);
  const int sb = (int)wr.sb, se = (int)wr.se;
  const int nfull = (se - sb) / U;

  const int row0 = sb / Ts, t0 = sb - row0 * Ts;
  const int64_t g = (br.r0 + row0) * (int64_t)p.steps + ts0 + t0;  // first step, global
  const uint32_t* mp = p.masks + g * 32 + lane;
  const uint32_t* vp = p.values + (g * 32 + lane) * 8;
  int lt = t0;

  SpmmBatch<U> A, B;
  pdl_launch_dependents();
  if (!p.early_weights) pdl_wait_previous();
  if (nfull > 0) load_steps_batch<U, SLICED>(A, vp, mp, lt, Ts, skip);
  if (p.early_weights) pdl_wait_previous();  // X (and Y, the workspace) may be the previous kernel's
  stage_x_slice<BP, kF32>(smem, p, P, ts0 * 32, (ts0 + Ts) * 32, NW * 32);
  __syncthreads();

  const uint32_t row_bytes = (uint32_t)P * kSlotWords * 4u;
  const uint32_t swz = ((lane >> 2) & 1) ? 16u : 0u;  // local word bit 2 == lane bit 2
  const uint32_t lane_col = smem_addr(tile) + row_bytes + (uint32_t)lane * (kSlotWords * 4u);
  constexpr uint32_t kStepBytes = 32u * kSlotWords * 4u;  // 32 words of slots
  // one token's sum of local row `row`: Y, or this slice's fp32 partial
  auto put = [&](int row, int j, float v) {
    const int64_t gr = br.r0 + row;
    if (!SLICED)
      p.Y[(int64_t)j * p.ldy + gr] = __float2half_rn(v);
    else
      p.partial[((int64_t)sl * p.batch + j) * p.rows + gr] = v;
  };
  auto store = [&](int row, const float (&v)[BP]) {  // the cut-row combine: all tokens
#pragma unroll
    for (int j = 0; j < BP; ++j)
      if (j < p.batch) put(row, j, v[j]);
  };

  int row = row0, t = t0;
  uint32_t col_addr = lane_col + kStepBytes * (uint32_t)t;
  float a[2][BP];                    // XF 0, 2, 3
  unsigned long long a2[2][BP / 2];  // XF 1: packed pairs of tokens
#pragma unroll
  for (int j = 0; j < BP; ++j) a[0][j] = a[1][j] = 0.f;
#pragma unroll
  for (int q = 0; q < BP / 2; ++q) a2[0][q] = a2[1][q] = 0ull;

  // A row's sums: reduced across the warp, each token's total on its own
  // lane, which stores it (whole row) or keeps it as a cut-row partial.
  auto finish = [&](bool whole) {
    float v[BR];
#pragma unroll
    for (int j = 0; j < BP; ++j) {
      v[j] = XF == 1 ? ((j & 1) ? pair_hi(a2[0][j >> 1]) + pair_hi(a2[1][j >> 1])
                                : pair_lo(a2[0][j >> 1]) + pair_lo(a2[1][j >> 1]))
                     : a[0][j] + a[1][j];
      a[0][j] = a[1][j] = 0.f;
    }
#pragma unroll
    for (int j = BP; j < BR; ++j) v[j] = 0.f;
#pragma unroll
    for (int q = 0; q < BP / 2; ++q) a2[0][q] = a2[1][q] = 0ull;
    const float total = warp_sum_tokens<BR>(v, lane);
    if (lane % kLanesPerToken == 0 && lane / kLanesPerToken < BP) {
      const int j = lane / kLanesPerToken;
      if (whole) {
        if (j < p.batch) put(row, j, total);
      } else {
        ((row == row0) ? pf : pl)[warp * BP + j] = total;
      }
    }
  };

  auto step = [&](uint32_t m, const uint32_t (&v)[8]) {
    if constexpr (XF == 1)
      decode_word_batch_f32<BP>(m, v, col_addr, row_bytes, swz, a2);
    else if constexpr (XF == 3)
      decode_word_batch_u<BP>(m, v, col_addr, row_bytes, a);
    else if constexpr (XF == 2)
      decode_word_batch_f32s<BP>(m, v, col_addr, row_bytes, swz, a);
    else
      decode_word_batch<BP>(m, v, col_addr, row_bytes, a);
    col_addr += kStepBytes;
    if (++t == Ts) {  // the row's slice complete
      finish(row != row0 || t0 == 0);
      t = 0;
      ++row;
      col_addr = lane_col;
    }
  };

  for (int i = 0; i < nfull; i += 2) {
    if (i + 1 < nfull) load_steps_batch<U, SLICED>(B, vp, mp, lt, Ts, skip);
#pragma unroll
    for (int u = 0; u < U; ++u) step(A.m[u], A.v[u]);
    if (i + 1 >= nfull) break;
    if (i + 2 < nfull) load_steps_batch<U, SLICED>(A, vp, mp, lt, Ts, skip);
#pragma unroll
    for (int u = 0; u < U; ++u) step(B.m[u], B.v[u]);
  }
  for (int s = sb + nfull * U; s < se; ++s) {
    SpmmBatch<1> one;
    load_steps_batch<1, SLICED>(one, vp, mp, lt, Ts, skip);
    step(one.m[0], one.v[0]);
  }
  if (se > sb && t != 0) finish(false);  // the warp's range ends inside a row
  note_range(rinfo, warp, lane, se > sb ? row0 : -1, t0 != 0, t != 0 ? row : row - 1, t != 0);

  __syncthreads();
  combine_cut_rows_n<NW, BP>(rinfo, pf, pl, store);
}

template <int NW, int U, int BP, int XF>
cudaError_t launch_spmm_t(const SpmmParams& p, int grid, int flags, cudaStream_t stream) {
  static int smem_set[64] = {0}, smem_full[64] = {0}, smem_sliced[64] = {0};
  const size_t smem = spmm_smem_bytes(p.pitch, NW, BP, XF);
  const int64_t block_steps = (p.rows_q + 2) * (int64_t)p.steps;
  if (p.words % 32 == 0 && block_steps < (int64_t)0x7FFFFFFF) {
    auto* k = p.slices == 1 ? spmm_full_kernel<NW, U, BP, XF, false>
                            : spmm_full_kernel<NW, U, BP, XF, true>;
    cudaError_t e = ensure_max_smem(reinterpret_cast<const void*>(k),
                                    p.slices == 1 ? smem_full : smem_sliced, 64);
    if (e != cudaSuccess) return e;
    return launch_kernel(k, grid, NW * 32, smem, stream, flags, p);
  }
  auto* k = spmm_kernel<NW, U, BP, XF>;
  cudaError_t e = ensure_max_smem(reinterpret_cast<const void*>(k), smem_set, 64);
  if (e != cudaSuccess) return e;
  return launch_kernel(k, grid, NW * 32, smem, stream, flags, p);
}

// One x-slot width, every variant (6-token slots exist for fp16 slots only).
template <int BP>
cudaError_t launch_spmm_variant(const SpmmParams& p, int variant, int grid, int flags,
                                cudaStream_t stream) {
  switch (variant) {
#define NM_SPMM_CASE(i)                                                              \
  case i:                                                                           \
    if constexpr (BP == 6 && kSpmmVariants[i][2] != 0) return cudaErrorInvalidValue; \
    else                                                                            \
      return launch_spmm_t<kSpmmVariants[i][0], kSpmmVariants[i][1], BP,             \
                           kSpmmVariants[i][2]>(p, grid, flags, stream);
    NM_SPMM_CASE(0) NM_SPMM_CASE(1) NM_SPMM_CASE(2) NM_SPMM_CASE(3) NM_SPMM_CASE(4)
    NM_SPMM_CASE(5) NM_SPMM_CASE(6) NM_SPMM_CASE(7) NM_SPMM_CASE(8) NM_SPMM_CASE(9)
#undef NM_SPMM_CASE
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nmk
