// pack.cu -- dense fp16 <-> N:M bitmask format, and the mask validator.
//
// Format (aimodeling.com article, "The Kernel Is the Other Half of the
// Answer"): one 32-bit mask word per 32 input columns, 16 set bits at 50%,
// with the 16 kept values of word w stored at the fixed offset 16*w of the
// row, in ascending column order.  Bit b of a word is column 32*w + b.
//
// Selection (the synthetic pruner standing in for the paper's offline
// SparseGPT pass): within each M-group keep the N = M/2 entries of largest
// key = fp16 bits & 0x7FFF (unsigned), the lower column winning a tie.
// Everything is integer work, so the output is bit-exact.
//
// One thread handles one mask word: it reads the 32 fp16 of its columns,
// ranks each entry inside its group (rank = entries that beat it), sets the
// mask bits of ranks < N, and compacts the kept values through a private
// 64-byte shared-memory slot (registers cannot be indexed by a data-dependent
// position).
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device.cuh"
#include "kernels.h"

namespace nmk {

static constexpr int kFormatThreads = 256;

template <int M, bool VEC>
__global__ void __launch_bounds__(kFormatThreads) pack_kernel(const uint16_t* __restrict__ W,
                                                              int64_t rows, int64_t words,
                                                              int64_t ld,
                                                              uint32_t* __restrict__ values,
                                                              uint32_t* __restrict__ masks) {
  __shared__ uint16_t slot[kFormatThreads * 34];  // 32 entries + 2 pad per thread
  uint16_t* my = slot + threadIdx.x * 34;
  const int64_t total = rows * words;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = g / words, w = g - r * words;
    const uint16_t* src = W + r * ld + 32 * w;
    uint16_t h[32];
    if (VEC) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = ld_stream_v4(src + 8 * q);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          h[8 * q + 2 * j] = (uint16_t)(u[j] & 0xFFFFu);
          h[8 * q + 2 * j + 1] = (uint16_t)(u[j] >> 16);
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) h[i] = src[i];
    }

    uint32_t mask = 0u;
#pragma unroll
    for (int g0 = 0; g0 < 32; g0 += M) {
#pragma unroll
      for (int i = 0; i < M; ++i) {
        const uint32_t ki = h[g0 + i] & 0x7FFFu;
        int rank = 0;
#pragma unroll
        for (int j = 0; j < M; ++j) {
          if (j == i) continue;
          const uint32_t kj = h[g0 + j] & 0x7FFFu;
          rank += (kj > ki || (kj == ki && j < i)) ? 1 : 0;
        }
        if (rank < M / 2) mask |= 1u << (g0 + i);
      }
    }

#pragma unroll
    for (int i = 0; i < 32; ++i) my[i] = h[i];
    uint32_t out[8];
    uint32_t m = mask;
#pragma unroll
    for (int k = 0; k < 16; k += 2) {
      const int b0 = __ffs(m) - 1;
      m &= m - 1u;
      const int b1 = __ffs(m) - 1;
      m &= m - 1u;
      out[k / 2] = (uint32_t)my[b0 & 31] | ((uint32_t)my[b1 & 31] << 16);
    }
    uint4* dst = reinterpret_cast<uint4*>(values + g * 8);
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
    masks[g] = mask;
  }
}

template <bool VEC>
__global__ void __launch_bounds__(kFormatThreads) unpack_kernel(const uint32_t* __restrict__ values,
                                                                const uint32_t* __restrict__ masks,
                                                                int64_t rows, int64_t words,
                                                                int64_t ld,
                                                                uint16_t* __restrict__ W) {
  __shared__ uint16_t slot[kFormatThreads * 18];  // 16 values + 2 pad per thread
  uint16_t* my = slot + threadIdx.x * 18;
  const int64_t total = rows * words;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = g / words, w = g - r * words;
    const uint32_t m = masks[g];
    const uint4* src = reinterpret_cast<const uint4*>(values + g * 8);
    const uint4 v0 = src[0], v1 = src[1];
    const uint32_t u[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      my[2 * j] = (uint16_t)(u[j] & 0xFFFFu);
      my[2 * j + 1] = (uint16_t)(u[j] >> 16);
    }
    uint16_t o[32];
    int k = 0;
#pragma unroll
    for (int b = 0; b < 32; ++b) {
      const bool set = (m >> b) & 1u;
      o[b] = set ? my[k & 15] : (uint16_t)0u;  // & 15 keeps corrupt words in bounds
      k += set ? 1 : 0;
    }
    uint16_t* dst = W + r * ld + 32 * w;
    if (VEC) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t t[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          t[j] = (uint32_t)o[8 * q + 2 * j] | ((uint32_t)o[8 * q + 2 * j + 1] << 16);
        reinterpret_cast<uint4*>(dst)[q] = make_uint4(t[0], t[1], t[2], t[3]);
      }
    } else {
#pragma unroll
      for (int b = 0; b < 32; ++b) dst[b] = o[b];
    }
  }
}

__global__ void __launch_bounds__(kFormatThreads) check_masks_kernel(
    const uint32_t* __restrict__ masks, int64_t n, unsigned long long* __restrict__ count) {
  unsigned bad = 0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    bad += (__popc(masks[i]) != 16) ? 1u : 0u;
  bad = __reduce_add_sync(0xFFFFFFFFu, bad);
  if ((threadIdx.x & 31) == 0 && bad) atomicAdd(count, (unsigned long long)bad);
}

static int format_grid(int64_t work) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t blocks = (work + kFormatThreads - 1) / kFormatThreads;
  const int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 8;
  return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

template <int M>
static void pack_dispatch(bool vec, int grid, cudaStream_t s, const uint16_t* W, int64_t rows,
                          int64_t words, int64_t ld, uint32_t* values, uint32_t* masks) {
  if (vec)
    pack_kernel<M, true><<<grid, kFormatThreads, 0, s>>>(W, rows, words, ld, values, masks);
  else
    pack_kernel<M, false><<<grid, kFormatThreads, 0, s>>>(W, rows, words, ld, values, masks);
}

cudaError_t launch_pack(const __half* W, int64_t rows, int64_t cols, int64_t ld, int M,
                        __half* values, uint32_t* masks, cudaStream_t stream) {
  const int64_t words = cols / 32;
  const bool vec = ((reinterpret_cast<uintptr_t>(W) & 15u) == 0) && (ld % 8 == 0);
  const int grid = format_grid(rows * words);
  const uint16_t* w16 = reinterpret_cast<const uint16_t*>(W);
  uint32_t* v32 = reinterpret_cast<uint32_t*>(values);
  switch (M) {
    case 4: pack_dispatch<4>(vec, grid, stream, w16, rows, words, ld, v32, masks); break;
    case 8: pack_dispatch<8>(vec, grid, stream, w16, rows, words, ld, v32, masks); break;
    case 16: pack_dispatch<16>(vec, grid, stream, w16, rows, words, ld, v32, masks); break;
    case 32: pack_dispatch<32>(vec, grid, stream, w16, rows, words, ld, v32, masks); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_unpack(const __half* values, const uint32_t* masks, int64_t rows,
                          int64_t cols, __half* W, int64_t ld, cudaStream_t stream) {
  const int64_t words = cols / 32;
  const bool vec = ((reinterpret_cast<uintptr_t>(W) & 15u) == 0) && (ld % 8 == 0);
  const int grid = format_grid(rows * words);
  const uint32_t* v32 = reinterpret_cast<const uint32_t*>(values);
  uint16_t* w16 = reinterpret_cast<uint16_t*>(W);
  if (vec)
    unpack_kernel<true><<<grid, kFormatThreads, 0, stream>>>(v32, masks, rows, words, ld, w16);
  else
    unpack_kernel<false><<<grid, kFormatThreads, 0, stream>>>(v32, masks, rows, words, ld, w16);
  return cudaGetLastError();
}

cudaError_t launch_check_masks(const uint32_t* masks, int64_t n_words,
                               unsigned long long* d_count, cudaStream_t stream) {
  const int grid = format_grid(n_words);
  check_masks_kernel<<<grid, kFormatThreads, 0, stream>>>(masks, n_words, d_count);
  return cudaGetLastError();
}

}  // namespace nmk
