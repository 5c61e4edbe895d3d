// device.cuh -- small inline-PTX helpers shared by the sm_103a kernels.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace nmk {

// 256-bit read-only streaming load (one mask word's 16 fp16 values).
// Weights are read exactly once per call, so they bypass L1 and are marked
// evict-first in L2 to leave room for x and y (PTX accepts the L2 eviction
// hint on 256-bit loads only; the narrower loads below skip L1 alone).
__device__ __forceinline__ void ld_stream_v8(const uint32_t* p, uint32_t (&v)[8]) {
  asm volatile(
      "ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7])
      : "l"(p));
}

__device__ __forceinline__ uint32_t ld_stream_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Read-only load that may stay in L1/L2 (x is reused by every block).
__device__ __forceinline__ uint4 ld_keep_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 256-bit read-only load that may stay in L1/L2 (x staging; p 32-byte aligned).
__device__ __forceinline__ void ld_keep_v8(const uint32_t* p, uint32_t (&v)[8]) {
  asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
                 "=r"(v[7])
               : "l"(p));
}

// Mask of the b low bits, (1 << b) - 1; b >= 32 (and ~0u) gives all ones.
__device__ __forceinline__ uint32_t low_bits(uint32_t b) {
  uint32_t r;
  asm("bmsk.clamp.b32 %0, %1, %2;" : "=r"(r) : "r"(0u), "r"(b));
  return r;
}

// Index of the most significant set bit, or 0xFFFFFFFF when w == 0.
__device__ __forceinline__ uint32_t msb_index(uint32_t w) {
  uint32_t b;
  asm("bfind.u32 %0, %1;" : "=r"(b) : "r"(w));
  return b;
}

// 1 << b with the PTX clamp: shift counts >= 32 give 0.
__device__ __forceinline__ uint32_t bit_at(uint32_t b) {
  uint32_t r;
  asm("shl.b32 %0, %1, %2;" : "=r"(r) : "r"(1u), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t bit_reverse(uint32_t w) {
  uint32_t r;
  asm("brev.b32 %0, %1;" : "=r"(r) : "r"(w));
  return r;
}

__device__ __forceinline__ uint16_t lds_u16(uint32_t saddr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(saddr));
  return v;
}

__device__ __forceinline__ float lds_f32(uint32_t saddr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(saddr));
  return v;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// fp32 += fp16 * fp16 in one rounding (mixed-precision FMA, sm_100+).
__device__ __forceinline__ float fma_f16f16_f32(uint16_t a, uint16_t b, float c) {
  float d;
  asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(c));
  return d;
}

// Programmatic dependent launch: let the next kernel on the stream be
// scheduled as soon as SMs free up, and wait for the previous kernel's
// completion (and memory) before touching anything it may have written.
// Both are no-ops when the launch does not use the attribute.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait_previous() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t h2) {
  __half2 h = *reinterpret_cast<const __half2*>(&h2);
  return __half22float2(h);
}

}  // namespace nmk
