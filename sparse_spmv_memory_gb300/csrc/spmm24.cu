// spmm24.cu -- small-batch SpMM, Y = W X for 1..8 tokens, when W's masks are
// 2:4 (every aligned group of four columns keeps exactly two), on the tensor
// cores with register operands (sm_103a).
//
// Why a separate kernel.  The CUDA-core SpMM (spmm_kernels.cuh) gathers, for
// every kept weight, the batch's x values at that weight's column from shared
// memory: 16 bytes per nonzero per lane at 8 tokens, which keeps the
// L1/shared-memory pipe ~92 % busy and the weight stream at ~64 % of HBM.
// With 2:4 masks the compact values are already aligned to the groups: the
// two values of group i of a mask word are exactly the 32-bit pair i of the
// word's 16 values.  A group's four dense columns are therefore two byte
// permutes of that one register (the group's 4 mask bits pick the selectors
// from a 16-entry table), with no data-dependent register index.  That makes
// a dense 16 x 16 fp16 A operand cheap to build in registers, and
// mma.sync.m16n8k16 (fp16 x fp16, fp32 accumulate) multiplies it with the 8
// tokens' x: x is read once per 16 rows instead of once per nonzero.
// tcgen05.mma would need A in shared or tensor memory (a store, a fence and a
// barrier per step between the lanes that build it and the thread that
// issues); here the operands never leave the registers of the warp that
// builds them, and the tensor pipe is 9-14 % busy: the weight loads in
// flight bound the kernel.
//
// Work and layout.  Rows are taken 16 at a time ("panels"); a panel is
// walked in units of 4 mask words (128 columns).  Lane l = 4g + q holds rows
// g and g + 8 of the panel and, in each unit, word 4c + q of both rows (one
// 32-byte load each: the 4 lanes of a group read one 128-byte line).  In the
// MMA for group i (i = 0..7) the k slots 2q, 2q+1 are columns 4i, 4i+1 of that
// word and k slots 2q+8, 2q+9 are columns 4i+2, 4i+3, for every g: A and B
// agree on every k, so the 8 MMAs of a unit cover its 128 columns.  The B
// operand (token g, the same columns) comes from a copy of x that every block
// writes into its shared memory in exactly that order first, so a warp's x
// loads for a unit are four conflict-free 512-byte reads.  When x (16 bytes
// per column) would take more than 128 KB, the columns are cut into slices,
// each taken by its own group of blocks.  Within a slice the flattened
// (panel, unit) sequence is cut evenly over the slice's blocks, and each
// block's range evenly over its warps (split_at), whatever the shape.  A
// panel that one warp holds whole (and that is not sliced) goes straight to
// y.  A panel cut between warps of a block is summed after one block barrier
// from the warps' shared-memory partials, in warp order.  Panels cut by a
// block boundary, and all panels of a sliced matrix, go through the
// workspace: the block's fp32 partial, then its unit count on the panel's
// counter; the warp that completes the count adds the partials slice by
// slice in block order and rounds to fp16.  The order does not depend on
// which warp finishes last (deterministic), and no warp waits for another.
// That warp also sets the partials and the counter back to zero, so the
// workspace is all zero between calls.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device.cuh"
#include "kernels.h"
#include "split.cuh"

namespace nmk {

// Byte-permute selectors that expand one 2:4 group.  For the group's mask
// nibble n, the k-th set column (k = 0, 1) takes half k of the group's value
// pair, every other column +0 (selector byte 4: the zero second operand).
// Low 16 bits: columns 0, 1 (one fp16 pair); high 16 bits: columns 2, 3.  A
// nibble with more than two set bits (not 2:4) gives its third and fourth
// columns +0, so a malformed word is still decoded in bounds.
__host__ __device__ constexpr uint32_t group_selectors(uint32_t nibble) {
  uint32_t sel = 0;
  uint32_t k = 0;
  for (uint32_t j = 0; j < 4; ++j) {
    uint32_t lo = 4, hi = 4;
    if ((nibble >> j) & 1u) {
      if (k < 2) {
        lo = 2 * k;
        hi = 2 * k + 1;
      }
      ++k;
    }
    sel |= (lo | (hi << 4)) << (16 * (j / 2) + 8 * (j % 2));
  }
  return sel;
}

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The weights of one unit for one lane: word 4c + q of rows g and g + 8.
struct Unit24 {
  uint32_t va[8], vb[8];
  uint32_t ma, mb;
};

// One column slice's share of the work: its units of every panel, flattened
// panel-major and cut evenly over the slice's blocks (and each block's range
// evenly over its warps).  Unit and panel indices fit 32 bits (the entry
// point refuses larger matrices); word indices may not.
struct Slice24 {
  int s;       // slice
  int c0;      // its first unit (128 columns each) within a panel
  int cs;      // its units per panel
  int64_t bq;  // panels * cs = bq * bps + br
  int br;
  int bps;     // blocks per slice

  __device__ __forceinline__ Slice24(const Spmm24Params& p, int slice) {
    s = slice;
    c0 = slice * p.cs;
    const bool last = slice + 1 == p.slices;
    cs = last ? p.units - c0 : p.cs;
    bq = last ? p.bq_last : p.bq;
    br = last ? p.br_last : p.br;
    bps = p.bps;
  }
  // first unit of block b of the slice
  __device__ __forceinline__ int at(int b) const { return (int)split_at(b, bq, br, bps); }
  // the block whose range holds unit u (ranges may be empty)
  __device__ __forceinline__ int owner(int u) const {
    const int64_t F = bq * bps + br;
    return (int)(((int64_t)(u + 1) * bps - 1) / F);
  }
};

// Where a lane's loads for a unit come from: the word index (row * words +
// word) of rows g and g + 8.  Rows past the end read the last row and use a
// zero mask (their columns expand to +0).
struct Cursor24 {
  int panel;
  int c;  // unit within the slice
  int64_t ia, ib;
  bool za, zb;  // rows in range

  __device__ __forceinline__ void seek(const Spmm24Params& p, const Slice24& sl, int pan, int cc,
                                       int g, int q) {
    panel = pan;
    c = cc;
    const int64_t ra = (int64_t)pan * 16 + g, rb = ra + 8;
    za = ra < p.rows;
    zb = rb < p.rows;
    const int64_t w = 4 * (sl.c0 + cc) + q;
    ia = (za ? ra : p.rows - 1) * p.words + w;
    ib = (zb ? rb : p.rows - 1) * p.words + w;
  }

  __device__ __forceinline__ void next(const Spmm24Params& p, const Slice24& sl, int g, int q) {
    if (c + 1 < sl.cs) {
      ++c;
      ia += 4;
      ib += 4;
    } else {
      seek(p, sl, panel + 1, 0, g, q);
    }
  }
};

// Weight loads.  A unit reads 128 bytes of values and 16 bytes of masks per
// row and the next unit of the same rows follows, so the loads ask L2 to
// fetch 256-byte pieces (.L2::256B): half as many separate DRAM accesses per
// row.  Values are read once (no L1 allocation, evict first in L2).
__device__ __forceinline__ void ld_values24(const uint32_t* p, uint32_t (&v)[8]) {
  asm volatile(
      "ld.global.nc.L1::no_allocate.L2::evict_first.L2::256B.v8.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7])
      : "l"(p));
}

__device__ __forceinline__ uint32_t ld_mask24(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ void load_weights24(const Spmm24Params& p, const Cursor24& cur,
                                               Unit24& u) {
  ld_values24(p.values + cur.ia * 8, u.va);
  ld_values24(p.values + cur.ib * 8, u.vb);
  u.ma = ld_mask24(p.masks + cur.ia);
  u.mb = ld_mask24(p.masks + cur.ib);
  if (!cur.za) u.ma = 0;
  if (!cur.zb) u.mb = 0;
}

// The 8 MMAs of one unit, group i into accumulator set i % A (A independent
// chains instead of one chain of 8 dependent MMAs).  x holds this unit's x
// (four 16-byte chunks); each chunk is reloaded from the block's shared copy
// with the next unit's as soon as its two MMAs have read it (next ==
// nullptr: no next unit), so x needs no second set of registers.
template <int A>
__device__ __forceinline__ void mma_unit24(const Unit24& u, uint4 (&x)[4], const uint4* next,
                                           const uint32_t* sel, float (&acc)[A][4]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t ta = sel[(u.ma >> (4 * i)) & 15u];
    const uint32_t tb = sel[(u.mb >> (4 * i)) & 15u];
    const uint32_t a0 = __byte_perm(u.va[i], 0u, ta);
    const uint32_t a1 = __byte_perm(u.vb[i], 0u, tb);
    const uint32_t a2 = __byte_perm(u.va[i], 0u, ta >> 16);
    const uint32_t a3 = __byte_perm(u.vb[i], 0u, tb >> 16);
    const uint4 xc = x[i >> 1];
    const uint32_t b0 = (i & 1) ? xc.z : xc.x;
    const uint32_t b1 = (i & 1) ? xc.w : xc.y;
    mma_16816(acc[i % A], a0, a1, a2, a3, b0, b1);
    if ((i & 1) && next) x[i >> 1] = next[32 * (i >> 1)];
  }
}

// Rounds a warp's sums of panel `panel` (lane 4g+q: rows g and g + 8, tokens
// 2q and 2q+1) to fp16 and stores them.  The 8 x 16 values go through the
// warp's 256-byte stage in shared memory so that each lane then writes 4
// consecutive rows of one token: a token's 16 rows are one 32-byte sector
// written by a single instruction (2-byte stores from 8 lanes split it in
// two, and partly written sectors of y that are not in L2 cost a DRAM read).
// Every lane of the warp calls it.
__device__ __forceinline__ void store_panel24(const Spmm24Params& p, int panel, int lane, float s0,
                                              float s1, float s2, float s3, __half* stage) {
  const int g = lane >> 2, q = lane & 3;
  stage[(2 * q) * 16 + g] = __float2half_rn(s0);
  stage[(2 * q + 1) * 16 + g] = __float2half_rn(s1);
  stage[(2 * q) * 16 + g + 8] = __float2half_rn(s2);
  stage[(2 * q + 1) * 16 + g + 8] = __float2half_rn(s3);
  __syncwarp();
  const int t = lane >> 2, r = 4 * (lane & 3);
  const int64_t row = (int64_t)panel * 16 + r;
  if (t < p.batch) {
    __half* y = p.Y + t * p.ldy + row;
    const __half* src = stage + t * 16 + r;
    if (p.y_vec && row + 3 < p.rows) {
      *reinterpret_cast<uint2*>(y) = *reinterpret_cast<const uint2*>(src);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (row + i < p.rows) y[i] = src[i];
    }
  }
  __syncwarp();
}

// Workspace slot `slot` (0: the block's first panel, 1: its last) of the
// grid's block `blk`: a panel cut by the block's range.
__device__ __forceinline__ float4* block_slot24(const Spmm24Params& p, int blk, int slot,
                                                int lane) {
  return p.part + ((int64_t)blk * 2 + slot) * 32 + lane;
}

// The slot of a panel that one block holds whole within slice s (column
// slices only): a block may hold any number of those.
__device__ __forceinline__ float4* slice_slot24(const Spmm24Params& p, int s, int panel,
                                                int lane) {
  return p.part_sp + ((int64_t)s * p.panels + panel) * 32 + lane;
}

// Counts `mine` units of a panel whose partial this warp has stored in the
// workspace (behind a fence).  Returns true if that completed the panel: the
// caller then adds the partials (combine_panel24).  Nothing waits on another
// warp.
__device__ __forceinline__ bool arrive_panel24(const Spmm24Params& p, int mine, int panel,
                                               int lane) {
  int old = 0;
  if (lane == 0) old = atomicAdd(p.cnt + panel, mine);
  old = __shfl_sync(0xFFFFFFFFu, old, 0);
  return old + mine == p.units;
}

__device__ __forceinline__ void add4(float4& a, const float4& b) {
  a.x += b.x;
  a.y += b.y;
  a.z += b.z;
  a.w += b.w;
}

// Adds a completed panel's workspace partials -- slice by slice, and within
// a slice in block order: the same order whichever warp completed it --
// rounds and stores it.  Every partial it reads and the panel's counter are
// set back to zero, so the workspace is all zero again when the call ends.
__device__ __forceinline__ void combine_panel24(const Spmm24Params& p, int panel, int lane,
                                                __half* stage) {
  __threadfence();
  float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int si = 0; si < p.slices; ++si) {
    const Slice24 sl(p, si);
    const int pb = panel * sl.cs, pe = pb + sl.cs;
    int B = sl.owner(pb);
    if (sl.owner(pe - 1) == B) {  // one block held this slice of the panel whole
      float4* at = slice_slot24(p, si, panel, lane);
      add4(sum, __ldcg(at));
      __stcg(at, zero);
      continue;
    }
    // 4 blocks at a time: all loads of a batch are issued before the first add
    int v0 = sl.at(B);
    while (v0 < pe) {
      float4 t[4];
      float4* at[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int v1 = sl.at(B + 1);
        at[j] = nullptr;
        if (v0 < pe && v1 > v0)
          at[j] = block_slot24(p, si * sl.bps + B, v0 / sl.cs == panel ? 0 : 1, lane);
        t[j] = at[j] ? __ldcg(at[j]) : zero;
        if (v0 < pe) {
          ++B;
          v0 = v1;
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (at[j]) {
          add4(sum, t[j]);
          __stcg(at[j], zero);
        }
    }
  }
  store_panel24(p, panel, lane, sum.x, sum.y, sum.z, sum.w, stage);
  if (lane == 0) p.cnt[panel] = 0;
}

// Y = W X for one column slice per group of p.bps blocks.  Every block first
// writes its slice's x into shared memory in MMA operand order -- chunk
// (4c + j) * 32 + l (16 bytes) is token l / 4's x at columns
// 32 (4c + l % 4) + 8j .. + 7 of unit c, tokens past the batch +0 -- so a
// warp's x loads for a unit are four conflict-free 512-byte shared reads.
// Behind x, each warp has two 512-byte partial slots (its first and last
// panel) for panels cut between warps of the block, and a 256-byte stage for
// the panels it stores.
template <int NW, int U, int A>
__global__ void __launch_bounds__(NW * 32, 1) spmm24_kernel(const Spmm24Params p) {
  __shared__ uint32_t sel[16];
  extern __shared__ uint4 xs24[];
  pdl_launch_dependents();
  if (threadIdx.x < 16) sel[threadIdx.x] = group_selectors(threadIdx.x);
  if (!p.early_weights) pdl_wait_previous();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int slice = blockIdx.x / p.bps;
  const Slice24 sl(p, slice);
  const int b = blockIdx.x - slice * p.bps;  // block within the slice
  const int b0 = sl.at(b), b1 = sl.at(b + 1);
  const int64_t nb = b1 - b0;
  const int u0 = b0 + (int)(nb * warp / NW), u1 = b0 + (int)(nb * (warp + 1) / NW);
  const int n = u1 - u0;
  const int C = sl.cs;
  const int p_first = u0 / C;
  const int c_first = u0 - p_first * C;
  float4* wslot = reinterpret_cast<float4*>(xs24 + (size_t)p.cs * 128);  // [NW][2][32]
  __half* stage = reinterpret_cast<__half*>(wslot + NW * 64) + warp * 128;  // [NW][8][16]

  Unit24 buf[U];
  Cursor24 ld;
  if (n > 0) {
    ld.seek(p, sl, p_first, c_first, g, q);
#pragma unroll
    for (int s = 0; s < U; ++s)
      if (s < n) {
        load_weights24(p, ld, buf[s]);
        ld.next(p, sl, g, q);
      }
  }
  if (p.early_weights) pdl_wait_previous();
  {
    // 8 loads per thread in flight before the first store: x may come from
    // DRAM (a layer's activations are not always still in L2)
    const int nk = C * 128;
    const __half* X = p.X + 32 * 4 * sl.c0;
    constexpr int kB = 8;
    for (int k0 = threadIdx.x; k0 < nk; k0 += kB * NW * 32) {
      uint4 v[kB];
#pragma unroll
      for (int t = 0; t < kB; ++t) {
        const int k = k0 + t * NW * 32;
        const int l = k & 31, j = (k >> 5) & 3, c = k >> 7;
        const int gg = l >> 2, qq = l & 3;
        v[t] = make_uint4(0u, 0u, 0u, 0u);
        if (k < nk && gg < p.batch) v[t] = ld_keep_v4(X + gg * p.ldx + 32 * (4 * c + qq) + 8 * j);
      }
#pragma unroll
      for (int t = 0; t < kB; ++t) {
        const int k = k0 + t * NW * 32;
        if (k < nk) xs24[k] = v[t];
      }
    }
  }
  __syncthreads();

  bool counted = false;  // this warp stored a whole panel's partial in the workspace
  if (n > 0) {
    // x runs one unit ahead of the products, the weights U units ahead
    uint4 x[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] = xs24[c_first * 128 + 32 * j + lane];
    int cx = c_first + 1 == C ? 0 : c_first + 1;  // the unit whose x loads next

    float acc[A][4];
#pragma unroll
    for (int a = 0; a < A; ++a) acc[a][0] = acc[a][1] = acc[a][2] = acc[a][3] = 0.f;
    int panel = p_first;
    int c = c_first;
    for (int k = 0; k < n; k += U) {
#pragma unroll
      for (int s = 0; s < U; ++s) {
        if (k + s < n) {
          const uint4* next = nullptr;
          if (k + s + 1 < n) {
            next = xs24 + cx * 128 + lane;
            cx = cx + 1 == C ? 0 : cx + 1;
          }
          mma_unit24<A>(buf[s], x, next, sel, acc);
          if (k + s + U < n) {
            load_weights24(p, ld, buf[s]);
            ld.next(p, sl, g, q);
          }
          const bool last = k + s + 1 == n;
          if (c + 1 == C || last) {
            // the warp is done with this panel; the accumulator sets are
            // added in a fixed order
            float4 t = make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
#pragma unroll
            for (int a = 1; a < A; ++a) add4(t, make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]));
            const int pb = panel * C, pe = pb + C;
            if (pb >= u0 && pe <= u1) {  // whole in this warp
              if (p.slices == 1) {
                store_panel24(p, panel, lane, t.x, t.y, t.z, t.w, stage);
              } else {
                __stcg(slice_slot24(p, slice, panel, lane), t);
                counted = true;
              }
            } else {  // cut between warps or blocks: summed in the block first
              wslot[(warp * 2 + (panel == p_first ? 0 : 1)) * 32 + lane] = t;
            }
#pragma unroll
            for (int a = 0; a < A; ++a) acc[a][0] = acc[a][1] = acc[a][2] = acc[a][3] = 0.f;
            ++panel;
            c = 0;
          } else {
            ++c;
          }
        }
      }
    }
  }
  const int p_last = n > 0 ? (u1 - 1) / C : -1;
  if (counted) {  // column slices: count the panels this warp held whole
    __threadfence();
    __syncwarp();
    for (int pan = p_first; pan <= p_last; ++pan) {
      const int pb = pan * C, pe = pb + C;
      if (pb >= u0 && pe <= u1 && arrive_panel24(p, C, pan, lane)) combine_panel24(p, pan, lane, stage);
    }
  }
  __syncthreads();
  if (n <= 0) return;
  // Each panel cut between warps of this block (or by the block's range) is
  // summed by its first contributing warp: the partials of the warps it
  // spans, in warp order.
  for (int e = 0; e < 2; ++e) {
    const int pan = e == 0 ? p_first : p_last;
    if (e == 1 && p_last == p_first) break;
    const int pb = pan * C, pe = pb + C;
    if (pb >= u0 && pe <= u1) continue;                   // whole in this warp
    if (e == 0 && !(pb == u0 || u0 == b0)) continue;      // began in an earlier warp
    float4 t = wslot[(warp * 2 + e) * 32 + lane];
    const int end = pe < b1 ? pe : b1;
    for (int v = warp + 1; v < NW; ++v) {
      const int v0 = b0 + (int)(nb * v / NW), v1 = b0 + (int)(nb * (v + 1) / NW);
      if (v0 >= end) break;
      if (v1 > v0) add4(t, wslot[(v * 2 + 0) * 32 + lane]);  // pan is warp v's first panel
    }
    if (pb >= b0 && pe <= b1 && p.slices == 1) {  // whole in this block
      store_panel24(p, pan, lane, t.x, t.y, t.z, t.w, stage);
      continue;
    }
    float4* dst = (pb >= b0 && pe <= b1) ? slice_slot24(p, slice, pan, lane)
                                         : block_slot24(p, blockIdx.x, pan == b0 / C ? 0 : 1, lane);
    __stcg(dst, t);
    __threadfence();
    __syncwarp();
    const int mine = (b1 < pe ? b1 : pe) - (b0 > pb ? b0 : pb);
    if (arrive_panel24(p, mine, pan, lane)) combine_panel24(p, pan, lane, stage);
  }
}

// (warps per block, units in flight per warp, accumulator sets).  Measured on
// the 70B layer's four matrices at 8 tokens, the step totals of 0, 1 and 4
// are within 0.5 % of each other; 1 is the default.
inline constexpr int kSpmm24Variants[][3] = {{16, 3, 2}, {20, 1, 4}, {16, 2, 1}, {12, 4, 2},
                                            {24, 1, 4}, {20, 2, 1}};
inline constexpr int kSpmm24VariantCount = sizeof(kSpmm24Variants) / sizeof(kSpmm24Variants[0]);

int spmm24_variant_count() { return kSpmm24VariantCount; }

int spmm24_variant_warps(int variant) {
  return (variant >= 0 && variant < kSpmm24VariantCount) ? kSpmm24Variants[variant][0] : 0;
}

// Column slices: the fewest whose x (16 bytes per column) fits 128 KB of a
// block's shared memory.  The rest of the SM's 256 KB of L1/shared memory
// holds the weight loads in flight; with x filling all of it (the 70B down
// projection as two 224 KB slices) the weight stream ran at ~55 % of HBM.
int spmm24_slices(int units, size_t smem_optin) {
  // room for the selector table and up to 32 warps' partial slots and stages
  int64_t per = ((int64_t)smem_optin - 256 - 40 * 1024) / 2048;  // units of x per block
  if (per > 64) per = 64;
  if (per < 1) return 0;
  return (int)((units + per - 1) / per);
}

size_t spmm24_workspace_bytes(int grid, int64_t panels, int slices) {
  return (size_t)grid * 2 * 32 * sizeof(float4) +
         (slices > 1 ? (size_t)slices * panels * 32 * sizeof(float4) : 0) +
         (size_t)(panels + 3) / 4 * 16;
}

// Lets `fn` take as much dynamic shared memory as the device allows next to
// its static shared memory (the selector table), once per device.
static cudaError_t allow_dynamic_smem24(const void* fn, int* done_flags) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && __atomic_load_n(&done_flags[dev], __ATOMIC_ACQUIRE)) return cudaSuccess;
  int optin = 0;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes a;
  e = cudaFuncGetAttributes(&a, fn);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           optin - (int)a.sharedSizeBytes);
  if (e == cudaSuccess && dev < 64) __atomic_store_n(&done_flags[dev], 1, __ATOMIC_RELEASE);
  return e;
}

template <int NW, int U, int A>
static cudaError_t launch24(const Spmm24Params& p, int grid, size_t smem, int flags,
                            cudaStream_t stream) {
  static int done[64];
  cudaError_t e =
      allow_dynamic_smem24(reinterpret_cast<const void*>(spmm24_kernel<NW, U, A>), done);
  if (e != cudaSuccess) return e;
  return launch_kernel(spmm24_kernel<NW, U, A>, grid, NW * 32, smem, stream, flags, p);
}

// grid: blocks per slice * slices (the caller rounds it).
cudaError_t launch_spmm24(const Spmm24Params& p0, int variant, int grid, int flags,
                          cudaStream_t stream) {
  if (variant < 0 || variant >= kSpmm24VariantCount || p0.slices < 1 || grid < p0.slices ||
      grid % p0.slices)
    return cudaErrorInvalidValue;
  const int nw = kSpmm24Variants[variant][0];
  Spmm24Params p = p0;
  p.bps = grid / p.slices;
  const int64_t F = p.panels * p.cs, Fl = p.panels * (p.units - (p.slices - 1) * p.cs);
  p.bq = F / p.bps;
  p.br = (int)(F % p.bps);
  p.bq_last = Fl / p.bps;
  p.br_last = (int)(Fl % p.bps);
  const size_t smem = (size_t)p.cs * 128 * sizeof(uint4) + (size_t)nw * 2 * 32 * sizeof(float4) +
                      (size_t)nw * 128 * sizeof(__half);
  switch (variant) {
    case 0: return launch24<16, 3, 2>(p, grid, smem, flags, stream);
    case 1: return launch24<20, 1, 4>(p, grid, smem, flags, stream);
    case 2: return launch24<16, 2, 1>(p, grid, smem, flags, stream);
    case 3: return launch24<12, 4, 2>(p, grid, smem, flags, stream);
    case 4: return launch24<24, 1, 4>(p, grid, smem, flags, stream);
    case 5: return launch24<20, 2, 1>(p, grid, smem, flags, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nmk
