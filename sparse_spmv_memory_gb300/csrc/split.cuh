// split.cuh -- how a matrix-vector launch divides its rows among blocks and
// warps, and how rows cut between warps are summed back in a fixed order.
//
// Every block owns a contiguous, balanced range of rows [r0, r1) with
// r0 = floor(rows * c / blocks), so range sizes differ by at most one and the
// longer ranges are spread evenly over the grid.  A row is T "steps" long (a
// step is what one warp reads in one go: 32 mask words for the sparse kernels,
// 512 columns for the dense one).  The block's F = nr*T steps, flattened
// row-major, are cut into NW contiguous ranges at floor(F * w / NW), so every
// warp streams the same number of bytes (+-1 step) whatever the shape.  A row
// that lies wholly inside one warp's range is finished by that warp; a row cut
// by a range boundary gets one partial sum per touching warp, and those are
// added in ascending warp order after a block barrier.  The result is
// therefore deterministic for a given shape and grid size.
//
// Why floor(n * c / parts) and not "q each, the first r one more": with the
// latter, most concurrent streams start exactly q rows (or steps) apart, and
// on GB300 that regular spacing measured 3-5 % slower on the decoder shapes
// (the streams line up on the same DRAM channels); the floor formula's
// alternating spacing avoids it.
//
// Nothing here divides by a run-time value in 64 bits: such a division is a
// long software sequence on the GPU, and on the single thread that combines a
// block's cut rows it measured about half a microsecond per call.  Each warp records
// the rows its range touches (first and last row, cut at start / at end) in
// shared memory as it goes, and the combine reads those records.
#pragma once

#include <stdint.h>

#include "device.cuh"

namespace nmk {

struct BlockRows {
  int64_t r0, r1;
};

// floor(n * c / parts) for n = q * parts + r (q and r computed on the host):
// c * q + floor(c * r / parts), whose product c * r fits 32 bits for any grid
// of up to 65536 parts -- the plain formula's boundaries without its 64-bit
// division.
__device__ __forceinline__ int64_t split_at(int64_t c, int64_t q, int r, int parts) {
  const uint64_t cr = (uint64_t)c * (uint64_t)r;
  const uint64_t extra = cr <= 0xFFFFFFFFull ? (uint64_t)((uint32_t)cr / (uint32_t)parts)
                                             : cr / (uint64_t)parts;
  return c * q + (int64_t)extra;
}

// Part c of n = q * parts + r units.
__device__ __forceinline__ BlockRows split_part(int64_t c, int64_t q, int r, int parts) {
  return {split_at(c, q, r, parts), split_at(c + 1, q, r, parts)};
}

// This block's rows, for rows = q * gridDim.x + r.
__device__ __forceinline__ BlockRows block_rows(int64_t q, int r) {
  return split_part(blockIdx.x, q, r, (int)gridDim.x);
}

// Pair-aligned variant: rows come in (gate, up) pairs that must stay in one
// block; q and r split the rows/2 pairs.
__device__ __forceinline__ BlockRows block_row_pairs(int64_t q, int r) {
  const BlockRows b = block_rows(q, r);
  return {2 * b.r0, 2 * b.r1};
}

struct WarpRange {
  int64_t sb, se;  // flattened steps [sb, se) of the block
};

// NW is a compile-time constant, so these divisions become multiplications.
template <int NW>
__device__ __forceinline__ WarpRange warp_range(int64_t F, int w) {
  return {F * w / NW, F * (w + 1) / NW};
}

// a / T for a step index a and a row length T: a 32-bit division whenever a
// fits (always, for any matrix the entry points accept on a full grid).
__device__ __forceinline__ int64_t div_steps(int64_t a, int T) {
  return a <= 0x7FFFFFFF ? (int64_t)((uint32_t)a / (uint32_t)T) : a / T;
}

// Per-warp record of the rows a warp's range touches, kept in shared memory:
// rinfo[4w + 0] = first local row (-1: empty range), [4w + 1] = 1 if the range
// starts inside that row, [4w + 2] = last local row, [4w + 3] = 1 if the range
// ends inside it.  Written by lane 0 when the warp is done.
__device__ __forceinline__ void note_range(int* rinfo, int warp, int lane, int first, bool cut_start,
                                           int last, bool cut_end) {
  if (lane != 0) return;
  rinfo[4 * warp + 0] = first;
  rinfo[4 * warp + 1] = cut_start ? 1 : 0;
  rinfo[4 * warp + 2] = last;
  rinfo[4 * warp + 3] = cut_end ? 1 : 0;
}

// Called by every lane of a warp when it has summed its part of local row
// `row` (all lanes hold the same total `v` after warp_sum).  `whole`: the
// row both starts and ends inside the warp's range, so v is final and goes to
// y.  Otherwise v is a partial: the warp's first row's goes to pf, its last
// row's to pl.
template <typename Store>
__device__ __forceinline__ void finish_row(int row, float v, bool whole, int first_row, int warp,
                                           int lane, float* pf, float* pl, Store&& store) {
  if (lane != 0) return;
  if (whole)
    store(row, v);
  else if (row == first_row)
    pf[warp] = v;
  else
    pl[warp] = v;
}

// After a block barrier: thread t < NW adds up the row that warp t's range
// cuts at its end, if warp t is that row's first contributor (the row starts
// inside warp t's range); the following warps contribute their first-row
// partials, in warp order, up to the warp whose range reaches the row's end.
template <int NW, typename Store>
__device__ __forceinline__ void combine_cut_rows(const int* rinfo, const float* pf,
                                                 const float* pl, Store&& store) {
  const int t = threadIdx.x;
  if (t >= NW) return;
  const int first = rinfo[4 * t], cs = rinfo[4 * t + 1], last = rinfo[4 * t + 2],
            ce = rinfo[4 * t + 3];
  if (first < 0 || !ce) return;
  if (last == first && cs) return;  // the row started in an earlier warp
  float sum = (last == first) ? pf[t] : pl[t];
  for (int u = t + 1; u < NW; ++u) {
    if (rinfo[4 * u] < 0) continue;
    sum += pf[u];  // row `last` is warp u's first row
    if (!(rinfo[4 * u + 3] && rinfo[4 * u + 2] == last)) break;
  }
  store(last, sum);
}

// The same two steps for N values per row (one per token of a batch):
// pf/pl hold N floats per warp, store receives the row and its N sums.
template <int N, typename Store>
__device__ __forceinline__ void finish_row_n(int row, const float (&v)[N], bool whole,
                                             int first_row, int warp, int lane, float* pf,
                                             float* pl, Store&& store) {
  if (lane != 0) return;
  if (whole) {
    store(row, v);
  } else {
    float* dst = (row == first_row) ? pf + warp * N : pl + warp * N;
#pragma unroll
    for (int j = 0; j < N; ++j) dst[j] = v[j];
  }
}

template <int NW, int N, typename Store>
__device__ __forceinline__ void combine_cut_rows_n(const int* rinfo, const float* pf,
                                                   const float* pl, Store&& store) {
  const int t = threadIdx.x;
  if (t >= NW) return;
  const int first = rinfo[4 * t], cs = rinfo[4 * t + 1], last = rinfo[4 * t + 2],
            ce = rinfo[4 * t + 3];
  if (first < 0 || !ce) return;
  if (last == first && cs) return;
  float sum[N];
  const float* own = (last == first) ? pf + t * N : pl + t * N;
#pragma unroll
  for (int j = 0; j < N; ++j) sum[j] = own[j];
  for (int u = t + 1; u < NW; ++u) {
    if (rinfo[4 * u] < 0) continue;
#pragma unroll
    for (int j = 0; j < N; ++j) sum[j] += pf[u * N + j];
    if (!(rinfo[4 * u + 3] && rinfo[4 * u + 2] == last)) break;
  }
  store(last, sum);
}

}  // namespace nmk
