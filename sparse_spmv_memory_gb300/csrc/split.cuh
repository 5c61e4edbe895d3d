// split.cuh -- how a matrix-vector launch divides its rows among blocks and
// warps, and how rows cut between warps are summed back in a fixed order.
//
// Every block owns a contiguous, balanced range of rows [r0, r1) (sizes
// differ by at most one).  A row is T "steps" long (a step is what one warp
// reads in one go: 32 mask words for the sparse kernel, 512 columns for the
// dense one).  The block's nr*T steps, flattened row-major, are cut into NW
// contiguous ranges of equal length (+-1), one per warp, so every warp
// streams the same number of bytes whatever the shape.  A row that lies
// wholly inside one warp's range is finished by that warp; a row cut by a
// range boundary gets one partial sum per touching warp, and those are added
// in ascending warp order after a block barrier.  The result is therefore
// deterministic for a given shape and grid size.
#pragma once

#include <stdint.h>

#include "device.cuh"

namespace nmk {

struct BlockRows {
  int64_t r0, r1;
};

__device__ __forceinline__ BlockRows block_rows(int64_t rows) {
  const int64_t G = gridDim.x, c = blockIdx.x;
  return {rows * c / G, rows * (c + 1) / G};
}

// Pair-aligned variant: rows come in (gate, up) pairs that must stay in one
// block; the rows/2 pairs are balanced over the blocks.
__device__ __forceinline__ BlockRows block_row_pairs(int64_t rows) {
  const int64_t G = gridDim.x, c = blockIdx.x, H = rows / 2;
  return {2 * (H * c / G), 2 * (H * (c + 1) / G)};
}

struct WarpRange {
  int64_t sb, se;  // flattened steps [sb, se) of the block
};

template <int NW>
__device__ __forceinline__ WarpRange warp_range(int64_t F, int w) {
  return {F * w / NW, F * (w + 1) / NW};
}

// Called by every lane of a warp when it has summed its part of local row
// `row` (all lanes hold the same total `v` after warp_sum).  Rows wholly
// inside the warp's range are written to y; cut rows go to pf/pl.
template <typename Store>
__device__ __forceinline__ void finish_row(int64_t row, float v, const WarpRange& wr, int T,
                                           int warp, int lane, float* pf, float* pl,
                                           Store&& store) {
  if (lane != 0) return;
  const int64_t beg = row * T, end = beg + T;
  if (beg >= wr.sb && end <= wr.se) {
    store(row, v);
  } else if (row == wr.sb / T) {
    pf[warp] = v;
  } else {
    pl[warp] = v;
  }
}

// After a block barrier: thread t < NW adds up the row that warp t's range
// cuts at its end, if warp t is that row's first contributor.
template <int NW, typename Store>
__device__ __forceinline__ void combine_cut_rows(int64_t F, int T, const float* pf,
                                                 const float* pl, Store&& store) {
  const int t = threadIdx.x;
  if (t >= NW) return;
  const WarpRange wr = warp_range<NW>(F, t);
  if (wr.sb == wr.se) return;
  const int64_t rf = wr.sb / T, rl = (wr.se - 1) / T;
  const bool cut_at_end = (wr.se % T) != 0;
  const bool first_contributor = (rl != rf) || (wr.sb % T == 0);
  if (!(cut_at_end && first_contributor)) return;
  float sum = (rl == rf) ? pf[t] : pl[t];
  for (int u = t + 1; u < NW; ++u) {
    const WarpRange wu = warp_range<NW>(F, u);
    if (wu.sb == wu.se) continue;
    sum += pf[u];  // row rl is warp u's first row
    if (wu.se >= (rl + 1) * T) break;
  }
  store(rl, sum);
}

// The same two steps for N values per row (one per token of a batch):
// pf/pl hold N floats per warp, store receives the row and its N sums.
template <int N, typename Store>
__device__ __forceinline__ void finish_row_n(int64_t row, const float (&v)[N], const WarpRange& wr,
                                             int T, int warp, int lane, float* pf, float* pl,
                                             Store&& store) {
  if (lane != 0) return;
  const int64_t beg = row * T, end = beg + T;
  if (beg >= wr.sb && end <= wr.se) {
    store(row, v);
  } else {
    float* dst = (row == wr.sb / T) ? pf + warp * N : pl + warp * N;
#pragma unroll
    for (int j = 0; j < N; ++j) dst[j] = v[j];
  }
}

template <int NW, int N, typename Store>
__device__ __forceinline__ void combine_cut_rows_n(int64_t F, int T, const float* pf,
                                                   const float* pl, Store&& store) {
  const int t = threadIdx.x;
  if (t >= NW) return;
  const WarpRange wr = warp_range<NW>(F, t);
  if (wr.sb == wr.se) return;
  const int64_t rf = wr.sb / T, rl = (wr.se - 1) / T;
  const bool cut_at_end = (wr.se % T) != 0;
  const bool first_contributor = (rl != rf) || (wr.sb % T == 0);
  if (!(cut_at_end && first_contributor)) return;
  float sum[N];
  const float* own = (rl == rf) ? pf + t * N : pl + t * N;
#pragma unroll
  for (int j = 0; j < N; ++j) sum[j] = own[j];
  for (int u = t + 1; u < NW; ++u) {
    const WarpRange wu = warp_range<NW>(F, u);
    if (wu.sb == wu.se) continue;
#pragma unroll
    for (int j = 0; j < N; ++j) sum[j] += pf[u * N + j];  // row rl is warp u's first row
    if (wu.se >= (rl + 1) * T) break;
  }
  store(rl, sum);
}

}  // namespace nmk
