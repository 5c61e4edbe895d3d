// spmm_variants.h -- the small-batch SpMM kernel variants, shared by the
// launch units and the plan.
#pragma once

namespace nmk {

// (warps per block, steps in flight per warp, x slot format).  At batch 8
// the kernel is issue-bound: 8 FMAs per nonzero per lane put a warp-step at
// ~300 instructions (ncu, 70B gate+up, general kernel: issue 78 % busy,
// shared-memory pipe 87 % busy from the 16-byte x gather per nonzero); the
// whole-step kernel's unpredicated walk and split-level token reduction
// raise it from ~55 % to ~61 % of the HBM rate there.  XF 3 helped the
// general kernel by 1-2 % at batch 4 only and is slower in the whole-step
// kernel.
// fp32 slots (XF 1: packed fp32x2 FMA; XF 2: scalar FMA) measured 1.5-1.7x
// slower than fp16 slots at batch 4-8 on GB300: every nonzero gathers
// BP x-values from shared memory per lane, so at batch 8 the gather already
// needs 16 B per nonzero with fp16 slots and twice that with fp32 slots --
// shared-memory bandwidth, not FMA issue, is the limit there.  They stay
// available for tuning; the defaults use fp16 slots.
inline constexpr int kSpmmVariants[][3] = {{16, 2, 0}, {20, 2, 0}, {12, 3, 0}, {24, 1, 0},
                                       {16, 2, 1}, {16, 2, 2}, {16, 2, 3}, {20, 2, 3},
                                       {24, 1, 3}, {12, 3, 3}};


inline constexpr int kSpmmVariantCount = sizeof(kSpmmVariants) / sizeof(kSpmmVariants[0]);

}  // namespace nmk
