// spmm_variants.h -- the small-batch SpMM kernel variants, shared by the
// launch units and the plan.
#pragma once

namespace nmk {

// (warps per block, steps in flight per warp, x slot format).  At 8 tokens
// the kernel is bound by the L1/shared-memory data pipe: every nonzero
// gathers a 16-byte x slot per lane (64 of a warp-step's 66 shared-memory
// wavefronts; ncu on the 70B gate+up: pipe 92 % busy, ~64 % of the HBM rate;
// the general kernel, with predicated steps, ran at ~55 %).  12-byte slots
// (5-6 tokens) gather 48 and the kernel turns issue-bound (81 %).  XF 3
// (16-bit x registers inside the PTX) helped the general kernel by 1-2 % at
// 4 tokens only and is slower in the whole-step kernel.  fp32 slots (XF 1:
// packed fp32x2 FMA; XF 2: scalar FMA) measured 1.5-1.7x slower than fp16
// slots at 4-8 tokens on GB300: they halve the FMA instructions but double
// the gathered bytes.  They stay available for tuning; the defaults use fp16
// slots.
inline constexpr int kSpmmVariants[][3] = {{16, 2, 0}, {20, 2, 0}, {12, 3, 0}, {24, 1, 0},
                                           {16, 2, 1}, {16, 2, 2}, {16, 2, 3}, {20, 2, 3},
                                           {24, 1, 3}, {12, 3, 3}};

inline constexpr int kSpmmVariantCount = sizeof(kSpmmVariants) / sizeof(kSpmmVariants[0]);

}  // namespace nmk
