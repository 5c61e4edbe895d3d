// prefill.cu -- Y = W X for a prefill-sized batch of tokens, W in the N:M
// bitmask format (compact fp16 values + one 32-bit mask word per 32 input
// columns), on the sm_103a tensor cores.
//
// The operation is the pages' SpMM regime (aimodeling.com article, "The
// Kernel Is the Other Half of the Answer", and news.bitwarelabs.com summary,
// "What's new": prefill is compute-bound, decode is bandwidth-bound).  The
// packed format is the same one nm_spmv streams, so a model keeps one copy of
// its weights for both regimes.
//
// Design (this library's own; the pages give no prefill kernel):
//  * A block owns a tile of BM = 128 rows of W and BN = NB * NMMA tokens; its
//    fp32 accumulator D (128 x BN) lives in tensor memory, row m in TMEM lane
//    m.  K advances one mask word (32 columns) per pipeline stage.
//  * Producer warps, each a short chain of asynchronous copies per stage so
//    that they run side by side: warp 0 loads the token tile of X by TMA
//    (BN x 32 fp16, 64-byte swizzle); warp 2 loads the tile's compact values
//    (128 rows x 16 fp16) by TMA; the mask words come by TMA from a warp of
//    their own, four stages per box on a barrier of the box's own, when the
//    mask pitch allows it, else by cp.async from warp 2.  Values and X
//    complete on the stage's "full" mbarrier.
//  * Warps 3..18 (densify), in DG groups that take alternate stages: expand
//    each row's 16 kept values into the 32 columns of a K-major,
//    64-byte-swizzled fp16 tile in shared memory, the layout the MMA
//    descriptor names.  A lane builds four adjacent columns as two pairs:
//    the rank of a pair's first column among the word's set bits (popc)
//    indexes its value in the compact row; one table-driven prmt places it,
//    its neighbour or zeros.
//  * MMA: one thread (warp 1), or two taking the even and odd stages into two
//    accumulators, issues tcgen05.mma kind::f16 (M = 128, N = NMMA, K = 16;
//    two per stage and N-part) on the densified tile and the X tile, and
//    tcgen05.commit frees the stage when those MMAs are done.
//  * Epilogue (warps 3..18): tcgen05.ld of the accumulator, fp32 -> fp16 RNE,
//    stores to Y[t][r]; or, under a K split across blocks (grid z: each block
//    one slice of the row's mask words), fp32 stores of the slice's sums, which
//    splitk_sum_kernel adds in slice order.
//  * The stage barriers are rings sized so that every parity wait is exact
//    (see Layout).  Every mbarrier wait gives up after kWaitLimitNs (counted
//    in g_wait_timeouts); the roles then skip to teardown, which waits for the
//    copies and MMAs already issued before tensor memory is freed.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "device.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace nmk {
namespace tc {

constexpr int BM = 128;                // rows of W per block = TMEM lanes
constexpr int BK = 32;                 // K columns per stage = one mask word
constexpr int ROW_BYTES = BK * 2;      // 64-byte rows of the swizzled tiles
constexpr int A_BYTES = BM * ROW_BYTES;  // densified W tile
constexpr int V_BYTES = BM * 32;       // compact values: 16 fp16 per row
constexpr int M_BYTES = BM * 4;        // one mask word per row (cp.async ring)
constexpr int MW = 4;                  // mask words per TMA box (16 bytes per row)
constexpr int MT_SLOT = BM * MW * 4;   // 2 KiB: the masks of MW consecutive stages
// Densify warps per block (DW, a kernel parameter) follow the producer and
// MMA warps.  16 measured best on GB300: 8 left the per-stage chains
// exposed, 24 lost to the extra shared-memory and issue contention.
// After them: a second MMA issuer (used by the two-issuer variants) and the
// producer of the mask boxes.
constexpr int FIRST_DENSIFY_WARP = 3;
__host__ __device__ constexpr int mma2_warp(int dw) { return FIRST_DENSIFY_WARP + dw; }
__host__ __device__ constexpr int mask_warp(int dw) { return FIRST_DENSIFY_WARP + dw + 1; }
__host__ __device__ constexpr int threads_for(int dw) { return (FIRST_DENSIFY_WARP + dw + 2) * 32; }

constexpr uint32_t tmem_cols_for(int n) {
  return n <= 32 ? 32u : n <= 64 ? 64u : n <= 128 ? 128u : n <= 256 ? 256u : 512u;
}

// MT: masks arrive by TMA, MW stages' worth per box, into MT_SLOTS slots
// (needs the row pitch of the mask array, words * 4 bytes, to be a multiple
// of 16); otherwise by 4-byte cp.async into a per-stage ring.  A slot is
// refilled once every densify warp has released it (a barrier per slot);
// MW * MT_SLOTS >= STAGES + MW - 1 boxes in flight keep the box of every
// stage in the pipeline resident while the densify warps reach it.
// MS: 0, one thread issues every stage's MMAs; 1, two threads take the even
// and odd stages into two accumulators that the epilogue adds.
constexpr int gcd_int(int a, int b) { return b ? gcd_int(b, a % b) : a; }

template <int NMMA, int NB, int STAGES, int DG, int MS, bool MT>
struct Layout {
  static constexpr int BN = NMMA * NB;
  static constexpr int B_BYTES = BN * ROW_BYTES;
  static constexpr int A_OFF = 0;
  static constexpr int B_OFF = A_OFF + STAGES * A_BYTES;
  static constexpr int V_OFF = B_OFF + STAGES * B_BYTES;
  static constexpr int M_OFF = V_OFF + STAGES * V_BYTES;
  static constexpr int MT_SLOTS = (STAGES + MW - 1 + MW - 1) / MW;
  static constexpr int M_REGION = MT ? MT_SLOTS * MT_SLOT : STAGES * M_BYTES;
  // Stage barriers.  A parity wait tells a phase from the one before it only,
  // so it is exact only if the waiter itself saw the barrier's previous phase
  // complete.  The "full" barriers therefore form a ring of lcm(STAGES, DG):
  // all phases of one belong to stages of one densify group, which waits for
  // each.  The "afull" barriers form a ring of 2 * STAGES when two MMA
  // issuers split an odd STAGES, so all phases of one belong to one issuer.
  // The "empty" barriers, one per shared-memory slot, are waited by
  // producers that issue every stage.
  static constexpr int FULL_RING = STAGES * DG / gcd_int(STAGES, DG);
  static constexpr int AFULL_RING = (MS && STAGES % 2) ? 2 * STAGES : STAGES;
  // barriers: full (ring), empty (per slot), afull (ring), accum, mfull,
  // mfree (per mask slot)
  static constexpr int BAR_OFF = M_OFF + M_REGION;
  static constexpr int N_BARS = FULL_RING + STAGES + AFULL_RING + 1 + 2 * MT_SLOTS;
  static constexpr int SLOT_OFF = BAR_OFF + N_BARS * 8;
  static constexpr int BYTES = SLOT_OFF + 16;
  static constexpr int SMEM = BYTES + 1024;  // room to align the base to 1024
  static constexpr uint32_t TMEM_COLS = tmem_cols_for(MS ? 2 * BN : BN);
  static_assert(!MS || 2 * BN <= 512, "two issuers keep two accumulators in tensor memory");
  static_assert(!MT || MW * MT_SLOTS >= STAGES + MW - 1, "mask slot reused too early");
  static_assert(NMMA % 16 == 0 && NMMA >= 16 && NMMA <= 256, "tcgen05 M=128 needs N in 16..256");
  static_assert(BN >= 64 && BN <= 512 && BN % 32 == 0, "epilogue reads 32-column chunks");
  static_assert(B_OFF % 1024 == 0 && (NMMA * ROW_BYTES) % 1024 == 0, "swizzled tiles 1024-aligned");
};

// RPW rows x 32 columns of one stage: lane (h, p) of warp wg builds columns
// 4p .. 4p+3 of rows r_i = wg * RPW + 4 i + h (h = lane / 8, p = lane % 8),
// i < RPW / 4, as two column pairs.  For a pair (2j, 2j+1) of the row's word
// the rank c of column 2j among the set bits indexes its value in the compact
// row; the values of rank c and c + 1 are loaded zero-extended and one prmt,
// its selector looked up from a 4-entry table by the pair's two mask bits,
// places them or zeros.  The shared-memory accesses are issued in three
// batches (mask words, values, stores) so that each batch's latency is paid
// once per stage rather than once per row.
// sMw: this stage's mask word of row 0; mstride: bytes from one row's word
// to the next row's.
template <int RPW>
__device__ __forceinline__ void densify_stage(uint32_t sA, uint32_t sV, uint32_t sMw,
                                              uint32_t mstride, int wg, int lane) {
  static_assert(RPW % 8 == 0, "the swizzle phases below need whole groups of 8 rows");
  constexpr int R = RPW / 4;
  const int h = lane >> 3, p = lane & 7;
  const uint32_t b0 = 4u * p;
  const uint32_t below = (1u << b0) - 1u;       // columns of the word left of 4p
  const uint32_t r_first = (uint32_t)(wg * RPW + h);
  // 64-byte swizzle: 16-byte chunk index ^= (row >> 1) & 3.  Row r_i gives
  // (r_i >> 1) & 3 = (2 i + (h >> 1)) & 3 = (2 i & 3) ^ (h >> 1), since
  // wg * RPW / 2 is a multiple of 4: two lane-constant offsets by i & 1.
  const uint32_t lane_chunk = (uint32_t)((p >> 1) ^ (h >> 1));
  const uint32_t in_chunk = (uint32_t)(p & 1) * 8u;
  const uint32_t off_even = (lane_chunk << 4) + in_chunk;           // i even: phase ^ 0
  const uint32_t off_odd = ((lane_chunk ^ 2u) << 4) + in_chunk;     // i odd:  phase ^ 2
  // prmt selectors by q (bit 0: column 2j kept, bit 1: 2j+1 kept) for the
  // values v (rank c) and w (rank c + 1): q 0 -> 0x3232 (0, 0),
  // 1 -> 0x3210 (v, 0), 2 -> 0x1032 (0, v), 3 -> 0x5410 (v, w).
  constexpr uint32_t kSelLo = 0x32103232u, kSelHi = 0x54101032u;
  uint32_t m[R], nib[R], v[R][4];
#pragma unroll
  for (int i = 0; i < R; ++i) m[i] = lds_u32(sMw + mstride * (r_first + 4 * i));
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const uint32_t r = r_first + 4 * i;
    const uint32_t c = __popc(m[i] & below);            // rank of column 4p
    nib[i] = (m[i] >> b0) & 15u;
    const uint32_t c2 = c + __popc(nib[i] & 3u);         // rank of column 4p + 2
    const uint32_t a0 = sV + 32u * r + 2u * c, a2 = sV + 32u * r + 2u * c2;
    v[i][0] = lds_u16_32(a0);
    v[i][1] = lds_u16_32(a0 + 2u);
    v[i][2] = lds_u16_32(a2);
    v[i][3] = lds_u16_32(a2 + 2u);
  }
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const uint32_t r = r_first + 4 * i;
    const uint32_t lo = prmt(v[i][0], v[i][1], prmt(kSelLo, kSelHi, (nib[i] & 3u) * 0x22u + 0x10u));
    const uint32_t hi = prmt(v[i][2], v[i][3], prmt(kSelLo, kSelHi, (nib[i] >> 2) * 0x22u + 0x10u));
    sts_u64(sA + r * ROW_BYTES + ((i & 1) ? off_odd : off_even), lo, hi);
  }
}

// DG: the densify warps form DG groups; group g expands stages g, g + DG,
// ... with 128 / (16 / DG) rows per warp.  Each stage costs a warp a fixed
// chain of barrier waits, fences and arrivals (hundreds of cycles of
// latency) besides its rows, so with DG groups that chain overlaps DG stages.
template <int NMMA, int NB, int STAGES, int G, int DG, int DW, int MS, bool MT>
__global__ void __launch_bounds__(threads_for(DW), 1)
    spmm_tc_kernel(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_x,
                   const __grid_constant__ CUtensorMap tm_m, const uint32_t* __restrict__ masks,
                   __half* __restrict__ Y, float* __restrict__ part, int64_t rows, int words,
                   int wslice, int64_t T, int64_t ldy, uint64_t wait_limit_ns, int stall_weights) {
  using L = Layout<NMMA, NB, STAGES, DG, MS, MT>;
  static_assert(DG == 1 || G == 1, "waiting on every second stage needs one densify group");
  // G = 2 waits on the odd stages' afull barriers only; with an even ring each
  // of those barriers serves odd stages alone, so every parity wait stays exact.
  static_assert(G == 1 || L::AFULL_RING % 2 == 0, "waiting on every second stage needs an even ring");
  static_assert(MS == 0 || G == 1, "each of two issuers waits on each of its stages");
  static_assert(DW % DG == 0 && DW % 4 == 0, "equal densify groups, whole TMEM quadrants");
  static_assert(threads_for(DW) <= 1024, "a block has at most 1024 threads");
  static_assert(DG <= MW, "every densify group must read every mask box, in order");
  constexpr int WPG = DW / DG;             // warps per densify group
  constexpr int RPW = BM / WPG;            // rows per warp and stage
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t sA = base + L::A_OFF, sB = base + L::B_OFF, sV = base + L::V_OFF,
                 sM = base + L::M_OFF, bars = base + L::BAR_OFF, slot = base + L::SLOT_OFF;
  constexpr int FB = L::FULL_RING, AB = L::AFULL_RING;
  // full / afull: by stage kt (rings of FB / AB); empty: by slot kt % STAGES.
  auto full = [&](int kt) { return bars + 8u * (kt % FB); };
  auto full_par = [&](int kt) { return (uint32_t)((kt / FB) & 1); };
  auto empty = [&](int s) { return bars + 8u * (FB + s); };
  auto afull = [&](int kt) { return bars + 8u * (FB + STAGES + kt % AB); };
  auto afull_par = [&](int kt) { return (uint32_t)((kt / AB) & 1); };
  const uint32_t accum = bars + 8u * (FB + STAGES + AB);
  // A mask box serves MW consecutive stages that may belong to different
  // densify groups, so it completes on a barrier of its own.
  auto mfull = [&](int slot) { return bars + 8u * (FB + STAGES + AB + 1 + slot); };
  // ... and is released on one when every densify warp has finished its last
  // stage in the box (the stages of a box may go to different MMA issuers, so
  // no single stage's completion implies that).
  auto mfree = [&](int slot) {
    return bars + 8u * (FB + STAGES + AB + 1 + L::MT_SLOTS + slot);
  };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // After a wait gave up (this launch or an earlier one not yet reset), the
  // block does nothing: the decision is block-uniform, taken before any
  // barrier, copy or tensor-memory allocation.
  if (__syncthreads_or(threadIdx.x == 0 && wait_aborted())) return;
  const int64_t r0 = (int64_t)blockIdx.y * BM;
  const int64_t n0 = (int64_t)blockIdx.x * L::BN;
  // K split: this block multiplies the mask words w0 .. w0 + nk - 1 (stage
  // kt is word w0 + kt); w0 is a multiple of MW, so mask boxes stay aligned.
  const int w0 = (int)blockIdx.z * wslice;
  const int nk = min(words - w0, wslice);

  if (warp == 0 && lane == 0) {
    for (int k = 0; k < FB; ++k)
      mbar_init(full(k), MT ? 2 : 2 + 32);    // two expect_tx arrivals (+ 32 cp.async arrivals)
    for (int s = 0; s < STAGES; ++s) mbar_init(empty(s), 1);  // tcgen05.commit
    for (int k = 0; k < AB; ++k) mbar_init(afull(k), WPG);    // one arrival per warp of the group
    mbar_init(accum, MS ? 2 : 1);             // final commit of each issuer
    for (int m = 0; m < L::MT_SLOTS; ++m) {
      mbar_init(mfull(m), 1);
      mbar_init(mfree(m), DW);
    }
    fence_mbar_init();
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_x);
    if (MT) prefetch_tmap(&tm_m);
  }
  if (warp == 1) {
    tmem_alloc(slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  uint32_t tmem_base;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(tmem_base) : "r"(slot) : "memory");

  // Teardown must not free shared memory under copies still in flight: a
  // producer waits (bounded) for the stages it issued among the last STAGES
  // of the row -- the final use of each slot, so the phase it waits for is
  // the slot's last.  A producer that stopped early on a timeout issued
  // nothing in the last 2 s worth waiting for.
  auto drain = [&](int last) {
    for (int kt = last; kt >= 0 && kt > nk - 1 - STAGES; --kt)
      mbar_wait(full(kt), full_par(kt), wait_limit_ns, false);
  };

  if (warp == 0) {
    // ---- X producer: the token tile of each stage -------------------------
    if (lane == 0) {
      int last = -1;
      for (int kt = 0; kt < nk; ++kt) {
        const int s = kt % STAGES, u = kt / STAGES;
        if (u > 0 && !mbar_wait(empty(s), (u - 1) & 1, wait_limit_ns)) break;
        mbar_arrive_expect_tx(full(kt), L::B_BYTES);
#pragma unroll
        for (int j = 0; j < NB; ++j)
          tma_load_2d(sB + s * L::B_BYTES + j * NMMA * ROW_BYTES, &tm_x, (w0 + kt) * BK,
                      (int)(n0 + j * NMMA), full(kt));
        last = kt;
      }
      drain(last);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ---- W producer: compact values (and, without MT, mask words) ----------
    // With MT one lane issues the values' TMA (the mask boxes have a warp of
    // their own); without, all lanes also gather the mask words by cp.async,
    // each arriving on the stage barrier when its copies land.
    // stall_weights (self-test only) issues nothing: every consumer's bounded
    // wait then runs out and the block tears down without storing Y.
    if ((!MT || lane == 0) && !stall_weights) {
      int last = -1;
      for (int kt = 0; kt < nk; ++kt) {
        const int s = kt % STAGES, u = kt / STAGES;
        int ok = 1;
        if (u > 0 && lane == 0) ok = mbar_wait(empty(s), (u - 1) & 1, wait_limit_ns);
        if (!MT) ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(full(kt), V_BYTES);
          tma_load_2d(sV + s * V_BYTES, &tm_v, (w0 + kt) * 16, (int)r0, full(kt));
        }
        if (!MT) {
#pragma unroll
          for (int i = 0; i < BM / 32; ++i) {
            const int rr = lane + 32 * i;
            const int64_t gr = r0 + rr;
            const bool in = gr < rows;
            cp_async_4(sM + s * M_BYTES + 4u * rr, masks + (in ? gr : 0) * words + w0 + kt,
                       in ? 4u : 0u);
          }
          cp_async_arrive_noinc(full(kt));
        }
        last = kt;
      }
      if (!MT) cp_async_wait_all();
      if (lane == 0) drain(last);
    }
    __syncwarp();
  } else if (warp == mask_warp(DW)) {
    // ---- mask producer (MT): one box of MW stages' mask words at a time -----
    // A slot is refilled only after every densify warp released it from the
    // slot's previous box.  This warp alone refills, in box order, so the
    // release waited for is always the previous box's.
    if (MT && lane == 0 && !stall_weights) {
      int nbox = 0;
      for (int kt = 0; kt < nk; kt += MW) {
        const int b = kt / MW, ms = b % L::MT_SLOTS;
        if (b >= L::MT_SLOTS &&
            !mbar_wait(mfree(ms), ((b / L::MT_SLOTS) - 1) & 1, wait_limit_ns))
          break;
        mbar_arrive_expect_tx(mfull(ms), MT_SLOT);
        tma_load_2d(sM + ms * MT_SLOT, &tm_m, w0 + kt, (int)r0, mfull(ms));
        nbox = kt / MW + 1;
      }
      const int b0 = nbox > L::MT_SLOTS ? nbox - L::MT_SLOTS : 0;  // boxes still in flight
      for (int b = b0; b < nbox; ++b)
        mbar_wait(mfull(b % L::MT_SLOTS), (b / L::MT_SLOTS) & 1, wait_limit_ns);
    }
    __syncwarp();
  } else if (warp == 1 || warp == mma2_warp(DW)) {
    // ---- MMA issuers ----------------------------------------------------
    // Each waits only on the densify barriers: the densify warps saw the
    // stage's "full" barrier complete (so the TMA-loaded X tile is visible
    // through their release-arrive).  With one densify group (DG == 1) every
    // warp arrives on the stages in order, so G = 2 may wait on every second
    // barrier only (afull(kt + 1) complete implies afull(kt)).  A barrier test,
    // a commit and each tcgen05.mma cost the issuing thread tens to hundreds
    // of cycles, so with MS == 1 two threads share the stages (even / odd,
    // into two accumulators).
    const int role = warp == 1 ? 0 : 1;
    if (lane == 0 && (role == 0 || MS != 0)) {
      constexpr uint32_t idesc = idesc_f16_f32(BM, NMMA);
      const int k0 = MS ? role : 0, kstep = MS ? 2 : G;
      const uint32_t dacc = tmem_base + (uint32_t)(MS && role ? L::BN : 0);
      for (int kt = k0; kt < nk; kt += kstep) {
        const int last = MS ? kt : (kt + G - 1 < nk ? kt + G - 1 : nk - 1);
        if (!mbar_wait(afull(last), afull_par(last), wait_limit_ns)) break;
        tc_fence_after_sync();
        for (int k = kt; k <= last; ++k) {
          const int s = k % STAGES;
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks) {
            const uint64_t ad = smem_desc_sw64(sA + s * A_BYTES + ks * 32);
#pragma unroll
            for (int j = 0; j < NB; ++j) {
              const uint64_t bd =
                  smem_desc_sw64(sB + s * L::B_BYTES + j * NMMA * ROW_BYTES + ks * 32);
              mma_f16(dacc + (uint32_t)(j * NMMA), ad, bd, idesc, (k != k0) || (ks != 0));
            }
          }
          // Only a slot that a producer refills gets its release: no one
          // waits for the last STAGES stages', and a commit's arrival is not
          // ordered with the accum commit's, so it could land after this
          // block ended, in the barriers of the next block on the SM.
          if (k + STAGES < nk) mma_commit(empty(s));
        }
      }
      mma_commit(accum);  // also after an early exit: completes once issued MMAs finish
    }
    __syncwarp();
  } else {
    // ---- densify, then epilogue -----------------------------------------
    const int dw = warp - FIRST_DENSIFY_WARP;
    const int grp = dw / WPG, wg = dw % WPG;
    bool ok = true;
    int box = -1;  // mask box this warp last waited for
    for (int kt = grp; kt < nk; kt += DG) {
      const int s = kt % STAGES;
      bool got = mbar_wait(full(kt), full_par(kt), wait_limit_ns);
      if (MT && kt / MW != box) {
        // The box's slot is refilled only after every densify warp released
        // it, so the phase this warp sees here is this box's.
        box = kt / MW;
        got = got && mbar_wait(mfull(box % L::MT_SLOTS), (box / L::MT_SLOTS) & 1, wait_limit_ns);
      }
      // The warp decides together, so no lane is left behind at a warp barrier.
      if (!__all_sync(0xFFFFFFFFu, got)) { ok = false; break; }
      const uint32_t sMw = MT ? sM + ((kt / MW) % L::MT_SLOTS) * MT_SLOT + (kt % MW) * 4u
                              : sM + s * M_BYTES;
      densify_stage<RPW>(sA + s * A_BYTES, sV + s * V_BYTES, sMw, MT ? MW * 4u : 4u, wg, lane);
      // Each lane orders its tile writes before the tensor core's reads; the
      // warp barrier then lets one release-arrive publish all 32 lanes' writes
      // (one arrival per warp: 32 arrivals on one barrier word serialise).
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(afull(kt));
        // This warp's last stage in the mask box: it has read the box (its
        // loads precede the release-arrive), so the slot may be refilled.
        if (MT && kt + DG >= MW * (kt / MW + 1)) mbar_arrive(mfree((kt / MW) % L::MT_SLOTS));
      }
    }
    if (!mbar_wait(accum, 0, wait_limit_ns)) ok = false;
    tc_fence_after_sync();
    // tcgen05.ld is a warp-wide instruction: the whole warp reads or none does.
    if (__all_sync(0xFFFFFFFFu, ok)) {
      const int quad = warp & 3;              // TMEM lanes 32*quad .. +31
      const int qi = dw >> 2;                 // this warp's index among its quadrant's warps
      constexpr int QW = DW / 4;              // warps per quadrant, striding the columns
      const int64_t r = r0 + 32 * quad + lane;
      const bool row_ok = r < rows;
      const uint32_t tbase = tmem_base + ((uint32_t)(32 * quad) << 16);
#pragma unroll 1
      for (int c0 = qi * 32; c0 < L::BN; c0 += QW * 32) {
        uint32_t v[32];
        tmem_ld_32(tbase + (uint32_t)c0, v);
        tmem_ld_wait();
        if (MS && nk > 1) {  // the odd stages' accumulator (none when nk == 1)
          uint32_t w[32];
          tmem_ld_32(tbase + (uint32_t)(L::BN + c0), w);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            v[i] = __float_as_uint(__uint_as_float(v[i]) + __uint_as_float(w[i]));
        }
        if (row_ok && part) {  // K split: this slice's fp32 sums, [slice][T][rows]
          float* pz = part + (int64_t)blockIdx.z * T * rows + r;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int64_t t = n0 + c0 + i;
            if (t < T) pz[t * rows] = __uint_as_float(v[i]);
          }
        } else if (row_ok) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int64_t t = n0 + c0 + i;
            if (t < T) Y[t * ldy + r] = __float2half_rn(__uint_as_float(v[i]));
          }
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    // Tensor memory is freed only after the MMAs that write it have completed:
    // one more bounded (not abortable) wait on the final commit, which a
    // normal run passed already.  An MMA issuer that stopped early committed
    // what it issued, so the barrier still completes.
    mbar_wait(accum, 0, wait_limit_ns, false);
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
}

// ---- host ------------------------------------------------------------------
struct Variant {
  int nmma, nb, stages, g, dg, dw, ms;
};
// Stage counts are the deepest that fit 227 KB of shared memory (4 for the
// first 512-token variant, kept as the shallower alternative).
constexpr Variant kVariants[] = {{256, 2, 4, 1, 2, 16, 0},  {256, 1, 7, 1, 2, 16, 1},
                                 {128, 1, 10, 1, 4, 16, 1}, {64, 1, 12, 1, 4, 16, 1},
                                 {256, 2, 5, 1, 4, 16, 0}};
constexpr int kVariantCount = sizeof(kVariants) / sizeof(kVariants[0]);

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiled encode_fn() {
  static EncodeTiled fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiled>(p);
  }();
  return fn;
}

static bool encode_2d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
                      uint64_t stride_bytes, uint32_t box_inner, uint32_t box_outer,
                      CUtensorMapSwizzle swz,
                      CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_FLOAT16) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dtype, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NMMA, int NB, int STAGES, int G, int DG, int DW, int MS, bool MT>
static cudaError_t launch_tc_mt(const SpmmTcParams& p, cudaStream_t stream) {
  using L = Layout<NMMA, NB, STAGES, DG, MS, MT>;
  CUtensorMap tm_v, tm_x, tm_m;
  memset(&tm_m, 0, sizeof(tm_m));
  if (MT && !encode_2d(&tm_m, p.masks, (uint64_t)p.words, (uint64_t)p.rows,
                       (uint64_t)p.words * 4, MW, BM, CU_TENSOR_MAP_SWIZZLE_NONE,
                       CU_TENSOR_MAP_DATA_TYPE_UINT32))
    return cudaErrorInvalidValue;
  if (!encode_2d(&tm_v, p.values, (uint64_t)p.words * 16, (uint64_t)p.rows,
                 (uint64_t)p.words * 32, 16, BM, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_2d(&tm_x, p.X, (uint64_t)p.words * 32, (uint64_t)p.T, (uint64_t)p.ldx * 2, BK,
                 NMMA, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  auto* k = spmm_tc_kernel<NMMA, NB, STAGES, G, DG, DW, MS, MT>;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) return e;
    attr_done[dev] = 1;
  }
  const int wslice = p.slices > 1 ? p.wslice : p.words;
  const dim3 grid((unsigned)((p.T + L::BN - 1) / L::BN), (unsigned)((p.rows + BM - 1) / BM),
                  (unsigned)(p.slices > 1 ? p.slices : 1));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads_for(DW));
  cfg.dynamicSmemBytes = L::SMEM;
  cfg.stream = stream;
  const uint64_t limit = p.wait_limit_ns ? p.wait_limit_ns : kWaitLimitNs;
  float* part = p.slices > 1 ? p.part : nullptr;
  return cudaLaunchKernelEx(&cfg, k, tm_v, tm_x, tm_m, p.masks, p.Y, part, p.rows, p.words,
                            wslice, p.T, p.ldy, limit, p.stall_weights);
}

// Y[t][r] = fp16(sum over slices z, in increasing z, of part[z][t][r]): the
// K split's fixed-order combine (one rounding, no atomics).  V = 4: each
// thread takes four consecutive rows (16-byte loads, one 8-byte store), and
// issues the slices' loads four at a time; the additions keep slice order.
__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

template <int V>
__global__ void __launch_bounds__(256) splitk_sum_kernel(const float* __restrict__ part,
                                                         int slices, int64_t T, int64_t rows,
                                                         __half* __restrict__ Y, int64_t ldy) {
  const int64_t plane = T * rows;
  for (int64_t t = blockIdx.y; t < T; t += gridDim.y) {
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * V; r < rows;
         r += (int64_t)gridDim.x * blockDim.x * V) {
      const float* q = part + t * rows + r;
      if (V == 4) {
        float4 acc = *reinterpret_cast<const float4*>(q);
        int z = 1;
        for (; z + 3 < slices; z += 4) {
          const float4 a = *reinterpret_cast<const float4*>(q + z * plane);
          const float4 b = *reinterpret_cast<const float4*>(q + (z + 1) * plane);
          const float4 c = *reinterpret_cast<const float4*>(q + (z + 2) * plane);
          const float4 d = *reinterpret_cast<const float4*>(q + (z + 3) * plane);
          acc = add4(add4(add4(add4(acc, a), b), c), d);
        }
        for (; z < slices; ++z) acc = add4(acc, *reinterpret_cast<const float4*>(q + z * plane));
        const __half2 lo = __floats2half2_rn(acc.x, acc.y), hi = __floats2half2_rn(acc.z, acc.w);
        uint2 w;
        w.x = *reinterpret_cast<const uint32_t*>(&lo);
        w.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(Y + t * ldy + r) = w;
      } else {
        float acc = q[0];
        for (int z = 1; z < slices; ++z) acc += q[z * plane];
        Y[t * ldy + r] = __float2half_rn(acc);
      }
    }
  }
}

static cudaError_t launch_splitk_sum(const SpmmTcParams& p, cudaStream_t stream) {
  // Four rows a thread when every row group of Y is 8-byte aligned (the
  // partial planes then are 16-byte aligned: the workspace is).
  const bool v4 = p.rows % 4 == 0 && p.ldy % 4 == 0 &&
                  (reinterpret_cast<uintptr_t>(p.Y) & 7) == 0;
  const int64_t per_block = v4 ? 1024 : 256;
  const int64_t bx = (p.rows + per_block - 1) / per_block;
  const dim3 grid((unsigned)(bx < 65535 ? bx : 65535), (unsigned)(p.T < 65535 ? p.T : 65535));
  if (v4)
    splitk_sum_kernel<4><<<grid, 256, 0, stream>>>(p.part, p.slices, p.T, p.rows, p.Y, p.ldy);
  else
    splitk_sum_kernel<1><<<grid, 256, 0, stream>>>(p.part, p.slices, p.T, p.rows, p.Y, p.ldy);
  return cudaGetLastError();
}

// Mask words by TMA when the mask array allows it (16-byte aligned, row pitch
// words * 4 a multiple of 16: every decoder shape), else by cp.async.
template <int NMMA, int NB, int STAGES, int G, int DG, int DW, int MS>
static cudaError_t launch_tc(const SpmmTcParams& p, cudaStream_t stream) {
  const bool mt = p.words % 4 == 0 && (reinterpret_cast<uintptr_t>(p.masks) & 15) == 0;
  return mt ? launch_tc_mt<NMMA, NB, STAGES, G, DG, DW, MS, true>(p, stream)
            : launch_tc_mt<NMMA, NB, STAGES, G, DG, DW, MS, false>(p, stream);
}

}  // namespace tc

int spmm_tc_variant_count() { return tc::kVariantCount; }

// Words per K slice when a row of `words` mask words is cut into at most
// `splits` slices: a multiple of four (one mask box), so every slice but the
// last is whole boxes.  The slice count is then ceil(words / slice).
int spmm_tc_slice_words(int words, int splits) {
  if (splits <= 1 || words <= 4) return words;
  const int w = (words + splits - 1) / splits;
  const int r = (w + 3) / 4 * 4;
  return r < words ? r : words;
}

int spmm_tc_slices(int words, int splits) {
  const int w = spmm_tc_slice_words(words, splits);
  return (words + w - 1) / w;
}

size_t spmm_tc_workspace_bytes(int64_t rows, int words, int64_t T, int splits) {
  const int z = spmm_tc_slices(words, splits);
  return z > 1 ? (size_t)z * (size_t)T * (size_t)rows * sizeof(float) : 0;
}

// Time model of a plan (variant, K slices), in ns: waves of blocks x (the
// slice's stages x the variant's time per 32-column stage + a block's fixed
// cost + its output stores: fp16 Y, or fp32 sums when split), plus, when
// split, the combine (a launch and its traffic).  Times per stage measured on
// GB300 over the decoder-layer shapes, one block per SM: 512 tokens 441 (5
// stages), 256 tokens 319 (7), 128 tokens 232 (10), 64 tokens 218 (12).  The
// other constants were fitted to a sweep of every (variant, 1..8 slices) over
// eight decoder matrices (4096..57344 rows, 4096..28672 columns) at 16, 64,
// 256, 512 and 2048 tokens, on which the model picks the fastest plan in
// every case.  A larger token tile does more work per stage; a smaller one,
// or a K split, fills more SMs when rows (or tokens) are few.
namespace {
struct Cand {
  int variant, tokens;
  double ns_per_stage;
};
constexpr Cand kCand[] = {{4, 512, 441.0}, {1, 256, 319.0}, {2, 128, 232.0}, {3, 64, 218.0}};
constexpr double kBlockNs = 3000.0;        // prologue, pipeline fill, teardown
constexpr double kStoreBytesPerNs = 80.0;  // one block's output stores (per SM)
constexpr double kCombineNs = 2500.0;      // the combine kernel's launch and ramp
constexpr double kCombineBytesPerNs = 8000.0;  // partial sums written, read; Y written
constexpr size_t kMaxSplitBytes = (size_t)256 << 20;

double plan_ns(const Cand& c, int64_t rows, int words, int64_t T, int sms, int splits) {
  const int64_t tiles = ((rows + 127) / 128) * ((T + c.tokens - 1) / c.tokens);
  const int z = spmm_tc_slices(words, splits);
  const int64_t waves = (tiles * z + sms - 1) / sms;
  const double out_bytes = (double)c.tokens * 128.0 * (z > 1 ? 4.0 : 2.0);
  double t = (double)waves * (spmm_tc_slice_words(words, splits) * c.ns_per_stage + kBlockNs +
                              out_bytes / kStoreBytesPerNs);
  if (z > 1)
    t += kCombineNs + (double)(4 * z + 4 * z + 2) * (double)T * (double)rows / kCombineBytesPerNs;
  return t;
}
}  // namespace

// The plan of least modelled time.  variant >= 0 fixes the variant; splits
// >= 1 fixes the slice request (1: no split); max_splits bounds the search.
void spmm_tc_default_plan(int64_t rows, int words, int64_t T, int sms, int variant, int splits,
                          int max_splits, int* variant_out, int* splits_out) {
  if (sms < 1) sms = 1;
  int best_v = variant >= 0 ? variant : 3, best_z = 1;
  double best_t = 0.0;
  for (const auto& c : kCand) {
    if (variant >= 0 && c.variant != variant) continue;
    const int lo = splits >= 1 ? splits : 1, hi = splits >= 1 ? splits : max_splits;
    for (int z = lo; z <= hi; ++z) {
      if (z > 1 && (spmm_tc_slices(words, z) != z ||
                    spmm_tc_workspace_bytes(rows, words, T, z) > kMaxSplitBytes))
        continue;
      const double t = plan_ns(c, rows, words, T, sms, z);
      if (best_t == 0.0 || t < best_t * 0.97) {  // prefer the earlier (larger tile, fewer slices)
        best_v = c.variant;
        best_z = z;
        best_t = t;
      }
    }
  }
  if (variant >= 0 && best_t == 0.0) best_z = splits >= 1 ? splits : 1;  // variant 0: not modelled
  *variant_out = best_v;
  *splits_out = best_z;
}

int spmm_tc_default_variant(int64_t rows, int64_t T, int sms) {
  int v, z;
  spmm_tc_default_plan(rows, 32, T, sms, -1, 1, 1, &v, &z);
  return v;
}

int spmm_tc_block_tokens(int variant) {
  return tc::kVariants[variant].nmma * tc::kVariants[variant].nb;
}

static cudaError_t launch_spmm_tc_main(const SpmmTcParams& p, int variant, cudaStream_t stream) {
  switch (variant) {
    case 0: return tc::launch_tc<256, 2, 4, 1, 2, 16, 0>(p, stream);
    case 1: return tc::launch_tc<256, 1, 7, 1, 2, 16, 1>(p, stream);
    case 2: return tc::launch_tc<128, 1, 10, 1, 4, 16, 1>(p, stream);
    case 3: return tc::launch_tc<64, 1, 12, 1, 4, 16, 1>(p, stream);
    case 4: return tc::launch_tc<256, 2, 5, 1, 4, 16, 0>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_spmm_tc(const SpmmTcParams& p, int variant, cudaStream_t stream) {
  cudaError_t e = launch_spmm_tc_main(p, variant, stream);
  if (e != cudaSuccess || p.slices <= 1) return e;
  return tc::launch_splitk_sum(p, stream);
}

cudaError_t read_wait_timeouts(unsigned long long* count, int reset) {
  cudaError_t e = cudaMemcpyFromSymbol(count, g_wait_timeouts, sizeof(*count));
  if (e != cudaSuccess || !reset) return e;
  const unsigned long long zero = 0;
  const unsigned int clear = 0;
  e = cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof(zero));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_wait_abort, &clear, sizeof(clear));
  return e;
}

}  // namespace nmk
