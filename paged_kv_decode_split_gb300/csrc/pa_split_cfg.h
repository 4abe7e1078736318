// pa_split_cfg.h -- compile-time shape of the split-KV decode kernel for one
// (head dim, cache type, query-row groups, K layout): warps, pipeline stages,
// shared memory, and how many of its CTAs share an SM.  Host code reads it to
// size plans; the kernel is built from it.
#pragma once

#include "../../include/pa.h"
#include "pa_internal.h"

namespace pa {

// KL: K cache layout -- 0: [num_blocks, Hkv, bs, D]; 1: the grouped
// [num_blocks, Hkv, D/16, bs, 16] (V is always [num_blocks, Hkv, bs, D]).
template <int D, int KVT, int WQ, int KL>
struct SplitCfg {
  static constexpr bool kFp8 = (KVT == PA_FP8_E4M3);
  static constexpr bool kGroupedK = (KL == 1);
  static constexpr int GRP = 16 * (kFp8 ? 1 : 2);     // grouped K: one key's 16-dim group, bytes
  static constexpr bool kBf16Mma = (KVT == PA_BF16);
  static constexpr int ESZ = kFp8 ? 1 : 2;            // bytes per cached element
  static constexpr int ROW = D * ESZ;                 // bytes per key row
  static constexpr int SWB = ROW < 128 ? ROW : 128;   // swizzle span = box row bytes
  static constexpr int CB = ROW / SWB;                // column blocks per key row
  // Head dims above 256 are cut into slices of 256 dims (128 when 256 does
  // not divide D), one consumer warp each: a warp forms the partial logits of
  // its slice, the slices' partials are summed through shared memory (every
  // warp of the row group adds them in the same order, so all hold the same
  // logits and softmax state), and each warp accumulates P V for its own
  // slice.  Stages are one 16-key tile.
  static constexpr bool kWide = D > 256;
  // Tensor-memory path (tcgen05): fp8 caches, head dim 128, K in rows, two to
  // four query-row groups (multi-token rows).  S^T = K Q^T and O^T += V^T P^T
  // run on tcgen05.mma (kind::f8f6f4) with the accumulators in TMEM, K and V^T
  // read straight from the TMA tiles, q and P as e4m3 hi + lo pairs; one warp
  // issues the MMAs and one warpgroup does the softmax, one thread per key.
  // TN: the pass's query rows (16, 24 or 32); the MMAs' N is 2 TN.
  static constexpr bool kTc = kFp8 && D == 128 && KL == 0 && WQ >= 2;
  static constexpr int TN = 8 * WQ;
  // Row sums of P': by an MMA of a block of ones (32 rows: the per-thread
  // sums would cost the softmax, there the bottleneck, registers and time)
  // or summed by the softmax threads (16 and 24 rows: four fewer MMAs per
  // stage for the issuing thread, about 90 cycles each, on the path that
  // releases a ring slot).  Measured: 3-token verify 0.559 -> 0.575 of the
  // copy peak and the skewed 3-token batch 90.6 -> 85.0 us with per-thread
  // sums; 4 tokens 0.503 -> 0.486 (so 32 rows keep the MMA).
  static constexpr bool kTcRowSumMma = TN >= 32;
  static constexpr int DS = kWide ? (D % 256 == 0 ? 256 : 128) : D;  // head dims per consumer warp
  static constexpr int ND = D / DS;                   // dim slices
  static constexpr int CBS = DS * ESZ / SWB;          // column blocks per slice
  static constexpr int KS = kWide ? 16 : kStageTensorBytes / ROW;  // keys per stage
  // partial-logit exchange of the dim slices: [stage parity][WQ][ND][32 lanes] float4
  static constexpr int SX_BYTES = kWide ? 2 * WQ * ND * 32 * 16 : 0;
  // Ring depth: 3 stages, or 2 where that lets two CTAs share an SM (wide
  // heads of 640 and 768 dims: 3 stages of 40-48 KB need more than half of
  // the SM's 228 KB of shared memory).
  // kTc: the ring's barriers and seven more (S computed x2, P written x2,
  // P V done x2, drain), the tensor-memory address and a reduction area, then
  // (1024-aligned) q as e4m3 hi and lo [32 rows][128 B] each, per-row limits,
  // references, factors and the epilogue's offsets and scales, and a block of
  // ones
  static constexpr int TC_TMEM_SLOT = 128;              // from DATA_BYTES (after the barriers)
  static constexpr int TC_RED_OFF = 512;                // reduction area [4][32] floats
  static constexpr int TC_Q_OFF = 1024;
  static constexpr int TC_ARR_OFF = TC_Q_OFF + 8192;    // row limits, references, factors
  static constexpr int TC_ONES_OFF = TC_ARR_OFF + 1024;  // 1 KB of e4m3 ones, 1024-aligned
  static constexpr int TC_COLS = TN == 16 ? 128 : 256;  // tensor-memory columns: 4 regions
  static constexpr int kFixedBytes = kTc ? 1024 + TC_ARR_OFF + 2048 : 1024 + 64 + SX_BYTES;
  static constexpr bool kTwoPerSm3 = 2 * (3 * 2 * KS * ROW + kFixedBytes + 1024) <= 228 * 1024;
  static constexpr bool kTwoPerSm2 = 2 * (2 * 2 * KS * ROW + kFixedBytes + 1024) <= 228 * 1024;
  static constexpr int NS = (kWide && !kTwoPerSm3 && kTwoPerSm2) ? 2 : 3;  // ring depth
  static constexpr int MTS = KS / 16;                 // 16-key tiles per stage
  // Key warps per row group: 4 for one row group, 2 for two or three, 1 for
  // four -- and 1 for three row groups of 256-dim heads (MTP verify: 18-24
  // query rows), whose epilogue then needs no exchange between key warps
  // (measured 7-10% faster there; 2-19% slower for two row groups or 128 dims).
  static constexpr int WK0 = (WQ == 1) ? 4 : ((WQ == 4 || (D == 256 && WQ == 3)) ? 1 : 2);
  static constexpr int WK = WK0 < MTS ? WK0 : MTS;   // key warps per row group
  static constexpr int T = MTS / WK;                  // tiles one warp handles per stage
  // Every key warp consumes every stage, in order, so a warp never waits on a
  // ring slot's use u+1 before it consumed use u -- which keeps the
  // parity-based mbarrier waits unambiguous.
  // consumer warps (kTc: one MMA-issuing warp, then one softmax warpgroup)
  static constexpr int NCW = kTc ? 5 : WQ * WK * ND;
  // Producer warps.  Issuing a stage's copies (one per lane) holds a warp
  // for about 100-140 cycles per 2 KB box, which capped a lone CTA near
  // 25 GB/s with 16-key pages.  Two producers (K copies from one, V copies
  // from the other) overlap that work -- they still share a per-CTA limit
  // of about 110-120 cycles per box, so a lone CTA gains about 20%, not 2x --
  // for head dims up to 128, where the extra warp still leaves two CTAs per
  // SM.
  static constexpr int NPW = (D <= 128 && 32 * (2 + NCW) <= 224) ? 2 : 1;
  static constexpr int THREADS = 32 * (NPW + NCW);
  static constexpr int TILE_BYTES = KS * ROW;         // one tensor, one stage
  static constexpr int BLOCK_BYTES = KS * SWB;        // one column block of a tile
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K then V
  static constexpr int DATA_BYTES = NS * STAGE_BYTES;
  static constexpr int DP = D + 4;                    // padded exchange row, floats
  static constexpr int EX_BYTES = WQ * WK * 8 * (DP + 2) * 4;
  static constexpr int SMEM_BYTES = DATA_BYTES + kFixedBytes;
  // One key warp per row group (every wide head dim): the epilogue needs no
  // exchange, each warp stores its own accumulators.
  static constexpr bool kDirectEpi = WK == 1;
  // The producer issues the next pass's first stages while the consumers
  // finish this one: with no exchange, or with one that fits in a ring slot
  // -- the slot of the pass's last stage, which the consumers then hold
  // until the exchange is done (kHoldSlot).
  static constexpr bool kHoldSlot = !kTc && !kDirectEpi && EX_BYTES <= STAGE_BYTES;
  static constexpr bool kPreIssue = kTc || kDirectEpi || kHoldSlot;
  // two CTAs per SM where the threads' registers and both rings fit (228 KB per SM)
  static constexpr int MIN_BLOCKS = (THREADS <= 224 && 2 * (SMEM_BYTES + 1024) <= 228 * 1024) ? 2 : 1;
  static_assert(!kTc || (THREADS == 224 && MIN_BLOCKS == 2), "tcgen05 path: 7 warps, 2 CTAs per SM");
  static_assert(!kWide || (WK == 1 && T == 1 && CBS * SWB == DS * ESZ && WQ <= 2),
                "sliced head dims: one key warp, one tile per stage, whole column blocks");
  static_assert(2 * NS * 8 <= 64, "mbarriers fit before the exchange area");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
  static_assert(KS % 16 == 0 && MTS % WK == 0, "whole 16-key tiles per warp");
  static_assert(MTS * CB * 2 <= 32, "a stage needs at most one copy per producer lane");
  static_assert(!kGroupedK || MTS * (1 + CB) <= 32, "grouped K: one copy per producer lane");
  static_assert(!kGroupedK || (16 * ROW) % 1024 == 0,
                "grouped K: every 16-key box starts on a 1024-byte swizzle repeat");
  static_assert(kTc || EX_BYTES <= DATA_BYTES, "epilogue exchange reuses the stage ring");
  static_assert(!kTc || (KS == 128 && SWB == 128 && CB == 1 && NS * 16 + 56 <= TC_TMEM_SLOT &&
                         TC_ONES_OFF + 1024 <= kFixedBytes - 1024 &&
                         TC_ARR_OFF + 5 * 128 + 32 * 8 + 32 * 4 <= TC_ONES_OFF &&
                         (DATA_BYTES + TC_ONES_OFF) % 1024 == 0),
                "tcgen05 path: 128-key stages of 128-byte rows; the fixed area's layout");
  static_assert(D % 32 == 0, "head_dim is a multiple of 32");
};

// CTAs of the split kernel for (D, cache type, row groups) that one SM holds
// at once (the kernel is built to reach this many; the 16-bit caches share one
// shape, fp8 stages are half as large).
template <int D>
constexpr int split_ctas_per_sm_d(int kv_dtype, int wq) {
  const bool f8 = kv_dtype == PA_FP8_E4M3;
  switch (wq) {
    case 1: return f8 ? SplitCfg<D, PA_FP8_E4M3, 1, 0>::MIN_BLOCKS : SplitCfg<D, PA_BF16, 1, 0>::MIN_BLOCKS;
    case 2:
      if constexpr (split_max_row_groups(D) >= 2)
        return f8 ? SplitCfg<D, PA_FP8_E4M3, 2, 0>::MIN_BLOCKS : SplitCfg<D, PA_BF16, 2, 0>::MIN_BLOCKS;
      return 1;
    case 3:
      if constexpr (split_max_row_groups(D) >= 3)
        return f8 ? SplitCfg<D, PA_FP8_E4M3, 3, 0>::MIN_BLOCKS : SplitCfg<D, PA_BF16, 3, 0>::MIN_BLOCKS;
      return 1;
    default:
      if constexpr (split_max_row_groups(D) >= 4)
        return f8 ? SplitCfg<D, PA_FP8_E4M3, 4, 0>::MIN_BLOCKS : SplitCfg<D, PA_BF16, 4, 0>::MIN_BLOCKS;
      return 1;
  }
}

inline int split_ctas_per_sm(int D, int kv_dtype, int wq) {
  switch (D) {
    case 64: return split_ctas_per_sm_d<64>(kv_dtype, wq);
    case 128: return split_ctas_per_sm_d<128>(kv_dtype, wq);
    case 256: return split_ctas_per_sm_d<256>(kv_dtype, wq);
    case 384: return split_ctas_per_sm_d<384>(kv_dtype, wq);
    case 512: return split_ctas_per_sm_d<512>(kv_dtype, wq);
    case 640: return split_ctas_per_sm_d<640>(kv_dtype, wq);
    case 768: return split_ctas_per_sm_d<768>(kv_dtype, wq);
    case 896: return split_ctas_per_sm_d<896>(kv_dtype, wq);
    default: return split_ctas_per_sm_d<1024>(kv_dtype, wq);
  }
}

}  // namespace pa
