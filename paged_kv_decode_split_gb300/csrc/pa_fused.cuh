// pa_fused.cuh -- the LSE merge fused into the split kernel, for decode-only
// plans ("[MiniMax-M3] Route the paged decode to aiter's FlyDSL kernel with
// work planner", section 6 item 5 and review item 7: the partial-softmax
// reduce after the split attention tiles costs a second launch and ~14%).
//
// A request r of L query rows (tokens) with K >= 2 pieces leaves, per kv head
// h, K x L normalised fp32 partial rows (piece k's row for token t at
// base + k * L + t, G q heads each) and their log2-sum-exps.  Here
// the CTAs that wrote them combine them, with no waits: pieces form groups of
// kFusedFanIn consecutive ones; a CTA that finishes a piece takes a ticket of
// its group (an atomic count per group, level and kv head), and the one that
// takes the group's last ticket merges the group's partials -- into the
// request's output rows when the group is the whole request, else into one
// partial stored in place of the group's first piece, after which it takes a
// ticket at the next level, where the groups' results are grouped in the same
// way.  So no CTA combines more than kFusedFanIn partials per step, and a
// request of K pieces needs ceil(log8 K) steps on its last CTA.
//
// Merge rule (log2 units, as the split kernel's partials):
//     M = max_i lse_i,  w_i = 2^(lse_i - M),  W = sum_i w_i,
//     o = sum_i w_i o_i / W,  lse = M + log2 W   (W = 0: o = 0, lse = -inf);
// at the last level a sink logit joins W once (add_sink), and o is rounded to
// the output type.
//
// Ordering: a named barrier of the consumer warps orders their partial stores
// before one thread's GPU-scope release fence and its relaxed ticket atomic;
// the taker of a group's last ticket fences again (acquire) before the barrier
// after which the consumer warps read the partials through L2 (ld.cg).
#pragma once

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// Merges items [first, first + count) of `level` of request r's tree for kv
// head h -- item i's row for token t lives in partial row
// base + (i << 3*level) * L + t -- for the L tokens and G q heads of h, one
// warp per (token, q head).  final: write the output rows orow + t;
// otherwise write the merged partials in place of item `first`.
template <int D>
__device__ __forceinline__ void fused_merge_group(const SplitParams& p, int h, int base, int L,
                                                  int first, int count, int level, bool final,
                                                  int orow, int cw, int ncw, int lane) {
  constexpr int VL = D / 32;            // outputs per lane
  constexpr int PB = VL <= 8 ? kFusedFanIn : (VL <= 16 ? 2 : 1);  // items loaded at once
  const float NEG_INF = -__int_as_float(0x7f800000);
  const int G = p.G, Hq = p.Hq;
  const int sh = kFusedLog2FanIn * level;
  for (int x = cw; x < L * G; x += ncw) {
    const int t = x / G, gq = x - t * G;  // token, q head of h
    const int hq = h * G + gq;
    float lse = NEG_INF;
    if (lane < count)
      lse = __ldcg(p.plan.part_lse +
                   static_cast<long long>(base + ((first + lane) << sh) * L + t) * Hq + hq);
    float M = lse;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float w = (lse == NEG_INF) ? 0.f : fast_exp2(lse - M);
    float W = w;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
    float acc[VL];
#pragma unroll
    for (int v = 0; v < VL; ++v) acc[v] = 0.f;
    for (int j0 = 0; j0 < count; j0 += PB) {
      float o[PB][VL];
#pragma unroll
      for (int k = 0; k < PB; ++k) {
        const int j = j0 + k;
        if (j < count) {
          const float* src = p.plan.part_o +
                             (static_cast<long long>(base + ((first + j) << sh) * L + t) * Hq + hq) * D +
                             lane * VL;
          if constexpr (VL % 4 == 0) {
#pragma unroll
            for (int v = 0; v < VL; v += 4) {
              const float4 x = __ldcg(reinterpret_cast<const float4*>(src + v));
              o[k][v] = x.x; o[k][v + 1] = x.y; o[k][v + 2] = x.z; o[k][v + 3] = x.w;
            }
          } else {
#pragma unroll
            for (int v = 0; v < VL; v += 2) {
              const float2 x = __ldcg(reinterpret_cast<const float2*>(src + v));
              o[k][v] = x.x;
              o[k][v + 1] = x.y;
            }
          }
        } else {
#pragma unroll
          for (int v = 0; v < VL; ++v) o[k][v] = 0.f;
        }
      }
#pragma unroll
      for (int k = 0; k < PB; ++k) {
        const float wj = __shfl_sync(0xffffffffu, w, (j0 + k) & 31);  // 0 past `count`
#pragma unroll
        for (int v = 0; v < VL; ++v) acc[v] += wj * o[k][v];
      }
    }
    if (final && orow + t >= p.num_tokens) {  // a row past the call's rows: the plan was not
      if (lane == 0) atomicOr(p.plan.err, PA_DEVERR_PLAN_OVERFLOW);  // made for this call
    } else if (final) {
      if (p.sinks) {  // the head's sink joins the denominator once, at the last level
        const float f = add_sink(M, __ldg(p.sinks + hq) * 1.4426950408889634f, W);
#pragma unroll
        for (int v = 0; v < VL; ++v) acc[v] *= f;
      }
      const float inv = W > 0.f ? 1.f / W : 0.f;
      uint32_t pk[VL / 2];
#pragma unroll
      for (int v = 0; v < VL; v += 2)
        pk[v / 2] = p.out_f16 ? pack2<false>(acc[v] * inv, acc[v + 1] * inv)
                              : pack2<true>(acc[v] * inv, acc[v + 1] * inv);
      uint16_t* dst = static_cast<uint16_t*>(p.out) + (static_cast<size_t>(orow + t) * Hq + hq) * D +
                      lane * VL;
      if constexpr (VL == 2) {
        *reinterpret_cast<uint32_t*>(dst) = pk[0];
      } else if constexpr (VL % 8 == 0) {
#pragma unroll
        for (int v = 0; v < VL / 2; v += 4)
          *reinterpret_cast<uint4*>(dst + 2 * v) = make_uint4(pk[v], pk[v + 1], pk[v + 2], pk[v + 3]);
      } else {
#pragma unroll
        for (int v = 0; v < VL / 2; v += 2)
          *reinterpret_cast<uint2*>(dst + 2 * v) = make_uint2(pk[v], pk[v + 1]);
      }
    } else {
      const float inv = W > 0.f ? 1.f / W : 0.f;
      const long long prow = static_cast<long long>(base + (first << sh) * L + t) * Hq + hq;
      float* dst = p.plan.part_o + prow * D + lane * VL;
#pragma unroll
      for (int v = 0; v < VL; v += 2)
        *reinterpret_cast<float2*>(dst + v) = make_float2(acc[v] * inv, acc[v + 1] * inv);
      if (lane == 0) p.plan.part_lse[prow] = W > 0.f ? M + __log2f(W) : NEG_INF;
    }
  }
}

// Called by every consumer thread (ct in [0, ncw * 32), consumer warp cw) once
// the item's partial rows (piece partial rows from `prow`, one per token of
// the request's L; request r, kv head h) are written.  Takes this piece's
// tickets up the tree and merges where it took a group's last one; orow is the
// request's first output row.
template <int D>
__device__ __noinline__ void fused_merge(const SplitParams& p, int r, int h, int prow, int orow, int L,
                                         int ct, int cw, int ncw, int lane) {
  __shared__ int s_last;
  const int2 pq = p.plan.preq[r];  // (first partial row, pieces)
  const int base = pq.x;
  int k = (prow - base) / L;       // this piece's index, then its group's at each level
  int K = pq.y;                    // items at this level
  for (int level = 0;; ++level) {
    const int first = (k >> kFusedLog2FanIn) << kFusedLog2FanIn;
    const int count = min(kFusedFanIn, K - first);
    named_barrier_sync(1, ncw * 32);  // every consumer's stores (and reads of s_last) are done
    if (ct == 0) {
      int* t = p.plan.tickets +
               (static_cast<long long>(level) * p.rows_cap +
                (base + (first << (kFusedLog2FanIn * level)) * L)) * p.Hkv + h;
      fence_acq_rel_gpu();  // release: the CTA's partials above precede the ticket
      const int prev = atomicAdd(t, 1);
      const int last = prev == count - 1;
      if (last) {
        *t = 0;               // the group is complete: ready for the next decode call
        fence_acq_rel_gpu();  // acquire: the other pieces' partials are visible
      }
      s_last = last;
    }
    named_barrier_sync(1, ncw * 32);
    if (!s_last) return;
    const bool final = K <= kFusedFanIn;
    fused_merge_group<D>(p, h, base, L, first, count, level, final, orow, cw, ncw, lane);
    if (final) return;
    k >>= kFusedLog2FanIn;
    K = (K + kFusedFanIn - 1) >> kFusedLog2FanIn;
  }
}

}  // namespace pa
