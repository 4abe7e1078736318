// pa_merge.cu -- LSE-weighted merge of the partial results of requests that
// were split into several partitions.
//
// "[MiniMax-M3] Route the paged decode to aiter's FlyDSL kernel with work
// planner", section 6 item 5 and review item 7: after the split attention
// tiles, a reduce combines each request's partitions by their log-sum-exp.
// The split kernel's partials are already normalised, so
//     out = sum_j 2^(lse_j - M) o_j / sum_j 2^(lse_j - M),   M = max_j lse_j.
//
// The planner lists the rows of requests with several pieces, each entry carrying
// what the merge needs (request, token, the first partial row and the row
// stride between partitions), so that the partial rows and log-sum-exps are
// addressed straight from the entry.  Rows with at most 8 pieces (listed
// first) are merged one warp per (row, q head) pair: every piece's log-sum-exp
// and partial slice are loaded at once and combined with shuffles.  Rows with
// more pieces take a whole CTA per pair: the CTA is cut into units of D/4 lanes
// (at most a warp), each unit holding one partial row with 4 outputs per lane;
// unit u merges partitions u, u + NU, ... online (running maximum, rescaled
// sum), with kMergeUnroll partitions' loads in flight, and the units are
// combined through shared memory.  With no multi-partition request the grid
// exits at once.  Rows of stale requests are not written (the split kernel's
// zero CTAs wrote them).
#include "../../include/pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kMergeThreads = 256;

template <int D>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeParams p) {
  constexpr int UL = D / 4 < 32 ? D / 4 : 32;  // lanes per unit
  constexpr int VPL = D / 4 / UL;               // float4 outputs per lane
  constexpr int NU = kMergeThreads / UL;        // units per CTA
  // partitions in flight per unit: 4, fewer for wide rows (registers)
  constexpr int kMergeUnroll = VPL <= 2 ? 4 : (VPL <= 4 ? 2 : 1);
  __shared__ float4 s_acc[NU][D / 4];
  __shared__ float s_m[NU];
  __shared__ float s_ws[NU];
  const float NEG_INF = -__int_as_float(0x7f800000);
  pdl_trigger();
  // What the planner wrote (the row lists and their counts) and the lengths
  // were complete before the split kernel started, so they are read before
  // waiting for the split kernel's partials.
  const int tid = threadIdx.x, u = tid / UL, ul = tid % UL;
  const int Hq = p.Hq;
  const int nfew = p.plan.counters[3];  // rows listed first: at most kWarpMergePieces pieces
  const int total = p.plan.counters[2] * Hq;
  const int warp = tid >> 5, lane = tid & 31;
  constexpr int kWarps = kMergeThreads / 32;
  // the first (row, head) pair of this warp's few-piece loop, fetched ahead
  const int wp0 = blockIdx.x * kWarps + warp;
  int4 e0 = make_int4(0, 0, 0, 0);
  int2 snap0 = make_int2(0, 0);
  int ctx0 = 0, c00 = 0, L0 = 0;
  if (wp0 < nfew * Hq) {
    e0 = p.plan.mrows[wp0 / Hq];
    const int r0 = e0.x & 4095;
    snap0 = p.plan.snap[r0];
    ctx0 = p.context_lens[r0];
    c00 = p.cu ? p.cu[r0] : r0;
    L0 = p.cu ? p.cu[r0 + 1] - c00 : 1;
  }
  pdl_wait();  // the split kernel's partials are complete
  // The split kernel is done with its work counter: reset it for the next decode.
  if (blockIdx.x == 0 && threadIdx.x == 0) p.plan.counters[1] = 0;

  // Rows with many pieces: one CTA per (row, q head) pair.
  for (int pair = blockIdx.x; pair < total; pair += gridDim.x) {
    const int4 e = p.plan.mrows[nfew + pair / Hq];
    const int r = e.x & 4095, parts = (e.x >> 12) + 1, tok = e.y, L = e.w;
    const int hq = pair % Hq;
    // staleness inputs; only the final store depends on them
    const int2 snap = p.plan.snap[r];
    const int ctx = p.context_lens[r];
    const int c0 = p.cu ? p.cu[r] : r;
    const int Lnow = p.cu ? p.cu[r + 1] - c0 : 1;

    float m = NEG_INF, ws = 0.f;
    float4 acc[VPL];
#pragma unroll
    for (int v = 0; v < VPL; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = u; j0 < parts; j0 += NU * kMergeUnroll) {
      float lse[kMergeUnroll];
      float4 o[kMergeUnroll][VPL];
#pragma unroll
      for (int k = 0; k < kMergeUnroll; ++k) {
        const int j = j0 + k * NU;
        lse[k] = NEG_INF;
#pragma unroll
        for (int v = 0; v < VPL; ++v) o[k][v] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j < parts) {
          const long long prow = static_cast<long long>(e.z + j * L) * Hq + hq;
          lse[k] = __ldcg(p.plan.part_lse + prow);
          const float4* src = reinterpret_cast<const float4*>(p.plan.part_o + prow * D);
#pragma unroll
          for (int v = 0; v < VPL; ++v) o[k][v] = __ldcg(src + ul + v * UL);
        }
      }
      float mb = m;
#pragma unroll
      for (int k = 0; k < kMergeUnroll; ++k) mb = fmaxf(mb, lse[k]);
      if (mb == NEG_INF) continue;  // no visible key in these partitions
      const float f = (m == NEG_INF) ? 0.f : fast_exp2(m - mb);
      ws *= f;
#pragma unroll
      for (int v = 0; v < VPL; ++v) {
        acc[v].x *= f; acc[v].y *= f; acc[v].z *= f; acc[v].w *= f;
      }
#pragma unroll
      for (int k = 0; k < kMergeUnroll; ++k) {
        if (lse[k] == NEG_INF) continue;
        const float w = fast_exp2(lse[k] - mb);
        ws += w;
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
          acc[v].x += w * o[k][v].x; acc[v].y += w * o[k][v].y;
          acc[v].z += w * o[k][v].z; acc[v].w += w * o[k][v].w;
        }
      }
      m = mb;
    }
    if (ul == 0) {
      s_m[u] = m;
      s_ws[u] = ws;
    }
#pragma unroll
    for (int v = 0; v < VPL; ++v) s_acc[u][ul + v * UL] = acc[v];
    __syncthreads();
    if (tid < D / 4 && snap.x == ctx && snap.y == Lnow) {
      float M = NEG_INF;
#pragma unroll
      for (int k = 0; k < NU; ++k) M = fmaxf(M, s_m[k]);
      float4 out = make_float4(0.f, 0.f, 0.f, 0.f);
      float W = 0.f;
      if (M != NEG_INF) {
#pragma unroll
        for (int k = 0; k < NU; ++k) {
          const float mk = s_m[k];
          if (mk == NEG_INF) continue;
          const float f = fast_exp2(mk - M);
          const float4 a = s_acc[k][tid];
          out.x += f * a.x; out.y += f * a.y; out.z += f * a.z; out.w += f * a.w;
          W += f * s_ws[k];
        }
      }
      if (p.sinks) {  // the head's sink joins the denominator once, here
        const float f = add_sink(M, __ldg(p.sinks + hq) * 1.4426950408889634f, W);
        out.x *= f; out.y *= f; out.z *= f; out.w *= f;
      }
      const float inv = W > 0.f ? 1.f / W : 0.f;
      const int t = c0 + tok;
      if (t >= p.num_tokens) {
        if (tid == 0) atomicOr(p.plan.err, PA_DEVERR_PLAN_OVERFLOW);
      } else {
        uint2 pk;
        if (p.out_f16) {
          pk.x = pack2<false>(out.x * inv, out.y * inv);
          pk.y = pack2<false>(out.z * inv, out.w * inv);
        } else {
          pk.x = pack2<true>(out.x * inv, out.y * inv);
          pk.y = pack2<true>(out.z * inv, out.w * inv);
        }
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) +
                                  (static_cast<size_t>(t) * Hq + hq) * D + 4 * tid) = pk;
      }
    }
    __syncthreads();  // shared memory is reused by the next pair
  }

  // Rows with few pieces: one warp per (row, q head) pair, the pieces' partials
  // loaded PB at a time (all at once up to head_dim 256), weights from shuffles.
  constexpr int VL = D / 32;  // outputs per lane
  constexpr int PB = VL <= 8 ? kWarpMergePieces : 2;
  for (int wp = wp0; wp < nfew * Hq; wp += gridDim.x * kWarps) {
    const bool first = wp == wp0;
    const int4 e = first ? e0 : p.plan.mrows[wp / Hq];
    const int r = e.x & 4095, parts = (e.x >> 12) + 1, tok = e.y, L = e.w;
    const int hq = wp % Hq;
    const int2 snap = first ? snap0 : p.plan.snap[r];
    const int ctx = first ? ctx0 : p.context_lens[r];
    const int c0 = first ? c00 : (p.cu ? p.cu[r] : r);
    const int Lnow = first ? L0 : (p.cu ? p.cu[r + 1] - c0 : 1);
    float lse = NEG_INF;
    if (lane < parts) lse = __ldcg(p.plan.part_lse + static_cast<long long>(e.z + lane * L) * Hq + hq);
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
    for (int j0 = 0; j0 < parts; j0 += PB) {
      float o[PB][VL];
#pragma unroll
      for (int k = 0; k < PB; ++k) {
        const int j = j0 + k;
        if (j < parts) {
          const float* src = p.plan.part_o + (static_cast<long long>(e.z + j * L) * Hq + hq) * D + lane * VL;
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
        const float wj = __shfl_sync(0xffffffffu, w, (j0 + k) & 31);  // w = 0 past `parts`
#pragma unroll
        for (int v = 0; v < VL; ++v) acc[v] += wj * o[k][v];
      }
    }
    if (snap.x != ctx || snap.y != Lnow) continue;  // stale: zeroed by the split kernel
    const int t = c0 + tok;
    if (t >= p.num_tokens) {
      if (lane == 0) atomicOr(p.plan.err, PA_DEVERR_PLAN_OVERFLOW);
      continue;
    }
    if (p.sinks) {
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
    uint16_t* dst = static_cast<uint16_t*>(p.out) + (static_cast<size_t>(t) * Hq + hq) * D + lane * VL;
    if constexpr (VL == 2) {
      *reinterpret_cast<uint32_t*>(dst) = pk[0];
    } else if constexpr (VL % 8 == 0) {  // 16-byte aligned: lane * VL * 2 bytes
#pragma unroll
      for (int v = 0; v < VL / 2; v += 4)
        *reinterpret_cast<uint4*>(dst + 2 * v) = make_uint4(pk[v], pk[v + 1], pk[v + 2], pk[v + 3]);
    } else {  // VL % 4 == 0: 8-byte aligned
#pragma unroll
      for (int v = 0; v < VL / 2; v += 2)
        *reinterpret_cast<uint2*>(dst + 2 * v) = make_uint2(pk[v], pk[v + 1]);
    }
  }
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, cudaStream_t s) {
  if (p.grid <= 0) return cudaSuccess;
#define PA_MERGE_CASE(DD) \
  case DD: return launch_pdl(merge_kernel<DD>, dim3(p.grid), dim3(kMergeThreads), 0, s, p);
  switch (p.D) {
    PA_MERGE_CASE(64)
    PA_MERGE_CASE(128)
    PA_MERGE_CASE(256)
    PA_MERGE_CASE(384)
    PA_MERGE_CASE(512)
    PA_MERGE_CASE(640)
    PA_MERGE_CASE(768)
    PA_MERGE_CASE(896)
    PA_MERGE_CASE(1024)
    default: return cudaErrorInvalidValue;
  }
#undef PA_MERGE_CASE
}

}  // namespace pa
