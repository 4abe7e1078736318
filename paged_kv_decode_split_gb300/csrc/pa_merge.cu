// pa_merge.cu -- LSE-weighted merge of the partial results of requests that
// were split into several partitions.
//
// "[MiniMax-M3] Route the paged decode to aiter's FlyDSL kernel with work
// planner", section 6 item 5 and review item 7: after the split attention
// tiles, a reduce combines each request's partitions by their log-sum-exp.
// The split kernel's partials are already normalised, so
//     out = sum_j 2^(lse_j - M) o_j / sum_j 2^(lse_j - M),   M = max_j lse_j.
//
// The planner lists the rows of multi-partition requests, each entry carrying
// what the merge needs (request, token, the first partial row and the row
// stride between partitions), so that the partial rows and log-sum-exps are
// addressed straight from the entry.  A persistent grid walks (row, q head)
// pairs, one CTA per pair at a time.  The CTA is cut into units of D/4 lanes
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
constexpr int kMergeUnroll = 4;  // partitions in flight per unit

template <int D>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeParams p) {
  constexpr int UL = D / 4 < 32 ? D / 4 : 32;  // lanes per unit
  constexpr int VPL = D / 4 / UL;               // float4 outputs per lane
  constexpr int NU = kMergeThreads / UL;        // units per CTA
  __shared__ float4 s_acc[NU][D / 4];
  __shared__ float s_m[NU];
  __shared__ float s_ws[NU];
  const float NEG_INF = -__int_as_float(0x7f800000);
  pdl_trigger();
  pdl_wait();  // the split kernel's partials are complete
  // The split kernel is done with its work counter: reset it for the next decode.
  if (blockIdx.x == 0 && threadIdx.x == 0) p.plan.counters[1] = 0;
  const int tid = threadIdx.x, u = tid / UL, ul = tid % UL;
  const int Hq = p.Hq;
  const int total = p.plan.counters[3] * Hq;

  for (int pair = blockIdx.x; pair < total; pair += gridDim.x) {
    const int4 e = p.plan.mrows[pair / Hq];
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
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, cudaStream_t s) {
  if (p.grid <= 0) return cudaSuccess;
  switch (p.D) {
    case 64: return launch_pdl(merge_kernel<64>, dim3(p.grid), dim3(kMergeThreads), 0, s, p);
    case 128: return launch_pdl(merge_kernel<128>, dim3(p.grid), dim3(kMergeThreads), 0, s, p);
    default: return launch_pdl(merge_kernel<256>, dim3(p.grid), dim3(kMergeThreads), 0, s, p);
  }
}

}  // namespace pa
