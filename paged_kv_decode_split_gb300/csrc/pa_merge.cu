// pa_merge.cu -- LSE-weighted merge of the partial results of requests that
// were split into several partitions.
//
// "[MiniMax-M3] Route the paged decode to aiter's FlyDSL kernel with work
// planner", section 6 item 5 and review item 7: after the split attention
// tiles, a reduce combines each request's partitions by their log-sum-exp.
// The split kernel's partials are already normalised, so
//     out = sum_j 2^(lse_j - M) o_j / sum_j 2^(lse_j - M),   M = max_j lse_j.
//
// The planner lists the (request, token) rows of multi-partition requests; a
// persistent grid walks (row, q head) pairs of that list, one CTA per pair at
// a time.  Inside a CTA the partitions are dealt to PG thread groups, each
// thread owning 4 consecutive outputs, and the groups are reduced through
// shared memory -- so a row with many partitions is merged with many loads in
// flight.  With no multi-partition request the grid exits at once.  Rows of
// stale requests are skipped (the split kernel's zero CTAs wrote them).
#include "../../include/pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kMergeThreads = 256;

template <int D>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeParams p) {
  constexpr int DL = D / 4;                // threads per group, 4 outputs each
  constexpr int PG = kMergeThreads / DL;   // partition groups
  __shared__ float s_max[kMergeThreads / 32];
  __shared__ float4 s_acc[PG][DL];
  __shared__ float s_w[PG];
  const float NEG_INF = -__int_as_float(0x7f800000);
  pdl_trigger();
  pdl_wait();  // the split kernel's partials are complete
  const int tid = threadIdx.x, g = tid / DL, dl = tid % DL;
  const int lane = tid & 31, warp = tid >> 5;
  const int Hq = p.Hq;
  const int total = p.plan.counters[3] * Hq;

  for (int pair = blockIdx.x; pair < total; pair += gridDim.x) {
    const int2 e = p.plan.mrows[pair / Hq];
    const int r = e.x, tok = e.y, hq = pair % Hq;
    const int2 snap = p.plan.snap[r];
    const int L = p.cu ? p.cu[r + 1] - p.cu[r] : 1;
    if (snap.x != p.context_lens[r] || snap.y != L) continue;  // stale: zeroed by the split kernel
    const int t = (p.cu ? p.cu[r] : r) + tok;
    if (t >= p.num_tokens) {
      if (tid == 0) atomicOr(p.plan.err, PA_DEVERR_PLAN_OVERFLOW);
      continue;
    }
    const int2 red = p.plan.reduce[r];
    const int first = red.x, parts = red.y;

    // pass 1: M = max_j lse_j
    float m = NEG_INF;
    for (int j = tid; j < parts; j += kMergeThreads) {
      const size_t prow = static_cast<size_t>(p.plan.part_row[first + j] + tok) * Hq + hq;
      m = fmaxf(m, __ldcg(p.plan.part_lse + prow));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) s_max[warp] = m;
    __syncthreads();
    float M = s_max[0];
#pragma unroll
    for (int w = 1; w < kMergeThreads / 32; ++w) M = fmaxf(M, s_max[w]);

    // pass 2: group g takes partitions g, g + PG, ...
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (M != NEG_INF) {
#pragma unroll 4
      for (int j = g; j < parts; j += PG) {
        const size_t prow = static_cast<size_t>(p.plan.part_row[first + j] + tok) * Hq + hq;
        const float lse = __ldcg(p.plan.part_lse + prow);
        const float w = (lse == NEG_INF) ? 0.f : fast_exp2(lse - M);
        const float4 v = __ldcg(reinterpret_cast<const float4*>(p.plan.part_o + prow * D) + dl);
        acc.x += w * v.x; acc.y += w * v.y; acc.z += w * v.z; acc.w += w * v.w;
        wsum += w;
      }
    }
    s_acc[g][dl] = acc;
    if (dl == 0) s_w[g] = wsum;
    __syncthreads();
    if (tid < DL) {
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      float W = 0.f;
#pragma unroll
      for (int k = 0; k < PG; ++k) {
        const float4 a = s_acc[k][tid];
        o.x += a.x; o.y += a.y; o.z += a.z; o.w += a.w;
        W += s_w[k];
      }
      const float inv = W > 0.f ? 1.f / W : 0.f;
      uint2 pk;
      if (p.out_f16) {
        pk.x = pack2<false>(o.x * inv, o.y * inv);
        pk.y = pack2<false>(o.z * inv, o.w * inv);
      } else {
        pk.x = pack2<true>(o.x * inv, o.y * inv);
        pk.y = pack2<true>(o.z * inv, o.w * inv);
      }
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) +
                                (static_cast<size_t>(t) * Hq + hq) * D + 4 * tid) = pk;
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
