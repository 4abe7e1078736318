// pa_merge.cu -- LSE-weighted merge of a request's partial results.
//
// "[MiniMax-M3] Route the paged decode to aiter's FlyDSL kernel with work
// planner", section 6 item 5 and review item 7: after the split attention
// tiles, a reduce combines each request's partitions by their log-sum-exp
// (exp_sums / max_logits / temporary_output).  Here the partials are already
// normalised: out = sum_j 2^(lse_j - M) o_j / sum_j 2^(lse_j - M), M = max lse.
//
// One CTA per output row t.  The row's request is found by binary search over
// cu_query_lens (vllm-rdna pull 29, Change 1).  Rows past cu[n], rows of
// requests without partitions and rows of a request whose lengths changed
// since the last plan refresh are written as zeros (the latter also raise
// PA_DEVERR_STALE_PLAN).  Requests with a single partition were written by the
// split kernel directly and are left untouched.
#include "../../include/pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kMergeThreads = 128;

__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeParams p) {
  const int t = blockIdx.x;
  int r = -1, tok = 0;
  if (p.cu) {
    if (t < p.cu[p.n]) {
      int lo = 0, hi = p.n;  // last r with cu[r] <= t
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.cu[mid] <= t)
          lo = mid;
        else
          hi = mid;
      }
      r = lo;
      tok = t - p.cu[r];
    }
  } else if (t < p.n) {
    r = t;
  }

  int parts = 0, first = 0;
  bool stale = false;
  if (r >= 0) {
    const int2 snap = p.plan.snap[r];
    const int L = p.cu ? p.cu[r + 1] - p.cu[r] : 1;
    stale = snap.x != p.context_lens[r] || snap.y != L;
    const int2 red = p.plan.reduce[r];
    first = red.x;
    parts = red.y;
    if (stale && threadIdx.x == 0) atomicOr(p.plan.err, PA_DEVERR_STALE_PLAN);
  }
  if (!stale && parts == 1) return;

  const int D = p.D;
  const int units = p.Hq * (D / 8);  // 8 output elements per unit
  uint16_t* orow = static_cast<uint16_t*>(p.out) + static_cast<size_t>(t) * p.Hq * D;
  if (stale || parts == 0) {
    for (int u = threadIdx.x; u < units; u += kMergeThreads)
      *reinterpret_cast<uint4*>(orow + u * 8) = make_uint4(0u, 0u, 0u, 0u);
    return;
  }

  const float NEG_INF = -__int_as_float(0x7f800000);
  for (int u = threadIdx.x; u < units; u += kMergeThreads) {
    const int hq = u / (D / 8);
    const int d0 = (u % (D / 8)) * 8;
    float M = NEG_INF;
    for (int j = 0; j < parts; ++j) {
      const size_t prow = static_cast<size_t>(p.plan.part_row[first + j] + tok) * p.Hq + hq;
      M = fmaxf(M, p.plan.part_lse[prow]);
    }
    float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (M != NEG_INF) {
      float wsum = 0.f;
      for (int j = 0; j < parts; ++j) {
        const size_t prow = static_cast<size_t>(p.plan.part_row[first + j] + tok) * p.Hq + hq;
        const float lse = p.plan.part_lse[prow];
        if (lse == NEG_INF) continue;
        const float w = fast_exp2(lse - M);
        wsum += w;
        const float4* src = reinterpret_cast<const float4*>(p.plan.part_o + prow * D + d0);
        const float4 a = src[0], b = src[1];
        o[0] += w * a.x; o[1] += w * a.y; o[2] += w * a.z; o[3] += w * a.w;
        o[4] += w * b.x; o[5] += w * b.y; o[6] += w * b.z; o[7] += w * b.w;
      }
      const float inv = 1.f / wsum;
#pragma unroll
      for (int k = 0; k < 8; ++k) o[k] *= inv;
    }
    uint4 pk;
    if (p.out_f16) {
      pk = make_uint4(pack2<false>(o[0], o[1]), pack2<false>(o[2], o[3]),
                      pack2<false>(o[4], o[5]), pack2<false>(o[6], o[7]));
    } else {
      pk = make_uint4(pack2<true>(o[0], o[1]), pack2<true>(o[2], o[3]),
                      pack2<true>(o[4], o[5]), pack2<true>(o[6], o[7]));
    }
    *reinterpret_cast<uint4*>(orow + hq * D + d0) = pk;
  }
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, cudaStream_t s) {
  if (p.num_tokens <= 0) return cudaSuccess;
  merge_kernel<<<p.num_tokens, kMergeThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
