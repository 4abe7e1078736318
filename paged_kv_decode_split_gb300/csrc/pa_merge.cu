// pa_merge.cu -- LSE-weighted merge of a request's partial results.
//
// "[MiniMax-M3] Route the paged decode to aiter's FlyDSL kernel with work
// planner", section 6 item 5 and review item 7: after the split attention
// tiles, a reduce combines each request's partitions by their log-sum-exp
// (exp_sums / max_logits / temporary_output).  Here the partials are already
// normalised: out = sum_j 2^(lse_j - M) o_j / sum_j 2^(lse_j - M), M = max lse.
//
// One warp per (output row t, q head).  The row's request is found by binary
// search over cu_query_lens (vllm-rdna pull 29, Change 1).  Lanes read 32
// partitions' log-sum-exps at a time (max, then weights kept in registers);
// the partial rows are then streamed with the weights broadcast by shuffle,
// each lane owning D/32 consecutive outputs.  Rows past cu[n], rows of
// requests without partitions and rows of a request whose lengths changed
// since the last plan refresh are written as zeros (the latter also raise
// PA_DEVERR_STALE_PLAN).  Requests with a single partition were written by the
// split kernel directly and are left untouched.
#include "../../include/pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kMergeWarps = 8;

template <int D>
__global__ void __launch_bounds__(32 * kMergeWarps) merge_kernel(const MergeParams p) {
  constexpr int EPL = D / 32;  // outputs per lane: 2, 4 or 8
  const int lane = threadIdx.x & 31;
  // The split kernel that ran before this one is done with its work-stealing
  // counter: reset it for the next decode call on this plan.
  if (blockIdx.x == 0 && threadIdx.x == 0) p.plan.counters[1] = 0;
  const long long pair = static_cast<long long>(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
  if (pair >= static_cast<long long>(p.num_tokens) * p.Hq) return;
  const int t = static_cast<int>(pair / p.Hq);
  const int hq = static_cast<int>(pair % p.Hq);

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
    if (stale && lane == 0 && hq == 0) atomicOr(p.plan.err, PA_DEVERR_STALE_PLAN);
  }
  if (!stale && parts == 1) return;

  uint16_t* orow = static_cast<uint16_t*>(p.out) + (static_cast<size_t>(t) * p.Hq + hq) * D + lane * EPL;
  float o[EPL];
#pragma unroll
  for (int k = 0; k < EPL; ++k) o[k] = 0.f;

  const float NEG_INF = -__int_as_float(0x7f800000);
  if (!stale && parts > 1) {
    // pass 1: the maximum log-sum-exp
    float M = NEG_INF;
    for (int j = lane; j < parts; j += 32) {
      const size_t prow = static_cast<size_t>(p.plan.part_row[first + j] + tok) * p.Hq + hq;
      M = fmaxf(M, p.plan.part_lse[prow]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if (M != NEG_INF) {
      // pass 2: 32 partitions at a time -- lane j holds weight and row of partition j
      float wsum = 0.f;
      for (int j0 = 0; j0 < parts; j0 += 32) {
        const int j = j0 + lane;
        float w = 0.f;
        size_t prow = 0;
        if (j < parts) {
          prow = static_cast<size_t>(p.plan.part_row[first + j] + tok) * p.Hq + hq;
          const float lse = p.plan.part_lse[prow];
          w = (lse == NEG_INF) ? 0.f : fast_exp2(lse - M);
        }
        wsum += w;
        const int cnt = min(32, parts - j0);
#pragma unroll 4
        for (int k = 0; k < cnt; ++k) {
          const float wk = __shfl_sync(0xffffffffu, w, k);
          const size_t rk = __shfl_sync(0xffffffffu, static_cast<unsigned long long>(prow), k);
          const float* src = p.plan.part_o + rk * D + lane * EPL;
          if constexpr (EPL == 2) {
            const float2 v = *reinterpret_cast<const float2*>(src);
            o[0] += wk * v.x; o[1] += wk * v.y;
          } else {
#pragma unroll
            for (int q = 0; q < EPL / 4; ++q) {
              const float4 v = *reinterpret_cast<const float4*>(src + 4 * q);
              o[4 * q] += wk * v.x; o[4 * q + 1] += wk * v.y;
              o[4 * q + 2] += wk * v.z; o[4 * q + 3] += wk * v.w;
            }
          }
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
      const float inv = 1.f / wsum;
#pragma unroll
      for (int k = 0; k < EPL; ++k) o[k] *= inv;
    }
  }

  uint32_t pk[EPL / 2];
#pragma unroll
  for (int k = 0; k < EPL / 2; ++k)
    pk[k] = p.out_f16 ? pack2<false>(o[2 * k], o[2 * k + 1]) : pack2<true>(o[2 * k], o[2 * k + 1]);
  if constexpr (EPL == 2) {
    *reinterpret_cast<uint32_t*>(orow) = pk[0];
  } else if constexpr (EPL == 4) {
    *reinterpret_cast<uint2*>(orow) = make_uint2(pk[0], pk[1]);
  } else {
    *reinterpret_cast<uint4*>(orow) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, cudaStream_t s) {
  if (p.num_tokens <= 0) return cudaSuccess;
  const long long pairs = static_cast<long long>(p.num_tokens) * p.Hq;
  const unsigned grid = static_cast<unsigned>((pairs + kMergeWarps - 1) / kMergeWarps);
  switch (p.D) {
    case 64: merge_kernel<64><<<grid, 32 * kMergeWarps, 0, s>>>(p); break;
    case 128: merge_kernel<128><<<grid, 32 * kMergeWarps, 0, s>>>(p); break;
    default: merge_kernel<256><<<grid, 32 * kMergeWarps, 0, s>>>(p); break;
  }
  return cudaGetLastError();
}

}  // namespace pa
