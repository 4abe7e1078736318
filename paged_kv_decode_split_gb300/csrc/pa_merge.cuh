// pa_merge.cuh -- the zero rows, written by extra CTAs of the split kernel.
//
// Rows past cu[n] (graph padding), rows of requests without partitions and
// rows of a request whose lengths changed since the last plan refresh are
// written as zeros (vllm-rdna pull 29, Change 1: padded tokens and zero-length
// requests come out as zeros); stale requests also raise PA_DEVERR_STALE_PLAN.
#pragma once

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// Rows [z*kZeroRows, (z+1)*kZeroRows) of the output: every row that no task of
// the plan writes is set to zero -- graph padding, rows of requests without
// partitions, rows of requests whose lengths differ from the plan's snapshot.
constexpr int kZeroRows = 64;

template <int D>
__device__ void zero_rows(const SplitParams& p, int z, int warp, int nwarps, int lane) {
  const int t_end = min(p.num_tokens, (z + 1) * kZeroRows);
  for (int t = z * kZeroRows + warp; t < t_end; t += nwarps) {
    int r = -1;
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
      }
    } else if (t < p.n) {
      r = t;
    }
    bool zero = r < 0;
    if (r >= 0) {
      const int2 snap = p.plan.snap[r];
      const int L = p.cu ? p.cu[r + 1] - p.cu[r] : 1;
      const bool stale = snap.x != p.context_lens[r] || snap.y != L;
      if (stale && lane == 0) atomicOr(p.plan.err, PA_DEVERR_STALE_PLAN);
      zero = stale || p.plan.reduce[r].y == 0;
    }
    if (!zero) continue;
    uint4* row = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + static_cast<size_t>(t) * p.Hq * D);
    for (int u = lane; u < p.Hq * D / 8; u += 32) row[u] = make_uint4(0u, 0u, 0u, 0u);
  }
}

}  // namespace pa
