// pa_plan.cu -- the on-device work planner / in-place refresh.
//
// Rule ("[MiniMax-M3] Route the paged decode to aiter's FlyDSL kernel with work
// planner", section 1: each request gets a partition count proportional to its
// real context length under a workgroup budget; section 5: capacity
// C = min(n*P, max(n, ceil(W/Hkv))); review item 2: per-task begin/end tiles
// plus seq_ctx).  With n_act requests that have S > 0 and a query row:
//   proportional: p = min(P, ceil(S/256), 1 + floor((C - n_act) * S / sum S))
//   uniform:      p = min(P, ceil(S/256), floor(C / n_act))
// Slots are request-major; part j of a request covers tiles
// [floor(j*nt/p), floor((j+1)*nt/p)).
//
// One CTA of 1024 threads, each owning 4 consecutive requests (n <= 4096):
// two block reductions (n_act, sum S), one block scan (slot, partial-row and
// extra-item offsets), then a slot-parallel fill that finds each slot's request
// by binary search over the scanned offsets.  It also writes the split
// kernel's launch order (slots by task length, longest first, by a counting
// sort over 128 quarter-octave length classes) and the extra work items that
// split the query rows of requests with more rows than one work item holds.
// No allocation, no host synchronisation: it can be captured in a CUDA graph.
#include "../../include/pa.h"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kThreads = 1024;
constexpr int kPer = kMaxSeqs / kThreads;  // requests per thread
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ long long warp_sum64(long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Inclusive block scan of three 32-bit counters (a warp-level pass, then one
// pass over the warp totals); block totals land in tot[0..2].
__device__ void block_scan3(int (&v)[3], int (*sw)[kWarps], int* tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int c = 0; c < 3; ++c) {
      const int x = __shfl_up_sync(0xffffffffu, v[c], o);
      if (lane >= o) v[c] += x;
    }
  }
  if (lane == 31) {
#pragma unroll
    for (int c = 0; c < 3; ++c) sw[c][warp] = v[c];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int c = 0; c < 3; ++c) {
      int w = lane < kWarps ? sw[c][lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += x;
      }
      if (lane < kWarps) sw[c][lane] = w;
      if (lane == kWarps - 1) tot[c] = w;
    }
  }
  __syncthreads();
  if (warp > 0) {
#pragma unroll
    for (int c = 0; c < 3; ++c) v[c] += sw[c][warp - 1];
  }
}

// Length class of a task of `len` >= 1 keys: 4 classes per octave, 0..127.
__device__ __forceinline__ int length_class(int len) {
  const int msb = 31 - __clz(len);
  const int frac = msb >= 2 ? (len >> (msb - 2)) & 3 : (len << (2 - msb)) & 3;
  return msb * 4 + frac;
}

__global__ void __launch_bounds__(kThreads) plan_kernel(const PlanParams p) {
  extern __shared__ int s_dyn[];
  int* s_first = s_dyn;            // [n] first slot
  int* s_parts = s_first + p.n;    // [n] partitions
  int* s_ctx = s_parts + p.n;      // [n] context length
  int* s_qlen = s_ctx + p.n;       // [n] query rows
  int* s_prow = s_qlen + p.n;      // [n] first partial row
  __shared__ long long s_red[kWarps];
  __shared__ int s_cnt[kWarps];
  __shared__ int s_bad;
  __shared__ int s_scan[3][kWarps];
  __shared__ int s_tot[3];
  __shared__ int s_bcnt[129];  // launch-order classes 127..0, then 128 = unused slots
  __shared__ long long s_sum, s_nact;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = p.n;
  if (tid == 0) s_bad = 0;
  __syncthreads();

  // ---- 1. lengths, activity, validity
  int S[kPer], L[kPer];
  long long my_sum = 0;
  int my_act = 0, my_bad = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int r = tid * kPer + k;
    S[k] = 0;
    L[k] = 0;
    if (r < n) {
      S[k] = p.context_lens[r];
      L[k] = p.cu ? p.cu[r + 1] - p.cu[r] : 1;
      if (L[k] < 0 || L[k] > p.max_qlen) my_bad = 1;
      if (S[k] > 0 && L[k] > 0) {
        my_act += 1;
        my_sum += S[k];
      }
    }
  }
  if (tid == 0 && p.cu && (p.cu[0] != 0 || p.cu[n] > p.max_tokens)) my_bad = 1;
  if (my_bad) atomicOr(&s_bad, 1);
  my_sum = warp_sum64(my_sum);
  int act_w = my_act;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) act_w += __shfl_xor_sync(0xffffffffu, act_w, o);
  if (lane == 0) {
    s_red[warp] = my_sum;
    s_cnt[warp] = act_w;
  }
  __syncthreads();
  if (tid == 0) {
    long long a = 0, c = 0;
    for (int w = 0; w < kWarps; ++w) {
      a += s_red[w];
      c += s_cnt[w];
    }
    s_sum = a;
    s_nact = c;
  }
  __syncthreads();
  const bool bad = s_bad != 0;
  const long long sum_s = s_sum, n_act = s_nact;
  const long long C = p.C;

  // ---- 2. partition counts, partial rows and extra row-chunk items per request
  int parts[kPer];
  int my_slots = 0, my_rows = 0, my_extra = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    parts[k] = 0;
    const int r = tid * kPer + k;
    if (r < n && !bad && S[k] > 0 && L[k] > 0) {
      const long long tiles = (static_cast<long long>(S[k]) + kTile - 1) / kTile;
      const long long share = (p.kind == PA_PLAN_UNIFORM)
                                  ? C / n_act
                                  : 1 + ((C - n_act) * static_cast<long long>(S[k])) / sum_s;
      long long v = p.P;
      if (tiles < v) v = tiles;
      if (share < v) v = share;
      parts[k] = static_cast<int>(v);
    }
    my_slots += parts[k];
    my_rows += parts[k] >= 2 ? parts[k] * L[k] : 0;
    my_extra += parts[k] * ((L[k] * p.G + p.rpc - 1) / p.rpc - 1);
  }

  // ---- 3. exclusive offsets (slots, partial rows, extra items)
  int inc[3] = {my_slots, my_rows, my_extra};
  block_scan3(inc, s_scan, s_tot);
  __syncthreads();
  int slot0 = inc[0] - my_slots, row0 = inc[1] - my_rows, extra0 = inc[2] - my_extra;
  const bool rows_overflow = static_cast<long long>(s_tot[1]) > p.rows_cap ||
                             static_cast<long long>(s_tot[2]) > p.max_extra;
  if (rows_overflow) {
    // Cannot happen for a plan built with these limits; empty the plan rather
    // than write partial rows past the scratch.
#pragma unroll
    for (int k = 0; k < kPer; ++k) parts[k] = 0;
    slot0 = 0;
    row0 = 0;
    extra0 = 0;
  }
  const int total_slots = rows_overflow ? 0 : s_tot[0];
  const int total_extra = rows_overflow ? 0 : s_tot[2];
  if (tid == 0 && (bad || rows_overflow)) atomicOr(p.dev.err, PA_DEVERR_PLAN_OVERFLOW);

#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int r = tid * kPer + k;
    if (r < n) {
      p.dev.reduce[r] = make_int2(slot0, parts[k]);
      p.dev.snap[r] = make_int2(S[k], L[k]);
      s_first[r] = slot0;
      s_parts[r] = parts[k];
      s_ctx[r] = S[k];
      s_qlen[r] = L[k];
      s_prow[r] = row0;
      // extra work items: row chunks 1.. of every slot of this request
      const int chunks = (L[k] * p.G + p.rpc - 1) / p.rpc;
      for (int j = 0; j < parts[k]; ++j)
        for (int c = 1; c < chunks; ++c)
          p.dev.extra[extra0 + j * (chunks - 1) + (c - 1)] = make_int2(slot0 + j, c);
      extra0 += parts[k] * (chunks - 1);
      slot0 += parts[k];
      row0 += parts[k] >= 2 ? parts[k] * L[k] : 0;
    }
  }
  if (tid < 129) s_bcnt[tid] = 0;
  if (tid == 0) {
    p.dev.counters[0] = total_extra;
    p.dev.counters[1] = 0;
  }
  __syncthreads();

  // ---- 4. slot fill (and launch-order class counts)
  auto slot_task = [&](int slot, int& r, int& tb, int& te) {
    int lo = 0, hi = n;  // last r with s_first[r] <= slot (it has parts > 0)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_first[mid] <= slot)
        lo = mid;
      else
        hi = mid;
    }
    r = lo;
    const int pr = s_parts[r];
    const int j = slot - s_first[r];
    const long long nt = (static_cast<long long>(s_ctx[r]) + kTile - 1) / kTile;
    tb = static_cast<int>((j * nt) / pr);
    te = static_cast<int>(((j + 1) * nt) / pr);
  };
  auto slot_class = [&](int slot) {
    if (slot >= total_slots) return 128;
    int r, tb, te;
    slot_task(slot, r, tb, te);
    const long long keys = min(static_cast<long long>(te) * kTile, static_cast<long long>(s_ctx[r])) -
                           static_cast<long long>(tb) * kTile;
    return 127 - length_class(static_cast<int>(keys));  // 0 = longest class
  };
  for (int slot = tid; slot < C; slot += kThreads) {
    atomicAdd(&s_bcnt[slot_class(slot)], 1);
    if (slot < total_slots) {
      int r, tb, te;
      slot_task(slot, r, tb, te);
      const int pr = s_parts[r];
      const int j = slot - s_first[r];
      p.dev.work[slot] = make_int4(r, tb, te, s_ctx[r]);
      p.dev.part_row[slot] = pr >= 2 ? s_prow[r] + j * s_qlen[r] : -1;
    } else {
      p.dev.work[slot] = make_int4(-1, 0, 0, 0);
      p.dev.part_row[slot] = -1;
    }
  }
  __syncthreads();
  // ---- 5. launch order: counting sort of the slots by length class
  if (tid == 0) {
    int pos = 0;
    for (int b = 0; b < 129; ++b) {
      const int c = s_bcnt[b];
      s_bcnt[b] = pos;
      pos += c;
    }
  }
  __syncthreads();
  for (int slot = tid; slot < C; slot += kThreads) p.dev.order[atomicAdd(&s_bcnt[slot_class(slot)], 1)] = slot;
}

}  // namespace

cudaError_t launch_plan(const PlanParams& p, cudaStream_t s) {
  static bool attr_done = false;
  const int smem = 5 * kMaxSeqs * static_cast<int>(sizeof(int));
  if (!attr_done) {
    cudaError_t e =
        cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  plan_kernel<<<1, kThreads, 5 * p.n * static_cast<int>(sizeof(int)), s>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
