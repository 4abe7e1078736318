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
// two block reductions (n_act, sum S), one block scan (slot and partial-row
// offsets), then a slot-parallel fill that finds each slot's request by binary
// search over the scanned offsets.  No allocation, no host synchronisation:
// it can be captured in a CUDA graph.
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

// Inclusive block scan of two 32-bit counters (one warp-level pass each plus
// one pass over the warp totals); writes the block total to *total.
__device__ void block_scan2(int& a, int& b, int* sa, int* sb, int* ta, int* tb) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int xa = __shfl_up_sync(0xffffffffu, a, o);
    const int xb = __shfl_up_sync(0xffffffffu, b, o);
    if (lane >= o) {
      a += xa;
      b += xb;
    }
  }
  if (lane == 31) {
    sa[warp] = a;
    sb[warp] = b;
  }
  __syncthreads();
  if (warp == 0) {
    int va = lane < kWarps ? sa[lane] : 0;
    int vb = lane < kWarps ? sb[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int xa = __shfl_up_sync(0xffffffffu, va, o);
      const int xb = __shfl_up_sync(0xffffffffu, vb, o);
      if (lane >= o) {
        va += xa;
        vb += xb;
      }
    }
    if (lane < kWarps) {
      sa[lane] = va;
      sb[lane] = vb;
    }
    if (lane == kWarps - 1) {
      *ta = va;
      *tb = vb;
    }
  }
  __syncthreads();
  if (warp > 0) {
    a += sa[warp - 1];
    b += sb[warp - 1];
  }
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
  __shared__ int s_scan_a[kWarps], s_scan_b[kWarps];
  __shared__ int s_total_slots, s_total_rows;
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

  // ---- 2. partition counts and partial rows per request
  int parts[kPer];
  int my_slots = 0, my_rows = 0;
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
  }

  // ---- 3. exclusive offsets (slots, partial rows)
  int inc_slots = my_slots, inc_rows = my_rows;
  block_scan2(inc_slots, inc_rows, s_scan_a, s_scan_b, &s_total_slots, &s_total_rows);
  __syncthreads();
  int slot0 = inc_slots - my_slots, row0 = inc_rows - my_rows;
  const bool rows_overflow = static_cast<long long>(s_total_rows) > p.rows_cap;
  if (rows_overflow) {
    // Cannot happen for a plan built with these limits; empty the plan rather
    // than write partial rows past the scratch.
#pragma unroll
    for (int k = 0; k < kPer; ++k) parts[k] = 0;
    slot0 = 0;
    row0 = 0;
  }
  const int total_slots = rows_overflow ? 0 : s_total_slots;
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
      slot0 += parts[k];
      row0 += parts[k] >= 2 ? parts[k] * L[k] : 0;
    }
  }
  __syncthreads();

  // ---- 4. slot fill
  for (int slot = tid; slot < C; slot += kThreads) {
    if (slot < total_slots) {
      int lo = 0, hi = n;  // last r with s_first[r] <= slot (it has parts > 0)
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_first[mid] <= slot)
          lo = mid;
        else
          hi = mid;
      }
      const int r = lo;
      const int pr = s_parts[r];
      const int j = slot - s_first[r];
      const long long nt = (static_cast<long long>(s_ctx[r]) + kTile - 1) / kTile;
      const int tb = static_cast<int>((j * nt) / pr);
      const int te = static_cast<int>(((j + 1) * nt) / pr);
      p.dev.work[slot] = make_int4(r, tb, te, s_ctx[r]);
      p.dev.part_row[slot] = pr >= 2 ? s_prow[r] + j * s_qlen[r] : -1;
    } else {
      p.dev.work[slot] = make_int4(-1, 0, 0, 0);
      p.dev.part_row[slot] = -1;
    }
  }
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
