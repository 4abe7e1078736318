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
#include "pa_device.cuh"
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

// Inclusive block scan of K 32-bit counters (a warp-level pass, then one pass
// over the warp totals); block totals land in tot[0..K-1].
template <int K>
__device__ void block_scan(int (&v)[K], int (*sw)[kWarps], int* tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int c = 0; c < K; ++c) {
      const int x = __shfl_up_sync(0xffffffffu, v[c], o);
      if (lane >= o) v[c] += x;
    }
  }
  if (lane == 31) {
#pragma unroll
    for (int c = 0; c < K; ++c) sw[c][warp] = v[c];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int c = 0; c < K; ++c) {
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
    for (int c = 0; c < K; ++c) v[c] += sw[c][warp - 1];
  }
}

// floor(a * b / c) for a, b >= 0, c > 0, a * b < 2^62 and a result below 2^24
// (here: a <= C < 2^24, b <= c): a single-precision estimate, then an exact
// int64 correction -- neither a 64-bit integer nor an fp64 division.
__device__ __forceinline__ long long floor_mul_div(long long a, long long b, long long c) {
  const long long num = a * b;
  long long q = static_cast<long long>(__fdividef(static_cast<float>(num), static_cast<float>(c)));
  if (q < 0) q = 0;
  while (q > 0 && q * c > num) --q;
  while ((q + 1) * c <= num) ++q;
  return q;
}

// floor(j * nt / p) for 0 <= j <= p <= 65536 and nt < 2^24, in 32-bit steps:
// nt = a*p + b  =>  j*nt/p = j*a + j*b/p, with j*b < p*p <= 2^32.
__device__ __forceinline__ int tile_split(int j, int nt, int p) {
  const unsigned a = static_cast<unsigned>(nt) / static_cast<unsigned>(p);
  const unsigned b = static_cast<unsigned>(nt) - a * static_cast<unsigned>(p);
  return static_cast<int>(j * a + (static_cast<unsigned>(j) * b) / static_cast<unsigned>(p));
}

// Length class of a task of `len` >= 1 keys: 4 classes per octave, 0..127.
__device__ __forceinline__ int length_class(int len) {
  const int msb = 31 - __clz(len);
  const int frac = msb >= 2 ? (len >> (msb - 2)) & 3 : (len << (2 - msb)) & 3;
  return msb * 4 + frac;
}

__global__ void __launch_bounds__(kThreads) plan_kernel(const PlanParams p) {
  pdl_trigger();  // the split kernel may be scheduled now; it waits for this one
  pdl_wait();     // ... and this one for whatever ran before it
  extern __shared__ int s_dyn[];
  int* s_first = s_dyn;            // [n] first slot
  int* s_parts = s_first + p.n;    // [n] partitions
  int* s_ctx = s_parts + p.n;      // [n] context length
  int* s_qlen = s_ctx + p.n;       // [n] query rows
  int* s_prow = s_qlen + p.n;      // [n] first partial row
  __shared__ long long s_red[kWarps];
  __shared__ int s_cnt[kWarps];
  __shared__ int s_bad;
  __shared__ int s_scan[4][kWarps];
  __shared__ int s_tot[4];
  __shared__ int s_bcnt[129];  // launch-order classes 127..0, then 128 = unused slots
  __shared__ long long s_sum, s_nact;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = p.n;
  const int per = (n + kThreads - 1) / kThreads;  // requests per thread, <= kPer
  if (tid == 0) s_bad = 0;
  __syncthreads();

  // ---- 1. lengths, activity, validity
  int S[kPer], L[kPer];
  long long my_sum = 0;
  int my_act = 0, my_bad = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int r = tid * per + k;
    S[k] = 0;
    L[k] = 0;
    if (k < per && r < n) {
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
  int my_slots = 0, my_rows = 0, my_extra = 0, my_mrows = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    parts[k] = 0;
    const int r = tid * per + k;
    if (k < per && r < n && !bad && S[k] > 0 && L[k] > 0) {
      const long long tiles = (static_cast<long long>(S[k]) + kTile - 1) / kTile;
      const long long share = (p.kind == PA_PLAN_UNIFORM)
                                  ? C / n_act
                                  : 1 + floor_mul_div(C - n_act, S[k], sum_s);
      long long v = p.P;
      if (tiles < v) v = tiles;
      if (share < v) v = share;
      parts[k] = static_cast<int>(v);
    }
    my_slots += parts[k];
    my_rows += parts[k] >= 2 ? parts[k] * L[k] : 0;
    my_extra += parts[k] * ((L[k] * p.G + p.rpc - 1) / p.rpc - 1);
    my_mrows += parts[k] >= 2 ? L[k] : 0;
  }

  // ---- 3. exclusive offsets (slots, partial rows, extra items)
  int inc[4] = {my_slots, my_rows, my_extra, my_mrows};
  block_scan<4>(inc, s_scan, s_tot);
  __syncthreads();
  int slot0 = inc[0] - my_slots, row0 = inc[1] - my_rows, extra0 = inc[2] - my_extra;
  int mrow0 = inc[3] - my_mrows;
  const bool rows_overflow = static_cast<long long>(s_tot[1]) > p.rows_cap ||
                             static_cast<long long>(s_tot[2]) > p.max_extra ||
                             s_tot[3] > p.max_tokens;
  if (rows_overflow) {
    // Cannot happen for a plan built with these limits; empty the plan rather
    // than write partial rows past the scratch.
#pragma unroll
    for (int k = 0; k < kPer; ++k) parts[k] = 0;
    slot0 = 0;
    row0 = 0;
    extra0 = 0;
    mrow0 = 0;
  }
  const int total_slots = rows_overflow ? 0 : s_tot[0];
  const int total_extra = rows_overflow ? 0 : s_tot[2];
  const int total_mrows = rows_overflow ? 0 : s_tot[3];
  if (tid == 0 && (bad || rows_overflow)) atomicOr(p.dev.err, PA_DEVERR_PLAN_OVERFLOW);

#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int r = tid * per + k;
    if (k < per && r < n) {
      p.dev.reduce[r] = make_int2(slot0, parts[k]);
      p.dev.snap[r] = make_int2(S[k], L[k]);
      s_first[r] = slot0;
      s_parts[r] = parts[k];
      s_ctx[r] = S[k];
      s_qlen[r] = L[k];
      s_prow[r] = row0;
      // extra work items: row chunks 1.. of every slot of this request
      const int chunks = (L[k] * p.G + p.rpc - 1) / p.rpc;
      if (chunks > 1)
        for (int j = 0; j < parts[k]; ++j)
          for (int c = 1; c < chunks; ++c)
            p.dev.extra[extra0 + j * (chunks - 1) + (c - 1)] = make_int2(slot0 + j, c);
      extra0 += parts[k] * (chunks - 1);
      if (parts[k] >= 2)
        for (int i = 0; i < L[k]; ++i)
          p.dev.mrows[mrow0 + i] = make_int4(r | ((parts[k] - 1) << 12), i, row0 + i, L[k]);
      mrow0 += parts[k] >= 2 ? L[k] : 0;
      slot0 += parts[k];
      row0 += parts[k] >= 2 ? parts[k] * L[k] : 0;
    }
  }
  if (tid < 129) s_bcnt[tid] = 0;
  if (tid == 0) {
    p.dev.counters[0] = total_extra;
    p.dev.counters[1] = 0;
    p.dev.counters[2] = 0;
    p.dev.counters[3] = total_mrows;
  }
  __syncthreads();

  // ---- 4. slot fill (and launch-order class counts)
  // Lanes of a warp that share a class add their count with one atomic.
  auto warp_claim = [&](int cls) {
    const unsigned peers = __match_any_sync(__activemask(), cls);
    const int leader = __ffs(peers) - 1;
    int base = 0;
    if (lane == leader) base = atomicAdd(&s_bcnt[cls], __popc(peers));
    base = __shfl_sync(peers, base, leader);
    return base + __popc(peers & ((1u << lane) - 1u));
  };
  // Task of an active slot and its launch-order class (0 = longest tasks).
  auto slot_fill = [&](int slot) {
    if (slot >= total_slots) {
      p.dev.work[slot] = make_int4(-1, 0, 0, 0);
      p.dev.part_row[slot] = -1;
      return 128;
    }
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
    const int nt = (s_ctx[r] + kTile - 1) / kTile;
    const int tb = tile_split(j, nt, pr);
    const int te = tile_split(j + 1, nt, pr);
    p.dev.work[slot] = make_int4(r, tb, te, s_ctx[r]);
    p.dev.part_row[slot] = pr >= 2 ? s_prow[r] + j * s_qlen[r] : -1;
    const int keys = min(te * kTile, s_ctx[r]) - tb * kTile;
    return 127 - length_class(keys);
  };
  constexpr int kCached = 4;  // classes kept in registers for the scatter (C <= 4096)
  int cls[kCached];
#pragma unroll
  for (int k = 0; k < kCached; ++k) cls[k] = -1;
  for (int slot = tid, k = 0; slot < C; slot += kThreads, ++k) {
    const int c = slot_fill(slot);
    if (k < kCached) cls[k] = c;
    warp_claim(c);
  }
  __syncthreads();
  // ---- 5. launch order: counting sort of the slots by length class
  if (warp == 0) {  // exclusive prefix over the 129 classes: 5 per lane, then a warp scan
    int v[5], sum = 0;
#pragma unroll
    for (int k = 0; k < 5; ++k) {
      const int b = lane * 5 + k;
      v[k] = b < 129 ? s_bcnt[b] : 0;
      sum += v[k];
    }
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += x;
    }
    int pos = inc - sum;
#pragma unroll
    for (int k = 0; k < 5; ++k) {
      const int b = lane * 5 + k;
      if (b < 129) s_bcnt[b] = pos;
      pos += v[k];
    }
  }
  __syncthreads();
  for (int slot = tid, k = 0; slot < C; slot += kThreads, ++k) {
    int c;
    if (k < kCached) {
      c = cls[k];
    } else {  // beyond the cached slots: recompute the class (C > 4096 only)
      int lo = 0, hi = n;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_first[mid] <= slot) lo = mid; else hi = mid;
      }
      if (slot >= total_slots) {
        c = 128;
      } else {
        const int nt = (s_ctx[lo] + kTile - 1) / kTile, j = slot - s_first[lo];
        const int tb = tile_split(j, nt, s_parts[lo]), te = tile_split(j + 1, nt, s_parts[lo]);
        c = 127 - length_class(min(te * kTile, s_ctx[lo]) - tb * kTile);
      }
    }
    p.dev.order[warp_claim(c)] = slot;
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
  return launch_pdl(plan_kernel, dim3(1), dim3(kThreads), 5 * p.n * static_cast<int>(sizeof(int)), s, p);
}

}  // namespace pa
