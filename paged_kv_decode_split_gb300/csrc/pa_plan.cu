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
// One CTA (128 threads up to 128 requests, else 1024), each thread owning up
// to 4 consecutive requests (n <= 4096):
// block reductions (n_act, sum S, sum of tiles), one block scan (slot, piece,
// partial-row, extra-item and merge-row offsets), then a slot-parallel fill
// that finds each slot's request by binary search over the scanned offsets.
// Beyond the plan itself it writes what the split kernel runs: every slot cut
// into pieces of about the mean slot length, or as short as allowed when the
// decode grid is more than one wave (at most Q; Q = 1 keeps tasks whole), in
// launch order (longest first, by a counting sort over 128
// quarter-octave length classes), the extra work items that split the query
// rows of requests with more rows than one work item holds, and the list of
// rows the merge combines.
// No allocation, no host synchronisation: it can be captured in a CUDA graph.
#include "../../include/pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kPer = 4;  // requests per thread at most: n <= 4 * kThreads

__device__ __forceinline__ long long warp_sum64(long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Inclusive block scan of K 32-bit counters (a warp-level pass, then one pass
// over the warp totals); block totals land in tot[0..K-1].
template <int kThreads, int K>
__device__ void block_scan(int (&v)[K], int (*sw)[kThreads / 32], int* tot) {
  constexpr int kWarps = kThreads / 32;
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
  if (warp == 0) {  // the K counters' warp totals, scanned together
    int w[K];
#pragma unroll
    for (int c = 0; c < K; ++c) w[c] = lane < kWarps ? sw[c][lane] : 0;
#pragma unroll
    for (int o = 1; o < kWarps; o <<= 1) {
#pragma unroll
      for (int c = 0; c < K; ++c) {
        const int x = __shfl_up_sync(0xffffffffu, w[c], o);
        if (lane >= o) w[c] += x;
      }
    }
#pragma unroll
    for (int c = 0; c < K; ++c) {
      if (lane < kWarps) sw[c][lane] = w[c];
      if (lane == kWarps - 1) tot[c] = w[c];
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

// Pieces for a slot of `nts` tiles when no piece may exceed `x` tiles: as
// few as that allows, but at most Q and each at least kMinPieceTiles long.
__device__ __forceinline__ int piece_count(int nts, int x, int Q) {
  if (Q <= 1) return 1;
  int q = (nts + x - 1) / x;
  q = min(q, nts / kMinPieceTiles);
  return max(1, min(q, Q));
}

// kThreads: 128 for batches of up to 128 requests (fewer idle warps on the
// one SM the planner runs on), 1024 up to 4096.
template <int kThreads>
__global__ void __launch_bounds__(kThreads) plan_kernel(const PlanParams p) {
  constexpr int kWarps = kThreads / 32;
  static_assert(kWarps <= 32, "warp totals are reduced by one warp, one per lane");
  pdl_trigger();  // the split kernel may be scheduled now; it waits for this one
  pdl_wait();     // ... and this one for whatever ran before it
  extern __shared__ int s_dyn[];
  int* s_first = s_dyn;            // [n] first slot
  int* s_parts = s_first + p.n;    // [n] partitions
  int* s_ctx = s_parts + p.n;      // [n] context length
  int* s_qlen = s_ctx + p.n;       // [n] query rows
  int* s_prow = s_qlen + p.n;      // [n] first partial row
  int* s_pfirst = s_prow + p.n;    // [n] first piece, in request order
  int* s_xfirst = s_pfirst + p.n;  // [n] first extra item
  int* s_t0 = s_xfirst + p.n;      // [n] first planned tile (sliding window; else 0)
  __shared__ long long s_red[kWarps], s_red2[kWarps];
  __shared__ int s_cnt[kWarps];
  __shared__ int s_bad;
  __shared__ int s_scan[6][kWarps];
  __shared__ int s_tot[6];
  __shared__ int s_bcnt[128];  // launch-order classes, longest first

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = p.n;
  const int per = (n + kThreads - 1) / kThreads;  // requests per thread, <= kPer
  if (tid == 0) s_bad = 0;
  for (int i = tid; i < 128; i += kThreads) s_bcnt[i] = 0;
  __syncthreads();

  // ---- 1. lengths, activity, validity; the planned range of each request
  // (with a sliding window: from the tile holding its first token's first
  // visible key; else from key 0), the sum of its lengths and of its tiles
  int S[kPer], L[kPer], T0[kPer];
  long long my_sum = 0, my_tiles = 0;
  int my_act = 0, my_bad = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int r = tid * per + k;
    S[k] = 0;
    L[k] = 0;
    T0[k] = 0;
    if (k < per && r < n) {
      S[k] = p.context_lens[r];
      L[k] = p.cu ? p.cu[r + 1] - p.cu[r] : 1;
      if (L[k] < 0 || L[k] > p.max_qlen) my_bad = 1;
      if (S[k] > 0 && L[k] > 0) {
        if (p.window > 0) {
          const long long first = static_cast<long long>(S[k]) - (L[k] - 1) - p.window;
          T0[k] = first > 0 ? static_cast<int>(first / kTile) : 0;
        }
        const int len = S[k] - T0[k] * kTile;
        my_act += 1;
        my_sum += len;
        my_tiles += (len + kTile - 1) / kTile;
      }
    }
  }
  if (tid == 0 && p.cu && (p.cu[0] != 0 || p.cu[n] > p.max_tokens)) my_bad = 1;
  if (my_bad) atomicOr(&s_bad, 1);
  my_sum = warp_sum64(my_sum);
  my_tiles = warp_sum64(my_tiles);
  int act_w = my_act;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) act_w += __shfl_xor_sync(0xffffffffu, act_w, o);
  if (lane == 0) {
    s_red[warp] = my_sum;
    s_red2[warp] = my_tiles;
    s_cnt[warp] = act_w;
  }
  __syncthreads();
  // every warp reduces the warp totals itself: no second barrier
  const long long sum_s = warp_sum64(lane < kWarps ? s_red[lane] : 0);
  const long long sum_tiles = warp_sum64(lane < kWarps ? s_red2[lane] : 0);
  long long n_act = lane < kWarps ? s_cnt[lane] : 0;
  n_act = warp_sum64(n_act);
  const bool bad = s_bad != 0;
  const long long C = p.C;

  // ---- 2. partitions per request (the plan rule)
  int parts[kPer], pcs[kPer], nbase[kPer], nbig[kPer];
  int my_maxslot = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    parts[k] = 0;
    nbase[k] = nbig[k] = 0;
    const int r = tid * per + k;
    if (k < per && r < n && !bad && S[k] > 0 && L[k] > 0) {
      const int len = S[k] - T0[k] * kTile;  // the planned range
      const long long tiles = (static_cast<long long>(len) + kTile - 1) / kTile;
      const long long share = (p.kind == PA_PLAN_UNIFORM)
                                  ? C / n_act
                                  : 1 + floor_mul_div(C - n_act, len, sum_s);
      long long v = p.P;
      if (tiles < v) v = tiles;
      if (share < v) v = share;
      parts[k] = static_cast<int>(v);
      // slots of a request have base or base + 1 tiles; `big` of them the latter
      const int nt = static_cast<int>(tiles);
      nbase[k] = nt / parts[k];
      nbig[k] = nt - nbase[k] * parts[k];
      my_maxslot = max(my_maxslot, nbase[k] + (nbig[k] ? 1 : 0));
    }
  }
  // ---- 2b. pieces.  When the decode grid has more CTAs than run at once
  // (C * Hkv > wave), a second wave of whole slots would leave SMs idle, so
  // every slot is cut as finely as allowed (pieces of kMinPieceTiles, at most
  // Q per slot) and the first wave's CTAs share them.  Else, when the slots
  // are uneven (the longest above 5/4 of the mean), no piece may exceed
  // x = ceil(sum tiles / (1.5 C)) tiles, which leaves about 1.5 to 2 waves of
  // pieces -- enough for the longest-first order to even out the CTAs'
  // finishing times; otherwise slots run whole.
  auto pieces_of = [&](int k, int x) {
    return parts[k] ? (parts[k] - nbig[k]) * piece_count(nbase[k], x, p.Q) +
                          (nbig[k] ? nbig[k] * piece_count(nbase[k] + 1, x, p.Q) : 0)
                    : 0;
  };
  int xcut = 1;  // longest piece, in tiles
  int qmax = 1;  // most pieces of one slot
  if (p.Q > 1) {
    int my_nslots = 0;
#pragma unroll
    for (int k = 0; k < kPer; ++k) my_nslots += parts[k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      my_maxslot = max(my_maxslot, __shfl_xor_sync(0xffffffffu, my_maxslot, o));
      my_nslots += __shfl_xor_sync(0xffffffffu, my_nslots, o);
    }
    __syncthreads();  // s_cnt of phase 1 has been read by every warp
    if (lane == 0) {
      s_cnt[warp] = my_maxslot;
      s_scan[0][warp] = my_nslots;
    }
    __syncthreads();
    int mx = max(1, lane < kWarps ? s_cnt[lane] : 0);
    long long ns = lane < kWarps ? s_scan[0][lane] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    ns = warp_sum64(ns);
    xcut = mx;
    if (p.wave > 0 && C * p.Hkv > p.wave)
      xcut = min(mx, kMinPieceTiles);
    else if (4ll * mx * ns > 5ll * sum_tiles)
      xcut = static_cast<int>(min(static_cast<long long>(mx),
                                  max(static_cast<long long>(kMinPieceTiles),
                                      (2 * sum_tiles + 3 * C - 1) / (3 * C))));
    qmax = piece_count(mx, xcut, p.Q);
    __syncthreads();  // s_scan is reused by the block scan below
  }

  // ---- 2c. pieces, partial rows, extra row-chunk items, merge rows per request
  // Merge rows are listed in two runs: rows of requests with at most
  // kWarpMergePieces pieces first (the merge gives each (row, head) a warp),
  // then rows with more (a whole CTA each).
  int my_slots = 0, my_pieces = 0, my_rows = 0, my_extra = 0, my_mfew = 0, my_mmany = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    pcs[k] = pieces_of(k, xcut);
    const int chunks = (L[k] * p.G + p.rpc - 1) / p.rpc;
    my_slots += parts[k];
    my_pieces += pcs[k];
    my_rows += pcs[k] >= 2 ? pcs[k] * L[k] : 0;
    my_extra += pcs[k] * (chunks > 1 ? chunks - 1 : 0);
    my_mfew += (pcs[k] >= 2 && pcs[k] <= kWarpMergePieces) ? L[k] : 0;
    my_mmany += pcs[k] > kWarpMergePieces ? L[k] : 0;
  }

  // ---- 3. exclusive offsets (slots, pieces, partial rows, extra items, merge rows)
  int inc[6] = {my_slots, my_pieces, my_rows, my_extra, my_mfew, my_mmany};
  block_scan<kThreads, 6>(inc, s_scan, s_tot);
  __syncthreads();
  int slot0 = inc[0] - my_slots, piece0 = inc[1] - my_pieces, row0 = inc[2] - my_rows;
  int extra0 = inc[3] - my_extra, mfew0 = inc[4] - my_mfew, mmany0 = s_tot[4] + inc[5] - my_mmany;
  const bool overflow = static_cast<long long>(s_tot[2]) > p.rows_cap ||
                        static_cast<long long>(s_tot[3]) > p.max_extra ||
                        static_cast<long long>(s_tot[4]) + s_tot[5] > p.max_tokens ||
                        static_cast<long long>(s_tot[1]) > C * p.Q;
  if (overflow) {
    // Cannot happen for a plan built with these limits; empty the plan rather
    // than write past the scratch.
#pragma unroll
    for (int k = 0; k < kPer; ++k) parts[k] = pcs[k] = 0;
    slot0 = piece0 = row0 = extra0 = mfew0 = mmany0 = 0;
  }
  const int total_slots = overflow ? 0 : s_tot[0];
  const int total_pieces = overflow ? 0 : s_tot[1];
  const int total_extra = overflow ? 0 : s_tot[3];
  const int total_mfew = overflow ? 0 : s_tot[4];
  const int total_mmany = overflow ? 0 : s_tot[5];
  if (tid == 0 && (bad || overflow)) atomicOr(p.dev.err, PA_DEVERR_PLAN_OVERFLOW);

#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int r = tid * per + k;
    if (k < per && r < n) {
      p.dev.reduce[r] = make_int2(slot0, parts[k]);
      p.dev.snap[r] = make_int2(S[k], L[k]);
      p.dev.preq[r] = make_int2(row0, pcs[k]);
      s_first[r] = slot0;
      s_parts[r] = parts[k];
      s_ctx[r] = S[k];
      s_qlen[r] = L[k];
      s_prow[r] = row0;
      s_pfirst[r] = piece0;
      s_xfirst[r] = extra0;
      s_t0[r] = T0[k];
      if (pcs[k] >= 2) {
        int& m0 = pcs[k] <= kWarpMergePieces ? mfew0 : mmany0;
        for (int i = 0; i < L[k]; ++i)
          p.dev.mrows[m0 + i] = make_int4(r | ((pcs[k] - 1) << 12), i, row0 + i, L[k]);
        m0 += L[k];
      }
      const int chunks = (L[k] * p.G + p.rpc - 1) / p.rpc;
      slot0 += parts[k];
      piece0 += pcs[k];
      row0 += pcs[k] >= 2 ? pcs[k] * L[k] : 0;
      extra0 += pcs[k] * (chunks > 1 ? chunks - 1 : 0);
    }
  }
  if (tid == 0) {
    p.dev.counters[0] = total_extra;
    p.dev.counters[1] = 0;
    p.dev.counters[2] = total_mmany;
    p.dev.counters[3] = total_mfew;
    p.dev.counters[4] = total_pieces;
    p.dev.counters[5] = 0;
  }
  __syncthreads();

  // Lanes of a warp that share a class add their count with one atomic and
  // take consecutive places in lane order (a count in phase 4, a launch
  // position in phase 5).  Counting with one atomic per lane in phase 4 was
  // measured too: the refresh is 0.1-0.5 us shorter, but the changed timing of
  // the warps reorders phase 5's places and the skewed D = 1024 split ran
  // 244 us instead of 234 us.
  auto warp_claim = [&](int cls, bool valid) {
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? cls : -1);
    const int leader = __ffs(peers) - 1;
    int base = 0;
    if (valid && lane == leader) base = atomicAdd(&s_bcnt[cls], __popc(peers));
    base = __shfl_sync(0xffffffffu, base, leader);
    return base + __popc(peers & ((1u << lane) - 1u));
  };
  // Slot `slot` (< total_slots): its request, tile range and the pieces of
  // the request's earlier slots.
  struct SlotInfo { int r, tb, te, q, before; };
  auto slot_info = [&](int slot) {
    SlotInfo o;
    int lo = 0, hi = n;  // last r with s_first[r] <= slot (it has parts > 0)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_first[mid] <= slot)
        lo = mid;
      else
        hi = mid;
    }
    o.r = lo;
    const int pr = s_parts[lo];
    const int j = slot - s_first[lo];
    const int t0 = s_t0[lo];
    const int nt = (s_ctx[lo] - t0 * kTile + kTile - 1) / kTile;
    const int rb = tile_split(j, nt, pr);  // relative to the planned range
    o.tb = t0 + rb;
    o.te = t0 + tile_split(j + 1, nt, pr);
    o.q = piece_count(o.te - o.tb, xcut, p.Q);
    const int base = nt / pr;
    const int qlo = piece_count(base, xcut, p.Q), qhi = piece_count(base + 1, xcut, p.Q);
    o.before = j * qlo + (rb - j * base) * (qhi - qlo);
    return o;
  };
  // Keys [kb, ke) of piece `sub` of a slot, and its launch-order class.
  auto piece_keys = [&](const SlotInfo& o, int sub, int& kb, int& ke) {
    const int nts = o.te - o.tb;
    const long long t0 = o.tb + tile_split(sub, nts, o.q);
    const long long t1 = o.tb + tile_split(sub + 1, nts, o.q);
    kb = static_cast<int>(t0 * kTile);
    ke = static_cast<int>(min(t1 * kTile, static_cast<long long>(s_ctx[o.r])));
    return 127 - length_class(ke - kb);
  };

  // ---- 4. work_info (the plan's task list) and the launch-order class counts
  constexpr int kCached = 4;  // slots per thread kept for phase 5 (C <= 4096)
  SlotInfo cache[kCached];
  for (int s0 = 0, it = 0; s0 < C; s0 += kThreads, ++it) {
    const int slot = s0 + tid;
    const bool act = slot < total_slots;
    SlotInfo o = {0, 0, 0, 0, 0};
    if (act) {
      o = slot_info(slot);
      p.dev.work[slot] = make_int4(o.r, o.tb, o.te, s_ctx[o.r]);
    } else if (slot < C) {
      p.dev.work[slot] = make_int4(-1, 0, 0, 0);
    }
#pragma unroll
    for (int c = 0; c < kCached; ++c)
      if (c == it) cache[c] = o;
    for (int sub = 0; sub < qmax; ++sub) {
      const bool valid = act && sub < o.q;
      int kb = 0, ke = 1, cls = 0;
      if (valid) cls = piece_keys(o, sub, kb, ke);
      warp_claim(cls, valid);
    }
  }
  __syncthreads();
  // ---- 5. launch order: counting sort of the pieces by length class
  if (warp == 0) {  // exclusive prefix over the 128 classes: 4 per lane, then a warp scan
    int v[4], sum = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[k] = s_bcnt[lane * 4 + k];
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
    for (int k = 0; k < 4; ++k) {
      s_bcnt[lane * 4 + k] = pos;
      pos += v[k];
    }
  }
  __syncthreads();
  for (int s0 = 0, it = 0; s0 < C; s0 += kThreads, ++it) {
    const int slot = s0 + tid;
    const bool act = slot < total_slots;
    SlotInfo o = {0, 0, 0, 0, 0};
    if (it < kCached) {
#pragma unroll
      for (int c = 0; c < kCached; ++c)
        if (c == it) o = cache[c];
    } else if (act) {
      o = slot_info(slot);
    }
    for (int sub = 0; sub < qmax; ++sub) {
      const bool valid = act && sub < o.q;
      int kb = 0, ke = 1, cls = 0;
      if (valid) cls = piece_keys(o, sub, kb, ke);
      const int pos = warp_claim(cls, valid);
      if (!valid) continue;
      const int r = o.r;
      const int npieces = (r + 1 < n ? s_pfirst[r + 1] : total_pieces) - s_pfirst[r];
      const int k = o.before + sub;  // piece index within the request
      p.dev.pieces[pos] = make_int4(r, kb, ke, npieces >= 2 ? s_prow[r] + k * s_qlen[r] : -1);
      const int chunks = (s_qlen[r] * p.G + p.rpc - 1) / p.rpc;
      for (int c = 1; c < chunks; ++c)
        p.dev.extra[s_xfirst[r] + k * (chunks - 1) + (c - 1)] = make_int2(pos, c);
    }
  }
}

}  // namespace

cudaError_t launch_plan(const PlanParams& p, cudaStream_t s) {
  // per device: the dynamic shared-memory limit of both planner shapes
  static std::atomic<int> state[kMaxDevices];
  const int smem = 8 * kMaxSeqs * static_cast<int>(sizeof(int));
  int unused = 0;
  const cudaError_t e = per_device_once(state, unused, [&](int&) {
    cudaError_t r =
        cudaFuncSetAttribute(plan_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(plan_kernel<1024>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    return r;
  });
  if (e != cudaSuccess) return e;
  const int dyn = 8 * p.n * static_cast<int>(sizeof(int));
  if (p.n <= 128) return launch_pdl(plan_kernel<128>, dim3(1), dim3(128), dyn, s, p);
  return launch_pdl(plan_kernel<1024>, dim3(1), dim3(1024), dyn, s, p);
}

}  // namespace pa
