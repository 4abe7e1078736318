// pa_split.cuh -- the split-KV paged decode kernel (one CTA per piece -- a plan
// task, or a cut of one -- and kv head; further pieces and row chunks are
// taken from a device counter by CTAs that finish early).
//
// What it computes ("[MiniMax-M3] Route the paged decode to aiter's FlyDSL
// kernel with work planner", sections 1 and 3; vllm-rdna pull 29, Change 1):
// task (r, tile_begin, tile_end, S) of the plan covers keys
// [tile_begin*256, min(tile_end*256, S)) of request r.  For every query row of
// r (token i of L, q head of kv head h) the CTA forms the partial softmax over
// the task's keys that the row may see (key < S - (L-1-i), and within the
// row's sliding window if there is one), and writes either the finished
// output row (when r has a single piece; an attention sink joins its
// denominator there) or a normalised fp32 partial plus its log2-sum-exp for
// the merge kernel.
//
// GB300 mapping:
//  * warp 0 is the producer: it walks the block table (32-entry windows,
//    coalesced) and issues the TMA tile loads (cp.async.bulk.tensor.2d,
//    128-byte swizzle, L2 evict-first; a K cache in the grouped layout
//    [num_blocks, Hkv, D/16, bs, 16] is read as 128-byte rows -- 4 (8 for
//    fp8) keys of one 16-dim group -- in 3-D boxes of every group of a page's
//    keys, also 128-byte swizzled) of the K and V rows of a stage's pages
//    from up to 32 lanes at once -- with pages of only 2-4 KB per head, one
//    issuing lane caps the stream at roughly half the HBM bandwidth -- into a
//    ring of NS stages (32 KB up to head_dim 256; one 16-key tile of K and V
//    for wider heads), completion counted in bytes on an mbarrier;
//  * up to head_dim 128 a second producer warp splits that work (warp 0 the
//    K copies, warp 1 the V copies, each walking the block table itself):
//    issuing holds a warp for about 100-140 cycles per 2 KB box, which kept
//    a CTA left alone at the end of a skewed batch near 25 GB/s; the two
//    warps share a per-CTA limit but overlap enough for about 20% more;
//  * consumer warps form (row group wq) x (key warp wk); every consumer warp
//    takes part in every stage (its key slice: T 16-key tiles handled
//    together -- independent MMA chains, one softmax reduction), so each warp
//    waits on the ring slots strictly in order;
//  * every mbarrier wait is bounded (4 s unless the plan sets another limit):
//    a wait that gives up raises PA_DEVERR_TIMEOUT and aborts the CTA's
//    pipeline (no further copies are issued or consumed); the producer then
//    drains the copies it issued before the CTA exits.  Every named barrier
//    and __syncthreads is still met on that path, so an aborted CTA returns;
//    a test hook (skip_stage) leaves one stage un-issued to exercise it;
//  * QK^T and PV are m16n8k16 tensor-core MMAs in "swap-AB" form: 16 keys
//    (QK) or 16 head dims (PV) on M, the 8 query rows of the group on N, so a
//    GQA group of 8 fills N exactly.  P moves from the QK accumulator to the
//    PV B fragment with movmatrix.trans, never through shared memory;
//  * the online softmax runs in the log2 domain and rescales lazily: the
//    running reference only moves when the tile maximum exceeds it by more
//    than 8 (probabilities stay below 2^8, exact in fp32 accumulators);
//  * fp8 e4m3 caches are converted in registers (cvt.f16x2.e4m3x2, exact) and
//    multiplied in fp16; k_scale is folded into the logit scale and v_scale
//    into the epilogue;
//  * the key warps of a row group are merged through shared memory at the end
//    of a pass;
//  * head dims above 256 are cut into 128- or 256-dim slices, one consumer
//    warp each, whose partial logits are summed through shared memory per
//    stage (see SplitCfg);
//  * a few extra CTAs at the end of the grid write the rows no task writes
//    (graph padding, empty or stale requests); requests with several
//    partitions are combined afterwards by the merge kernel.
#pragma once

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_fused.cuh"
#include "pa_merge.cuh"
#include "pa_split_cfg.h"

namespace pa {

// Byte offset of 16-byte chunk `chunk` of row `row` inside a column block whose
// base is aligned to the swizzle repeat: the TMA 128B (64B) swizzle XORs the
// chunk index with address bits [9:7] ([8:7]).  Adding a multiple of 8 rows to
// `row` only adds 8*SWB per 8 rows, so callers add tile bases separately.
template <int SWB>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  const uint32_t o = static_cast<uint32_t>(row * SWB + chunk * 16);
  constexpr uint32_t mask = (SWB == 128) ? 7u : 3u;
  return o ^ (((o >> 7) & mask) << 4);
}

// Counts a finished CTA (thread 0, after its last claim); the last CTA of the
// grid resets the work counter and this count for the next decode call.
__device__ __forceinline__ void cta_finished(const SplitParams& p) {
  if (atomicAdd(p.plan.counters + 5, 1) == static_cast<int>(gridDim.x) - 1) {
    p.plan.counters[1] = 0;
    p.plan.counters[5] = 0;
  }
}

template <int D, int KVT, int WQ, int KL>
__global__ void __launch_bounds__(SplitCfg<D, KVT, WQ, KL>::THREADS,
                                  SplitCfg<D, KVT, WQ, KL>::MIN_BLOCKS)
    split_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                 const SplitParams p) {
  using Cfg = SplitCfg<D, KVT, WQ, KL>;
  constexpr int NQ = 8 * WQ;  // query rows per pass
  constexpr int T = Cfg::T;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  float* ex = reinterpret_cast<float*>(smem_raw + (base - raw));
  const uint32_t bar_full = base + Cfg::DATA_BYTES;
  const uint32_t bar_empty = bar_full + 8 * Cfg::NS;
  float4* sx = reinterpret_cast<float4*>(smem_raw + (base - raw) + Cfg::DATA_BYTES + 64);
  __shared__ int s_abort;  // set when a bounded wait gave up
  // Both producer warps issue (K copies and V copies) when a stage takes more
  // than one box per tensor; with pages that hold a whole stage (one box
  // each) warp 0 issues both and warp 1 idles.
  const bool dual = Cfg::NPW == 2 && (Cfg::kGroupedK || Cfg::CB > 1 || p.bs < Cfg::KS);
  if (warp == 0 && lane == 0) {  // all of this overlaps the planner's tail
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
    s_abort = 0;
    for (int s = 0; s < Cfg::NS; ++s) {
      mbar_init(bar_full + 8 * s, dual ? 2 : 1);  // one expect-tx arrival per issuing warp
      // released by every consumer warp, or (tensor-memory path) by the commit
      // of the stage's P V
      mbar_init(bar_empty + 8 * s, Cfg::kTc ? 1 : Cfg::NCW);
    }
    if constexpr (Cfg::kTc) {
      const uint32_t b = bar_full + 16 * Cfg::NS;
      for (int i = 0; i < 2; ++i) {
        mbar_init(b + 8 * i, 1);       // S^T buffer i computed (a commit)
        mbar_init(b + 16 + 8 * i, 4);  // P' of a stage of parity i written (each softmax warp)
        mbar_init(b + 32 + 8 * i, 1);  // P V of a stage of parity i completed (a commit)
      }
      mbar_init(b + 48, 1);            // the last commit before the tensor memory is released
    }
    fence_barrier_init();
  }
  pdl_wait();  // the plan (and everything before this kernel) is complete
  // The merge kernel may be scheduled once every CTA of this grid has got
  // here, i.e. once all of them are resident: its CTAs take what is left of
  // the SMs, read the planner's row lists and then wait for this whole grid to
  // complete before they read a partial or reset the work counter that this
  // kernel takes items from.
  pdl_trigger();
  if (blockIdx.x >= static_cast<unsigned>(p.C * p.Hkv)) {  // zero-row CTA
    zero_rows<D>(p, blockIdx.x - p.C * p.Hkv, warp, Cfg::THREADS / 32, lane);
    if constexpr (D <= 256)
      if (p.fused && threadIdx.x == 0) cta_finished(p);
    return;
  }
  if constexpr (Cfg::kTc) {
    // Tensor memory: four regions of 2 TN columns (hi then lo) at multiples of
    // 32 (16 rows) or 64 columns -- S^T buffers 0 and 1, O^T, L^T; two CTAs
    // per SM take at most the SM's 512
    if (warp == Cfg::NPW) tc_alloc(base + Cfg::DATA_BYTES + Cfg::TC_TMEM_SLOT, Cfg::TC_COLS);
    tc_fence_before();
  }
  // Items (piece, kv head) are numbered piece-major: item i is piece i / Hkv,
  // head i % Hkv.  The first `nst` of them belong to CTAs 0..nst-1, one each,
  // and the rest come from the work counter.  nst = C * Hkv (every CTA starts
  // on an item of its own) unless the planner cut the slots into more pieces
  // than C and the grid is more than one wave: then only the CTAs of the
  // first wave own one (a later CTA would run its own after everyone else).
  // Only thread 0 (prologue and claims) uses it.
  int nst = p.C * p.Hkv;
  // This CTA's first item -- item blockIdx, when it is below nst -- read
  // together with the counts it depends on.  Item slots are double-buffered:
  // round k reads slot k & 1 while the producer may already claim round
  // k + 1's item into the other slot.
  __shared__ int s_item[2][4];
  __shared__ int4 s_rec[2];
  __shared__ int s_npieces, s_nextra;
  __shared__ int s_pre;  // 1: the next round's slot already holds its item
  if (threadIdx.x == 0) {
    const int npieces = p.plan.counters[4];
    const int nextra = p.plan.counters[0];
    const int4 rec = p.plan.pieces[blockIdx.x / p.Hkv];  // < C: inside the array
    if (npieces > p.C && p.resident > 0 && p.resident < nst) nst = p.resident;
    s_npieces = npieces;
    s_nextra = nextra;
    s_rec[0] = rec;
    s_pre = 0;
    const int late = npieces * p.Hkv > nst ? npieces * p.Hkv - nst : 0;
    const bool mine = static_cast<int>(blockIdx.x) < nst &&
                      static_cast<int>(blockIdx.x / p.Hkv) < npieces;
    s_item[0][0] = mine ? static_cast<int>(blockIdx.x / p.Hkv) : -1;
    s_item[0][1] = mine ? static_cast<int>(blockIdx.x % p.Hkv) : 0;
    s_item[0][2] = 0;
    s_item[0][3] = (mine || late > 0 || nextra > 0) ? 1 : 0;  // 0: nothing now or later
  }
  __syncthreads();
  // Warp-uniform view of the abort flag; raising it sets PA_DEVERR_TIMEOUT.
  auto aborted = [&]() {
    return __shfl_sync(0xffffffffu, *reinterpret_cast<volatile int*>(&s_abort), 0) != 0;
  };
  auto wait_all = [&](uint32_t bar, uint32_t parity) {
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, parity, p.plan.err, p.wait_ns));
    if (!ok && lane == 0) *reinterpret_cast<volatile int*>(&s_abort) = 1;
    return ok;
  };

  const int G = p.G;
  const int Hkv = p.Hkv;
  int it = 0;      // stages so far (producer and consumers count alike)
  int issued = 0;  // producer: stages [0, issued) were issued (a prefix: issuing stops at an abort)

  // Work items: first this CTA's own (piece, kv head) in launch order -- the
  // planner sorts pieces longest first -- then, until none are left, from one
  // device counter: the items from nst on (in launch order), then the extra
  // row chunks of requests with many query rows.
  // Takes the next item from the device counter into slot `sl` (one thread).
  // The producer calls it as soon as it has issued the last stage of an item,
  // so that the claim and the record load overlap the consumers' last stages;
  // the loop head calls it when that did not happen.
  auto claim_next = [&](int sl) {
    const int npieces = s_npieces, nextra = s_nextra;
    const int late = npieces * Hkv > nst ? npieces * Hkv - nst : 0;
    int pos = -1, hh = 0, chunk = 0, valid = 1;
    if (late == 0 && nextra == 0) {
      valid = 0;
    } else {
      int idx = atomicAdd(p.plan.counters + 1, 1);
      if (idx < late) {
        pos = (nst + idx) / Hkv;
        hh = (nst + idx) % Hkv;
      } else if ((idx -= late) < nextra * Hkv) {
        const int2 e = p.plan.extra[idx / Hkv];
        pos = e.x;
        chunk = e.y;
        hh = idx % Hkv;
      } else {
        valid = 0;
      }
      if (pos >= 0) s_rec[sl] = p.plan.pieces[pos];
    }
    s_item[sl][0] = pos;
    s_item[sl][1] = hh;
    s_item[sl][2] = chunk;
    s_item[sl][3] = valid;
  };
  // What an item covers: request r, kv head h, its rows [row_lo, row_hi) in
  // passes of NQ, keys [kb, ke_task); ok = false when the plan was refreshed
  // from other lengths (the zero CTAs handle the request) or the row chunk is
  // empty.
  struct ItemGeo {
    int r, h, S, row0, L, prow_base, row_lo, row_hi, npass, kb, ke_task;
    bool ok;
  };
  auto item_geo = [&](int sl) {
    ItemGeo q;
    const int4 pc = s_rec[sl];
    q.r = pc.x;
    q.h = s_item[sl][1];
    q.S = p.context_lens[q.r];
    q.row0 = p.cu ? p.cu[q.r] : q.r;
    q.L = p.cu ? p.cu[q.r + 1] - q.row0 : 1;
    const int2 snap = p.plan.snap[q.r];
    q.prow_base = pc.w;
    q.row_lo = s_item[sl][2] * p.rpc;
    q.row_hi = min(q.L * G, q.row_lo + p.rpc);
    q.npass = (q.row_hi - q.row_lo + NQ - 1) / NQ;
    q.kb = pc.y;
    q.ke_task = min(pc.z, q.S);
    q.ok = snap.x == q.S && snap.y == q.L && q.row_lo < q.row_hi;
    return q;
  };
  // Last key any row of pass `pass` of item q may see.
  auto geo_key_end = [&](const ItemGeo& q, int pass) {
    const int last_row = min(q.row_hi, q.row_lo + (pass + 1) * NQ) - 1;
    const int last_tok = last_row / G;
    return min(q.ke_task, q.S - (q.L - 1 - last_tok));
  };
  // Producer: block-table entries [kb / bs, + 64) of the piece in item slot
  // sl, 32 per register -- read from the piece record alone, so that these
  // loads are in flight together with the length checks of item_geo.
  auto bt_window = [&](int sl, int& cur, int& nxt) {
    const int4 pc = s_rec[sl];
    const int* bt = p.block_tables + static_cast<size_t>(pc.x) * p.max_blocks;
    const int np = min((pc.z + p.bs - 1) / p.bs, p.max_blocks);
    const int w0 = pc.y / p.bs;
    cur = (w0 + lane < np) ? __ldg(bt + w0 + lane) : -1;
    nxt = (w0 + 32 + lane < np) ? __ldg(bt + w0 + 32 + lane) : -1;
  };
  // Producer: issues stage s of a pass over keys [q.kb, ke) into ring stage
  // `it` (the caller advances it); win / cur / nxt: the block-table window.
  const uint64_t policy = l2_evict_first_policy();
  const int box_rows = p.bs < Cfg::KS ? p.bs : Cfg::KS;
  const uint32_t box_bytes = static_cast<uint32_t>(box_rows * Cfg::SWB);
  auto issue_stage = [&](const ItemGeo& q, int s, int ke, int& win, int& cur, int& nxt) {
    const int bs = p.bs;
    const int buf = it % Cfg::NS;
    if (warp == 1 && !dual) return;
    if (aborted()) return;
    if (it >= Cfg::NS && !wait_all(bar_empty + 8 * buf, ((it / Cfg::NS) & 1) ^ 1)) return;
    issued = it + 1;
    // Test hook: this stage is counted as issued (the drain waits on it) but
    // neither copied nor armed, so every wait on it gives up after wait_ns.
    if (it == p.skip_stage) return;
    const int* bt = p.block_tables + static_cast<size_t>(q.r) * p.max_blocks;
    const int npages = min((q.S + bs - 1) / bs, p.max_blocks);
    const int key0 = q.kb + s * Cfg::KS;
    const int nkeys = min(Cfg::KS, ke - key0);
    const int nbox = (nkeys + box_rows - 1) / box_rows;
    while (key0 / bs >= win + 32) {  // a stage spans at most 16 pages: [win, win + 48)
      win += 32;
      cur = nxt;
      nxt = (win + 32 + lane < npages) ? __ldg(bt + win + 32 + lane) : -1;
    }
    // copy c of this stage (one per lane): K/V by c & 1, column block and
    // row box from c >> 1; with grouped K, lanes [0, MTS) copy K -- one box
    // of 16 keys by every 16-dim group each -- and the others V.  With two
    // producer warps, warp 0 copies K and warp 1 V, one box per lane.
    const int c = lane;
    bool is_v;
    int rb, cb;
    if (dual) {
      is_v = warp == 1;
      rb = (Cfg::kGroupedK && !is_v) ? c : c / Cfg::CB;
      cb = (Cfg::kGroupedK && !is_v) ? 0 : c % Cfg::CB;
    } else if constexpr (Cfg::kGroupedK) {
      is_v = c >= Cfg::MTS;
      rb = is_v ? (c - Cfg::MTS) / Cfg::CB : c;
      cb = is_v ? (c - Cfg::MTS) % Cfg::CB : 0;
    } else {
      is_v = (c & 1) != 0;
      rb = (c >> 1) / Cfg::CB;
      cb = (c >> 1) % Cfg::CB;
    }
    const int key = key0 + rb * ((Cfg::kGroupedK && !is_v) ? 16 : box_rows);
    const int pidx = key / bs;
    const int widx = min(pidx - win, 63);
    const int pc = __shfl_sync(0xffffffffu, cur, widx & 31);
    const int pn = __shfl_sync(0xffffffffu, nxt, widx & 31);
    const int page = widx < 32 ? pc : pn;
    const int nbox_k = Cfg::kGroupedK ? (nkeys + 15) / 16 : nbox;  // grouped K: 16-key boxes
    if (lane == 0) {
      // bytes this warp's copies bring: K's and V's, or its own tensor's
      const uint32_t kbytes = Cfg::kGroupedK ? nbox_k * 16 * Cfg::ROW : nbox * box_bytes * Cfg::CB;
      const uint32_t vbytes = nbox * box_bytes * Cfg::CB;
      mbar_arrive_expect_tx(bar_full + 8 * buf,
                            !dual ? kbytes + vbytes : (warp == 0 ? kbytes : vbytes));
    }
    __syncwarp();
    if (rb < ((Cfg::kGroupedK && !is_v) ? nbox_k : nbox)) {
      const bool bad = page < 0 || page >= p.num_blocks || pidx >= p.max_blocks;
      if (bad) atomicOr(p.plan.err, PA_DEVERR_BAD_PAGE);  // the copy reads zeros
      if (Cfg::kGroupedK && !is_v) {
        // coordinates {byte in 128-byte row, 128-byte row of the group in
        // the page, (page * Hkv + head) * D/16 + group}
        const int slab = bad ? p.num_blocks * p.Hkv : page * p.Hkv + q.h;
        const uint32_t dst = base + buf * Cfg::STAGE_BYTES +
                             static_cast<uint32_t>(rb * 16 * Cfg::ROW);
        tma_load_3d(dst, &tmk, 0, (key % bs) * Cfg::GRP / 128, slab * (D / 16),
                    bar_full + 8 * buf, policy);
      } else {
        const int y = bad ? p.total_rows : (page * p.Hkv + q.h) * bs + (key % bs);
        const uint32_t dst = base + buf * Cfg::STAGE_BYTES + (is_v ? Cfg::TILE_BYTES : 0) +
                             cb * Cfg::BLOCK_BYTES + static_cast<uint32_t>(rb * box_rows * Cfg::SWB);
        tma_load_2d(dst, is_v ? &tmv : &tmk, cb * (Cfg::SWB / Cfg::ESZ), y, bar_full + 8 * buf,
                    policy);
      }
    }
  };
  // Producer: stages of the coming pass issued ahead, and the block-table
  // window after them.
  int pre_n = 0, pre_win = 0, pre_cur = -1, pre_nxt = -1;

  for (int round = 0;; ++round) {
    if (round > 0) {  // round 0's item was set up with the prologue
      __syncthreads();  // everyone has read the previous item
      if (threadIdx.x == 0) {
        if (s_pre)
          s_pre = 0;  // claimed ahead by the producer
        else
          claim_next(round & 1);
      }
      __syncthreads();
    }
    const int sl = round & 1;
    if (!s_item[sl][3]) break;
    if (s_item[sl][0] < 0) continue;  // no piece for this CTA: look for extra items
    // Block-table window of the piece's first pages, loaded by the producer
    // alongside the length checks (entries past the piece's end are not used).
    int bt_cur = -1, bt_nxt = -1;
    if (warp < Cfg::NPW) bt_window(sl, bt_cur, bt_nxt);
    const ItemGeo cg = item_geo(sl);
    const int h = cg.h;
    const int r = cg.r;

    // A plan refreshed from other lengths: the split kernel's zero CTAs zero
    // these rows and report it; this piece does nothing.  Likewise a row chunk
    // past the request's rows.
    if (!cg.ok) continue;
    const int S = cg.S;
    const int row0 = cg.row0;
    const int L = cg.L;
    const int prow_base = cg.prow_base;  // -1: write the output rows directly
    const int row_lo = cg.row_lo;        // this item's rows [row_lo, row_hi)
    const int row_hi = cg.row_hi;
    const int npass = cg.npass;
    const int kb = cg.kb;                // first key of the piece
    const int ke_task = cg.ke_task;
    auto pass_key_end = [&](int pass) { return geo_key_end(cg, pass); };

  if (warp < Cfg::NPW) {
    // ------------------------------------------------------------ producer
    for (int pass = 0; pass < npass; ++pass) {
      const int ke = pass_key_end(pass);
      const int nst = ke > kb ? (ke - kb + Cfg::KS - 1) / Cfg::KS : 0;
      // block-table entries [win, win + 64) live in cur / nxt
      int win = kb / p.bs, cur = bt_cur, nxt = bt_nxt, s0 = 0;
      if (pre_n > 0) {  // the first stages were issued at the end of the last pass
        s0 = pre_n;
        win = pre_win;
        cur = pre_cur;
        nxt = pre_nxt;
        pre_n = 0;
      }
      for (int s = s0; s < nst; ++s, ++it) issue_stage(cg, s, ke, win, cur, nxt);
      // Last stage of the item issued: claim the next one (into the other
      // slot) while the consumers finish this one.
      if (pass == npass - 1 && warp == 0 && lane == 0 &&
          *reinterpret_cast<volatile int*>(&s_abort) == 0) {
        claim_next(sl ^ 1);
        s_pre = 1;
      }
      // the other producer warp reads the claimed item below
      if constexpr (Cfg::NPW > 1) named_barrier_sync(6, 32 * Cfg::NPW);
      if constexpr (Cfg::kPreIssue) {
        // While the consumers finish this pass, issue the first stages (at
        // most NS - 1) of the next one -- this item's next row pass, or the
        // next item's first -- into the ring slots they have released.  The
        // slot of this pass's last stage holds their exchange and is
        // released after it.
        __syncwarp();  // lane 0's claim is visible to the warp
        if (nst > 0 && !aborted()) {
          ItemGeo nq = cg;
          bool have = pass + 1 < npass;
          int npass_idx = pass + 1;
          int ncur = bt_cur, nnxt = bt_nxt;
          if (!have && s_item[sl ^ 1][3] && s_item[sl ^ 1][0] >= 0) {
            bt_window(sl ^ 1, ncur, nnxt);
            nq = item_geo(sl ^ 1);
            have = nq.ok;
            npass_idx = 0;
          }
          if (have) {
            const int nke = geo_key_end(nq, npass_idx);
            const int nn = nke > nq.kb ? (nke - nq.kb + Cfg::KS - 1) / Cfg::KS : 0;
            const int np = nn < Cfg::NS - 1 ? nn : Cfg::NS - 1;
            int nwin = nq.kb / p.bs;
            for (int s = 0; s < np; ++s, ++it) issue_stage(nq, s, nke, nwin, ncur, nnxt);
            pre_n = np;
            pre_win = nwin;
            pre_cur = ncur;
            pre_nxt = nnxt;
          }
        }
      }
      __syncthreads();  // pairs with the consumers' end-of-pass barrier
    }
  } else if constexpr (Cfg::kTc) {
  // ------------------------------- consumers on tensor memory (tcgen05), fp8
  // Warp NPW issues the MMAs (one thread); the next four warps -- one per
  // tensor-memory lane quadrant -- do the softmax, one thread per key of a
  // 128-key stage (per head dim in the epilogue).  q and P' are held as
  // e4m3 hi + lo pairs stacked along the MMA's N (2 TN columns: hi rows,
  // then lo rows), so every product is one MMA per 32-key (or 32-dim) step,
  // and the two halves of a result are added where they are read.
  // Stage g of the pass:
  //   S^T[128 keys x 2TN] = K [q_hi; q_lo]^T into S buffer g & 1 (A = the K
  //     tile, K-major; B = q * 2^qexp, K-major);
  //   P' = 64 * 2^(logit - m_ref) for every key and row (f16 exponential),
  //     as e4m3 hi and lo, written over the stage's K tile (dead once S is
  //     computed): the 2 TN bytes of key k -- hi for every row, then lo --
  //     in chunks of 16 (16 of the MMA's N rows each), chunk c at c * 2048
  //     + k * 16 (MN-major, no swizzle), so each softmax thread stores whole
  //     16-byte rows;
  //   O^T[128 dims x 2TN] += V^T P'^T (A = the V tile read MN-major) and,
  //   for 32-row passes, L^T[128 x 2TN] += 1 P'^T (A = a block of ones read
  //     for all 128 rows): L is every row's sum of the very weights O was
  //     accumulated with (for fewer rows each softmax thread sums its key's
  //     share); the commit frees the ring slot.
  // The issuing thread runs S(g + 2) as soon as that stage has landed and
  // stage g's P' is written (S buffer g & 1 then free) -- the softmax warps
  // wait on it first -- and P V(g) as soon as P'(g) is written, which
  // releases the ring slot; so the softmax of stage g + 1 works on an S
  // computed while stage g's softmax ran.  A row's reference m_ref moves (O and L rescaled) only when a logit
  // exceeds it by more than 2.8 (log2 units): P' stays below 2^8.8, inside
  // e4m3's range (448).
  // Barriers (by stage parity where two operations of a kind can be
  // outstanding): S computed [2], P' written [2], P V done [2], and one for
  // the last commit before the tensor memory is released.
  constexpr int TN = Cfg::TN;
  constexpr int TN2 = 2 * TN;
  const int ct = threadIdx.x - 32 * Cfg::NPW;  // consumer thread
  const int cw = warp - Cfg::NPW;              // 0: the MMA warp
  const int st = ct - 32;                      // softmax thread
  const int sw = cw - 1;                       // softmax warp
  const int quad = warp & 3;                   // the TMEM lane quadrant this warp may access
  const int kk = quad * 32 + lane;             // its key in a stage / its head dim in the epilogue
  const float NEG_INF = -__int_as_float(0x7f800000);
  const float POS_INF = __int_as_float(0x7f800000);
  uint8_t* smb = smem_raw + (base - raw);
  const uint32_t q_hi = base + Cfg::DATA_BYTES + Cfg::TC_Q_OFF;
  const uint32_t q_lo = q_hi + TN * 128;
  const uint32_t ones = base + Cfg::DATA_BYTES + Cfg::TC_ONES_OFF;
  int* s_lim = reinterpret_cast<int*>(smb + Cfg::DATA_BYTES + Cfg::TC_ARR_OFF);
  int* s_llo = s_lim + 32;
  float* s_mref = reinterpret_cast<float*>(s_llo + 32);  // the row's reference m_ref
  float* s_nm = s_mref + 32;                             // 6 - m_ref (log2 of 64, less m_ref)
  float* s_fac = s_nm + 32;                              // rescale factors, then row sums
  long long* s_off = reinterpret_cast<long long*>(s_fac + 32);  // epilogue: a row's element offset
  float* s_scl = reinterpret_cast<float*>(s_off + 32);          // epilogue: a row's scale
  float* s_red = reinterpret_cast<float*>(smb + Cfg::DATA_BYTES + Cfg::TC_RED_OFF);  // [4 warps][32]
  const uint32_t bar_s = bar_full + 16 * Cfg::NS;
  const uint32_t bar_p = bar_s + 16;
  const uint32_t bar_o = bar_p + 16;
  const volatile int* abort_flag = reinterpret_cast<volatile int*>(&s_abort);
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smb + Cfg::DATA_BYTES + Cfg::TC_TMEM_SLOT);
  const uint32_t tl = tmem + (static_cast<uint32_t>(quad * 32) << 16);  // this warp's lanes
  // tensor-memory regions (each 2 TN columns, hi then lo) at multiples of CS:
  // S buffers 0 and 1, O^T, L^T
  constexpr int CS = TN2 <= 32 ? 32 : 64;
  constexpr uint32_t kColO = 2 * CS, kColL = 3 * CS;
  constexpr uint32_t kIdQK = tc_idesc(0, 0, TN2, 128);  // K (K-major) x q (K-major)
  constexpr uint32_t kIdPV = tc_idesc(1, 1, TN2, 128);  // V^T (MN-major) x P' (MN-major)
  constexpr uint32_t kIdL = tc_idesc(0, 1, TN2, 128);   // ones (K-major) x P' (MN-major)
  constexpr bool kRsMma = Cfg::kTcRowSumMma;            // row sums by MMA, else per thread
  // Softmax warps: a bounded wait that also ends once the pipeline aborted
  // (warp-uniform result; a failure raises the abort).
  auto wait_sm = [&](uint32_t bar, uint32_t parity) {
    const bool ok = __all_sync(0xffffffffu, mbar_wait_or_abort(bar, parity, p.plan.err, p.wait_ns, abort_flag));
    if (!ok && lane == 0) *reinterpret_cast<volatile int*>(&s_abort) = 1;
    return ok;
  };
  tc_fence_after();  // the tensor-memory address written at allocation

  for (int pass = 0; pass < npass; ++pass) {
    const int pass_base = row_lo + pass * NQ;
    const int ke = pass_key_end(pass);
    const int nst = ke > kb ? (ke - kb + Cfg::KS - 1) / Cfg::KS : 0;

    float qs = 1.f;
    if (cw > 0) {
      // ---- rows of the pass: key limits; q * 2^qexp as e4m3 hi + lo (exact
      // for bf16 / fp16 q up to the last bits of elements 2^10 below the largest)
      if (st < TN) {
        const int n = pass_base + st;
        const int K = S - (L - 1 - n / G);
        s_lim[st] = (st < NQ && n < row_hi) ? min(ke_task, K) : kb;  // rows past the pass: padding
        s_llo[st] = p.window > 0 ? max(0, K - p.window) : 0;
        s_mref[st] = NEG_INF;
        s_nm[st] = POS_INF;
      }
      if (kRsMma && st < 64)  // the block of e4m3 ones (0x38) read as every row of L's A operand
        *reinterpret_cast<uint4*>(smb + (ones - base) + st * 16) =
            make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
      float qv[32];
      const int qrow = st >> 2, qpart = st & 3;  // 32 head dims [32 qpart, +32) of row qrow
      float amax = 0.f;
      {
        const int n = pass_base + qrow;
        const int tok = n / G;
        const bool ok = qrow < NQ && n < row_hi && row0 + tok < p.num_tokens;
        const size_t qoff = ok ? (static_cast<size_t>(row0 + tok) * p.Hq + h * G + n % G) * D + 32 * qpart : 0;
        const uint4* qp = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) + qoff);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 w = ok ? qp[i] : make_uint4(0u, 0u, 0u, 0u);
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float2 f;
            if (p.out_f16) {
              f = __half22float2(*reinterpret_cast<const __half2*>(&ws[j]));
            } else {
              const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&ws[j]);
              f = make_float2(__low2float(b), __high2float(b));
            }
            qv[8 * i + 2 * j] = f.x;
            qv[8 * i + 2 * j + 1] = f.y;
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (lane == 0) s_red[sw * 32] = amax;
      named_barrier_sync(2, 128);
      amax = fmaxf(fmaxf(s_red[0], s_red[32]), fmaxf(s_red[64], s_red[96]));
      int qexp = 0;  // q is scaled by 2^qexp: its largest element lands in [128, 256)
      if (amax > 0.f) {
        int x;
        frexpf(amax, &x);
        qexp = min(100, max(-100, 8 - x));
      }
      qs = exp2f(static_cast<float>(qexp));
      if (qrow < TN) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {  // two 16-byte chunks (16 dims each) of the row
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int i = 16 * c + 4 * w;
            const float a0 = qv[i] * qs, a1 = qv[i + 1] * qs, a2 = qv[i + 2] * qs, a3 = qv[i + 3] * qs;
            const uint32_t h01 = f32x2_to_e4m3x2(a0, a1), h23 = f32x2_to_e4m3x2(a2, a3);
            const float2 r01 = e4m3x2_to_f32x2(h01), r23 = e4m3x2_to_f32x2(h23);
            const uint32_t l01 = f32x2_to_e4m3x2(a0 - r01.x, a1 - r01.y);
            const uint32_t l23 = f32x2_to_e4m3x2(a2 - r23.x, a3 - r23.y);
            hw[w] = h01 | (h23 << 16);
            lw[w] = l01 | (l23 << 16);
          }
          const uint32_t off = static_cast<uint32_t>(qrow * 128 + (((2 * qpart + c) ^ (qrow & 7)) << 4));
          *reinterpret_cast<uint4*>(smb + (q_hi - base) + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(smb + (q_lo - base) + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
      fence_proxy_async_smem();  // q and the ones are read by the tensor cores
    }
    named_barrier_sync(1, 160);  // q, the ones and the row limits are written

    if (cw == 0) {
      // ------------------------------------------------------- MMA issuer
      if (lane == 0 && nst > 0) {  // one lane: no warp-collective calls in here
        const uint64_t dq = tc_desc(q_hi, 16, 1024);  // +2 per 32-byte step along K
        const uint64_t d1 = tc_desc(ones, 16, 0);     // SBO 0: one 8-row block for all 128 rows
        // Two kinds of work, taken as their inputs become ready, S first
        // (the softmax warps wait on it): S(nq) = K [q_hi; q_lo]^T once
        // stage nq has landed and S buffer nq & 1 is free (stage nq - 2's P'
        // written, i.e. np >= nq - 1), and P V(np) once P'(np) is written
        // (its commit frees the ring slot).
        // Short suspending tries on both; a wait without progress for
        // wait_ns gives up.
        int np = 0, nq = 0;
        bool ok = true;
        unsigned long long t_idle = 0;
        while (np < nst) {
          bool did = false;
          if (nq < nst && nq <= np + 1) {
            const int g = it + nq;
            const int slot = g % Cfg::NS;
            if (mbar_try_wait_hint(bar_full + 8 * slot, (g / Cfg::NS) & 1, 20)) {
              tc_fence_after();
              const uint64_t dk = tc_desc(base + slot * Cfg::STAGE_BYTES, 16, 1024);
              const uint32_t sd = tmem + static_cast<uint32_t>((g & 1) * CS);
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) tc_mma_e4m3(sd, dk + 2 * ks, dq + 2 * ks, kIdQK, ks > 0);
              tc_commit(bar_s + 8 * (g & 1));
              ++nq;
              did = true;
            }
          }
          if (!did && np < nq) {
            const int g = it + np;
            if (mbar_try_wait_hint(bar_p + 8 * (g & 1), (g >> 1) & 1, 20)) {
              // ---- O^T += V^T P'^T and L^T += 1 P'^T; the commit frees the ring slot
              tc_fence_after();
              const int slot = g % Cfg::NS;
              const uint32_t kt = base + slot * Cfg::STAGE_BYTES;
              const uint64_t dv = tc_desc(kt + Cfg::TILE_BYTES, 16, 1024);  // +256 per 32 keys
              const uint64_t dp = tc_desc(kt, 128, 2048, 0u);               // +32 per 32 keys
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                tc_mma_e4m3(tmem + kColO, dv + 256 * ks, dp + 32 * ks, kIdPV, np > 0 || ks > 0);
              if constexpr (kRsMma) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                  tc_mma_e4m3(tmem + kColL, d1 + 2 * ks, dp + 32 * ks, kIdL, np > 0 || ks > 0);
              }
              tc_commit(bar_empty + 8 * slot);
              tc_commit(bar_o + 8 * (g & 1));
              ++np;
              did = true;
            }
          }
          if (did) {
            t_idle = 0;
          } else {
            if (*abort_flag) {
              ok = false;
              break;
            }
            const unsigned long long t = global_ns();
            if (t_idle == 0) {
              t_idle = t;
            } else if (t - t_idle > p.wait_ns) {
              atomicOr(p.plan.err, PA_DEVERR_TIMEOUT);
              ok = false;
              break;
            }
          }
        }
        if (!ok) *reinterpret_cast<volatile int*>(&s_abort) = 1;
      }
      __syncwarp();
    } else {
      // ----------------------------------------------------------- softmax
      const float c2 = p.scale_log2 / qs;  // logit (log2 units) = S^T * c2
      int vis_lo = 0, vis_hi = 0x7fffffff;  // keys every real row of the pass sees
      for (int j = 0; j < TN; ++j) {
        if (j < NQ && pass_base + j < row_hi) {
          vis_lo = max(vis_lo, s_llo[j]);
          vis_hi = min(vis_hi, s_lim[j]);
        }
      }
      // P' = 64 * 2^(logit - m_ref) = 2^(S * c2 + 6 - m_ref) for every row,
      // as f16 pairs (rows 2i, 2i + 1); masked keys give 0.  Returns whether
      // some P' exceeds 2^8.8 (e4m3's largest is 448): the reference must
      // move first.
      auto make_p = [&](const float (&sv)[TN], bool sfull, int kabs, int nkeys, uint32_t (&ph)[TN / 2]) {
        const float4* nm4 = reinterpret_cast<const float4*>(s_nm);
        uint32_t mx = 0u;
#pragma unroll
        for (int q4 = 0; q4 < TN / 4; ++q4) {
          const float4 nm = nm4[q4];
          float a[4] = {fmaf(sv[4 * q4], c2, nm.x), fmaf(sv[4 * q4 + 1], c2, nm.y),
                        fmaf(sv[4 * q4 + 2], c2, nm.z), fmaf(sv[4 * q4 + 3], c2, nm.w)};
          if (!sfull) {
            const int4 lim = reinterpret_cast<const int4*>(s_lim)[q4];
            const int4 llo = reinterpret_cast<const int4*>(s_llo)[q4];
            const bool in = kk < nkeys;
            if (!(in && kabs < lim.x && kabs >= llo.x)) a[0] = NEG_INF;
            if (!(in && kabs < lim.y && kabs >= llo.y)) a[1] = NEG_INF;
            if (!(in && kabs < lim.z && kabs >= llo.z)) a[2] = NEG_INF;
            if (!(in && kabs < lim.w && kabs >= llo.w)) a[3] = NEG_INF;
          }
          ph[2 * q4] = ex2_f16x2(f32x2_to_f16x2(a[0], a[1]));
          ph[2 * q4 + 1] = ex2_f16x2(f32x2_to_f16x2(a[2], a[3]));
          mx = max_f16x2(mx, max_f16x2(ph[2 * q4], ph[2 * q4 + 1]));
        }
        const float2 m2 = __half22float2(*reinterpret_cast<const __half2*>(&mx));
        return fmaxf(m2.x, m2.y) > 445.f;
      };
      float lp[kRsMma ? 1 : TN];  // (row sums per thread) this key's share of each row's sum
#pragma unroll
      for (int j = 0; j < (kRsMma ? 1 : TN); ++j) lp[j] = 0.f;
      for (int s = 0; s < nst; ++s) {
        const int g = it + s;
        const int slot = g % Cfg::NS;
        const int sb = g & 1;
        const uint32_t kt = base + slot * Cfg::STAGE_BYTES;
        const uint32_t vt = kt + Cfg::TILE_BYTES;
        const int key0 = kb + s * Cfg::KS;
        const int nkeys = min(Cfg::KS, ke - key0);
        const int kabs = key0 + kk;
        // every key of the stage visible to every row: no masks
        const bool sfull = nkeys == Cfg::KS && key0 >= vis_lo && key0 + Cfg::KS <= vis_hi;
        const bool live = !aborted() && wait_sm(bar_s + 8 * sb, (g >> 1) & 1);
        float sv[TN];
        uint32_t ph[TN / 2];
        bool over = false;  // some P' would exceed 2^8.8 (e4m3's largest is 448)
        if (live) {
          tc_fence_after();
          uint32_t a[TN2];
          tc_ld<TN2>(tl + static_cast<uint32_t>(sb * CS), a);
#pragma unroll
          for (int j = 0; j < TN; ++j) sv[j] = __uint_as_float(a[j]) + __uint_as_float(a[TN + j]);
          over = make_p(sv, sfull, kabs, nkeys, ph);
        } else {
#pragma unroll
          for (int j = 0; j < TN; ++j) sv[j] = 0.f;
#pragma unroll
          for (int j = 0; j < TN / 2; ++j) ph[j] = 0u;
        }
        if (named_barrier_or(2, 128, over)) {
          // A new reference per row: the running maximum; O and L rescaled.
          // Kept compact (it runs on few stages): the row maxima go through
          // shared memory -- the stage's K tile, dead since S was computed
          // and not yet overwritten by P' -- as [TN rows][128 keys] floats,
          // 16-byte groups XOR-swizzled by the row so that the readers below
          // (8 rows per warp, 4 threads per row) hit distinct banks.
          float* tt = reinterpret_cast<float*>(smb + (kt - base));
#pragma unroll
          for (int j = 0; j < TN; ++j) {
            bool vis = live && kk < nkeys;
            if (!sfull) vis = vis && kabs < s_lim[j] && kabs >= s_llo[j];
            tt[j * 128 + (kk ^ ((j & 7) << 2))] = vis ? sv[j] * c2 : NEG_INF;
          }
          named_barrier_sync(2, 128);
          if (st < 4 * TN) {  // 4 threads per row, 32 keys (8 float4) each
            const int j = st >> 2, part = st & 3;
            float m = NEG_INF;
#pragma unroll 1
            for (int i = 0; i < 8; ++i) {
              const int f4 = (part * 8 + i) ^ (j & 7);
              const float4 v = reinterpret_cast<const float4*>(tt + j * 128)[f4];
              m = fmaxf(m, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
            }
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            if (part == 0) {
              const float mo = s_mref[j];
              const float mn = fmaxf(mo, m);
              s_fac[j] = (mo == NEG_INF) ? 0.f : fast_exp2(mo - mn);
              s_mref[j] = mn;
              s_nm[j] = (mn == NEG_INF) ? POS_INF : 6.f - mn;
            }
          }
          named_barrier_sync(2, 128);
          if constexpr (!kRsMma) {
            const float4* f4 = reinterpret_cast<const float4*>(s_fac);
#pragma unroll
            for (int q4 = 0; q4 < TN / 4; ++q4) {
              const float4 f = f4[q4];
              lp[4 * q4] *= f.x;
              lp[4 * q4 + 1] *= f.y;
              lp[4 * q4 + 2] *= f.z;
              lp[4 * q4 + 3] *= f.w;
            }
          }
          // the previous stage's P V (the only one that can be outstanding)
          if (s > 0 && wait_sm(bar_o + 8 * ((g - 1) & 1), ((g - 1) >> 1) & 1)) {
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < (kRsMma ? 2 : 1) * TN2; c += 16) {  // O hi, O lo (, L hi, L lo)
              const uint32_t col = (c < TN2 ? kColO + c : kColL + (c - TN2));
              uint32_t ov[16];
              tc_ld<16>(tl + col, ov);
#pragma unroll
              for (int i = 0; i < 16; ++i)
                ov[i] = __float_as_uint(__uint_as_float(ov[i]) * s_fac[(c % TN2 + i) % TN]);
              tc_st<16>(tl + col, ov);
            }
          }
          make_p(sv, sfull, kabs, nkeys, ph);  // every P' is now at most 2^8.8
        }
        if constexpr (!kRsMma) {
#pragma unroll
          for (int i = 0; i < TN / 2; ++i) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ph[i]));
            lp[2 * i] += f.x;
            lp[2 * i + 1] += f.y;
          }
        }
        // P' as e4m3 hi + lo: the words of 4 rows' hi bytes, then of their lo
        // bytes, 4 words per 16-byte store
        if (!aborted()) {
          uint32_t pw[TN / 2];
#pragma unroll
          for (int w = 0; w < TN / 4; ++w) {
            const uint32_t x0 = ph[2 * w], x1 = ph[2 * w + 1];
            const uint32_t h0 = f16x2_to_e4m3x2(x0), h1 = f16x2_to_e4m3x2(x1);
            const uint32_t l0 = f16x2_to_e4m3x2(sub_f16x2(x0, e4m3x2_to_f16x2(h0)));
            const uint32_t l1 = f16x2_to_e4m3x2(sub_f16x2(x1, e4m3x2_to_f16x2(h1)));
            pw[w] = h0 | (h1 << 16);
            pw[TN / 4 + w] = l0 | (l1 << 16);
          }
#pragma unroll
          for (int c = 0; c < TN / 8; ++c)
            *reinterpret_cast<uint4*>(smb + (kt - base) + static_cast<uint32_t>(c * 2048 + kk * 16)) =
                make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
          if (kk >= nkeys) {  // keys past the piece: their V rows may hold anything (0 * NaN)
            uint4* vr = reinterpret_cast<uint4*>(smb + (vt - base) + kk * 128);
#pragma unroll
            for (int i = 0; i < 8; ++i) vr[i] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        fence_proxy_async_smem();  // P' and the zeroed rows are read by the tensor cores
        tc_fence_before();         // the S reads (and O / L rescale) precede the MMAs that follow
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_p + 8 * sb);
      }

      // ---------------------------------------------------------- epilogue
      // the last P V (and L) is complete, and with it every earlier one
      const int gl = it + nst - 1;
      const bool have_o = nst > 0 && !aborted() && wait_sm(bar_o + 8 * (gl & 1), (gl >> 1) & 1);
      tc_fence_after();
      if constexpr (kRsMma) {
        if (sw == 0) {  // row sums: every lane of L holds them all
          uint32_t a[TN2];
          if (have_o) {
            tc_ld<TN2>(tl + kColL, a);
          } else {
#pragma unroll
            for (int j = 0; j < TN2; ++j) a[j] = 0u;
          }
          if (lane == 0) {
#pragma unroll
            for (int j = 0; j < TN; ++j) s_fac[j] = __uint_as_float(a[j]) + __uint_as_float(a[TN + j]);
          }
        }
        named_barrier_sync(2, 128);
      } else {
        // row sums: the threads' shares, over the warp by a transpose-reduce
        // (each exchange halves the rows a lane holds: TNP - 1 shuffles in
        // all, lane l ending with row l of TNP = 32, or row l / 2 of 16),
        // then over the 4 warps
        constexpr int TNP = TN <= 16 ? 16 : 32;
        float v[TNP];
#pragma unroll
        for (int j = 0; j < TNP; ++j) v[j] = j < TN ? lp[j] : 0.f;
#pragma unroll
        for (int o = 16, n = TNP; n > 1; o >>= 1, n >>= 1) {
          const bool up = (lane & o) != 0;
#pragma unroll
          for (int i = 0; i < n / 2; ++i) {
            const float send = up ? v[i] : v[i + n / 2];
            const float keep = up ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
        }
        if constexpr (TNP == 16) v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
        const int row = TNP == 32 ? lane : lane >> 1;
        if (row < TN && (TNP == 32 || (lane & 1) == 0)) s_red[sw * 32 + row] = v[0];
        named_barrier_sync(2, 128);
        if (st < TN) s_fac[st] = s_red[st] + s_red[32 + st] + s_red[64 + st] + s_red[96 + st];
        named_barrier_sync(2, 128);
      }
      // Per row, once (thread st = row): where it goes and by what it is
      // scaled (1 / l with the sink, v_scale, the factor 64 of P'; 0 for a
      // row with no visible key), and a partial's log2-sum-exp.
      if (st < TN) {
        const int j = st;
        const int n = pass_base + j;
        long long off = -1;
        float scl = 0.f;
        if (j < NQ && n < row_hi) {
          const int tok = n / G;
          const int hq = h * G + n % G;
          const float M = s_mref[j];
          float lsum = M != NEG_INF ? s_fac[j] * (1.f / 64.f) : 0.f;  // the row sums carry the 64 of P'
          if (prow_base < 0) {
            float f = 1.f;
            if (p.sinks) f = add_sink(M, __ldg(p.sinks + hq) * 1.4426950408889634f, lsum);
            const float inv = lsum > 0.f ? p.v_scale / (64.f * lsum) : 0.f;
            scl = M != NEG_INF ? f * inv : 0.f;
            const int trow = row0 + tok;
            if (trow >= p.num_tokens)
              atomicOr(p.plan.err, PA_DEVERR_PLAN_OVERFLOW);
            else
              off = (static_cast<long long>(trow) * p.Hq + hq) * D;
          } else {
            const float inv = lsum > 0.f ? p.v_scale / (64.f * lsum) : 0.f;
            scl = M != NEG_INF ? inv : 0.f;
            const long long prow = static_cast<long long>(prow_base + tok) * p.Hq + hq;
            off = prow * D;
            p.plan.part_lse[prow] = lsum > 0.f ? M + __log2f(lsum) : NEG_INF;
          }
        }
        s_off[j] = off;
        s_scl[j] = scl;
      }
      float ov[TN];
      {
        uint32_t a[TN2];
        if (have_o) {
          tc_ld<TN2>(tl + kColO, a);
        } else {
#pragma unroll
          for (int j = 0; j < TN2; ++j) a[j] = 0u;
        }
#pragma unroll
        for (int j = 0; j < TN; ++j) ov[j] = __uint_as_float(a[j]) + __uint_as_float(a[TN + j]);
      }
      named_barrier_sync(2, 128);
      const int d = kk;  // this thread's head dim
      if (prow_base < 0) {
        uint16_t* o16 = static_cast<uint16_t*>(p.out) + d;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
          const long long off = s_off[j];
          const float x = ov[j] * s_scl[j];
          if (off >= 0)
            o16[off] = static_cast<uint16_t>((p.out_f16 ? pack2<false>(x, 0.f) : pack2<true>(x, 0.f)) & 0xffffu);
        }
      } else {
        float* po = p.plan.part_o + d;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
          const long long off = s_off[j];
          if (off >= 0) po[off] = ov[j] * s_scl[j];
        }
      }
    }
    it += nst;
    // Fused merge: the consumers of the CTA that finished a request's last
    // piece (of a group) combine the pieces' partials.
    if (p.fused && prow_base >= 0 && pass == npass - 1)
      fused_merge<D>(p, r, h, prow_base, row0, L, ct, cw, Cfg::NCW, lane);
    tc_fence_before();
    __syncthreads();  // pairs with the producer's end-of-pass barrier
    tc_fence_after();
  }
  } else {
  // -------------------------------------------------------------- consumers
  const int cw = warp - Cfg::NPW;
  const int wq = cw % WQ;
  const int wk = (cw / WQ) % Cfg::WK;
  const int wd = cw / (WQ * Cfg::WK);  // head-dim slice: dims [wd * DS, (wd + 1) * DS)
  constexpr int DS = Cfg::DS;
  const int ks0 = wd * (DS / 16);      // first k-step (16 dims) of the slice
  const int g = lane >> 2;  // MMA groupID
  const int t = lane & 3;   // MMA thread-in-group
  const float sl2 = p.scale_log2;
  const float NEG_INF = -__int_as_float(0x7f800000);
  constexpr float kRescale = 8.f;  // lazy-rescale threshold, log2 units
  const int ct = threadIdx.x - 32 * Cfg::NPW;  // consumer thread index

  // Per-thread swizzled offsets inside a 16-key tile (16-bit caches).
  const int lrowK = (lane & 7) + ((lane >> 3) & 1) * 8;  // ldmatrix row, K (A operand)
  const int lchkK = (lane >> 4) & 1;
  const int lrowV = (lane & 7) + ((lane >> 4) & 1) * 8;  // ldmatrix.trans row, V^T (A operand)
  const int lchkV = (lane >> 3) & 1;
  // Grouped K: a stage holds one box per 16-key tile, [D/16 groups][16 keys][16
  // dims] (16 * ROW bytes, 1024-byte aligned), 128-byte swizzled as a run of
  // 128-byte rows: linear offset o = group * 16 * GRP + key * GRP + byte lands
  // at o ^ (((o >> 7) & 7) << 4).  16-bit: group j's ldmatrix row of this lane
  // sits at j * 512 + kswz[j & 1]; fp8: key g + 8h of group j at j * 256 + h * 128
  // + ((g ^ ((2j + h) & 7)) * 16) + 4t.
  uint32_t kswz[2] = {0u, 0u};
  if constexpr (Cfg::kGroupedK && !Cfg::kFp8) {
    const uint32_t lin = static_cast<uint32_t>(lrowK * 32 + lchkK * 16);  // < 512
    kswz[0] = lin ^ (((lin >> 7) & 3u) << 4);
    kswz[1] = lin ^ ((((lin >> 7) & 3u) | 4u) << 4);
  }

  for (int pass = 0; pass < npass; ++pass) {
    const int pass_base = row_lo + pass * NQ;
    const int ke = pass_key_end(pass);
    const int nst = ke > kb ? (ke - kb + Cfg::KS - 1) / Cfg::KS : 0;

    // Key limits of this thread's two accumulator columns (query rows): keys
    // [llo, lim) are visible (llo > 0 only under a sliding window).
    int lim[2], llo[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int n = pass_base + 8 * wq + 2 * t + e;
      const int K = S - (L - 1 - n / G);  // causal range [0, K) of this row's token
      lim[e] = (n < row_hi) ? min(ke_task, K) : kb;
      llo[e] = p.window > 0 ? max(0, K - p.window) : 0;
    }
    const int vis_lo = max(llo[0], llo[1]);  // keys [vis_lo, vis_hi) are visible to both rows
    const int vis_hi = min(lim[0], lim[1]);

    // Q^T as the B operand of QK^T: row n = groupID of this warp's 8 rows;
    // k-step ks of the slice is global k-step ks0 + ks.
    uint32_t qf[DS / 16][2];
    {
      const int n = pass_base + 8 * wq + g;
      const int tok = n / G;
      const bool ok = n < row_hi && row0 + tok < p.num_tokens;
      const size_t qoff = ok ? (static_cast<size_t>(row0 + tok) * p.Hq + h * G + n % G) * D : 0;
      if constexpr (!Cfg::kFp8) {
        const uint16_t* qp = static_cast<const uint16_t*>(p.q) + qoff;
#pragma unroll
        for (int ks = 0; ks < DS / 16; ++ks) {
          const int kg = ks0 + ks;
          qf[ks][0] = ok ? *reinterpret_cast<const uint32_t*>(qp + 16 * kg + 2 * t) : 0u;
          qf[ks][1] = ok ? *reinterpret_cast<const uint32_t*>(qp + 16 * kg + 2 * t + 8) : 0u;
        }
      } else {
        // fp16 operands; head-dim order permuted to match the fp8 K fragment:
        // k-step ks uses d = cb*SWB + t*(SWB/4) + 4j + {0,1 | 2,3} (row-major
        // K), or d = 16ks + 4t + {0,1 | 2,3} (grouped K).
        constexpr int KPB = Cfg::SWB / 16;  // k-steps per column block
#pragma unroll
        for (int ks = 0; ks < DS / 16; ++ks) {
          const int kg = ks0 + ks;
          const int d = Cfg::kGroupedK ? 16 * kg + 4 * t
                                       : (kg / KPB) * Cfg::SWB + t * (Cfg::SWB / 4) + 4 * (kg % KPB);
          float v0 = 0.f, v1 = 0.f, v2 = 0.f, v3 = 0.f;
          if (ok) {
            const uint2 raw4 = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.q) + qoff + d);
            if (p.out_f16) {
              const __half2 a = *reinterpret_cast<const __half2*>(&raw4.x);
              const __half2 b = *reinterpret_cast<const __half2*>(&raw4.y);
              v0 = __low2float(a); v1 = __high2float(a); v2 = __low2float(b); v3 = __high2float(b);
            } else {
              const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&raw4.x);
              const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&raw4.y);
              v0 = __low2float(a); v1 = __high2float(a); v2 = __low2float(b); v3 = __high2float(b);
            }
          }
          qf[ks][0] = pack2<false>(v0, v1);
          qf[ks][1] = pack2<false>(v2, v3);
        }
      }
    }

    float m[2] = {NEG_INF, NEG_INF};  // reference (lazily updated running max)
    float l[2] = {0.f, 0.f};          // this thread's share of the row sums
    float acc[DS / 16][4];
#pragma unroll
    for (int dt = 0; dt < DS / 16; ++dt) acc[dt][0] = acc[dt][1] = acc[dt][2] = acc[dt][3] = 0.f;

    const bool warp_active = pass_base + 8 * wq < row_hi;

    for (int s = 0; s < nst; ++s) {
      const int sit = it + s;
      const int buf = sit % Cfg::NS;
      const int key0 = kb + s * Cfg::KS;
      const int rbase = wk * T * 16;  // row of this warp's first key in the stage
      // Whether this warp computes on the stage; the same for every slice warp
      // of a row group, which therefore all meet at the logit exchange.
      const bool busy = warp_active && key0 + rbase < ke;
      if (aborted() || !wait_all(bar_full + 8 * buf, (sit / Cfg::NS) & 1)) {
        // A gave-up wait aborts the pipeline; slice warps still take part in
        // the exchange barrier so that none of their row group waits on them.
        if constexpr (Cfg::ND > 1)
          if (busy) named_barrier_sync(2 + wq, Cfg::ND * 32);
        continue;
      }
      const uint32_t kt = base + buf * Cfg::STAGE_BYTES;
      const uint32_t vt = kt + Cfg::TILE_BYTES;

      if (busy) {

        // ---- S^T[16 keys x 8 rows] = K Q^T for T tiles
        float c[T][4];
#pragma unroll
        for (int tt = 0; tt < T; ++tt) c[tt][0] = c[tt][1] = c[tt][2] = c[tt][3] = 0.f;
        if constexpr (!Cfg::kFp8) {
          float c2[4] = {0.f, 0.f, 0.f, 0.f};  // second chain when T == 1
#pragma unroll
          for (int ks = 0; ks < DS / 16; ++ks) {
            const int kg = ks0 + ks;  // (kg & 3) == (ks & 3): DS / 16 is a multiple of 4
            const uint32_t ko = kt + (kg / 4) * Cfg::BLOCK_BYTES + swz<Cfg::SWB>(lrowK, (ks % 4) * 2 + lchkK);
#pragma unroll
            for (int tt = 0; tt < T; ++tt) {
              uint32_t a0, a1, a2, a3;
              if constexpr (Cfg::kGroupedK)
                ldsm_x4(kt + (rbase + 16 * tt) * Cfg::ROW + kg * 512 + kswz[ks & 1], a0, a1, a2, a3);
              else
                ldsm_x4(ko + (rbase + 16 * tt) * Cfg::SWB, a0, a1, a2, a3);
              if (T == 1 && (ks & 1))
                mma16816<Cfg::kBf16Mma>(c2, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
              else
                mma16816<Cfg::kBf16Mma>(c[tt], a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
            }
          }
          if (T == 1) {
            c[0][0] += c2[0]; c[0][1] += c2[1]; c[0][2] += c2[2]; c[0][3] += c2[3];
          }
        } else if constexpr (Cfg::kGroupedK) {
          // grouped fp8 K: a 16-dim group of a key is 16 bytes; thread t takes
          // dims 4t..4t+3 of keys g and g + 8 (two conflict-free 32-bit loads
          // per k-step), matched by the Q fragment's head-dim order
#pragma unroll
          for (int tt = 0; tt < T; ++tt) {
            const uint32_t kg = kt + (rbase + 16 * tt) * Cfg::ROW + 4 * t;
#pragma unroll
            for (int ks = 0; ks < DS / 16; ++ks) {
              // ((2 * (ks0 + ks)) & 7) == ((2 * ks) & 7): DS / 16 is a multiple of 4
              const uint32_t w0 = lds32(kg + (ks0 + ks) * 256 + ((g ^ ((2 * ks) & 7)) << 4));
              const uint32_t w1 = lds32(kg + (ks0 + ks) * 256 + 128 + ((g ^ ((2 * ks + 1) & 7)) << 4));
              uint32_t a0, a1, a2, a3;
              e4m3x4_to_f16x2x2(w0, a0, a2);
              e4m3x4_to_f16x2x2(w1, a1, a3);
              mma16816<false>(c[tt], a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
            }
          }
        } else {
          constexpr int KPB = Cfg::SWB / 16;
          constexpr int CPT = Cfg::SWB / 64;  // 16-byte chunks per thread per row
#pragma unroll
          for (int tt = 0; tt < T; ++tt) {
            const int rt = rbase + 16 * tt;
#pragma unroll
            for (int cb = 0; cb < Cfg::CBS; ++cb) {  // the slice's column blocks
              uint32_t wg[4 * CPT], wg8[4 * CPT];
#pragma unroll
              for (int k = 0; k < CPT; ++k) {
                const uint32_t o = kt + (wd * Cfg::CBS + cb) * Cfg::BLOCK_BYTES + rt * Cfg::SWB +
                                   swz<Cfg::SWB>(g, t * CPT + k);
                const uint4 x = lds128(o);
                const uint4 y = lds128(o + 8 * Cfg::SWB);
                wg[4 * k] = x.x; wg[4 * k + 1] = x.y; wg[4 * k + 2] = x.z; wg[4 * k + 3] = x.w;
                wg8[4 * k] = y.x; wg8[4 * k + 1] = y.y; wg8[4 * k + 2] = y.z; wg8[4 * k + 3] = y.w;
              }
#pragma unroll
              for (int j = 0; j < KPB; ++j) {
                uint32_t a0, a1, a2, a3;
                e4m3x4_to_f16x2x2(wg[j], a0, a2);
                e4m3x4_to_f16x2x2(wg8[j], a1, a3);
                mma16816<false>(c[tt], a0, a1, a2, a3, qf[cb * KPB + j][0], qf[cb * KPB + j][1]);
              }
            }
          }
        }

        // ---- sliced head dims: sum the slices' partial logits (same order in
        // every warp of the row group)
        if constexpr (Cfg::ND > 1) {
          float4* xs = sx + ((s & 1) * WQ + wq) * Cfg::ND * 32;
          xs[wd * 32 + lane] = make_float4(c[0][0], c[0][1], c[0][2], c[0][3]);
          named_barrier_sync(2 + wq, Cfg::ND * 32);
          float4 a = xs[lane];
#pragma unroll
          for (int k = 1; k < Cfg::ND; ++k) {
            const float4 b = xs[k * 32 + lane];
            a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
          }
          c[0][0] = a.x; c[0][1] = a.y; c[0][2] = a.z; c[0][3] = a.w;
        }

        // ---- online softmax (log2 domain), lazily rescaled
        float sv[T][4];
        float mx0 = NEG_INF, mx1 = NEG_INF;
        // Both of this thread's rows see every key of the warp's T tiles on
        // all but the boundary stages (range end, window start): no masks.
        const int kw0 = key0 + rbase;
        if (kw0 >= vis_lo && kw0 + 16 * T <= vis_hi) {
#pragma unroll
          for (int tt = 0; tt < T; ++tt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) sv[tt][e] = c[tt][e] * sl2;
            mx0 = fmaxf(mx0, fmaxf(sv[tt][0], sv[tt][2]));
            mx1 = fmaxf(mx1, fmaxf(sv[tt][1], sv[tt][3]));
          }
        } else {
#pragma unroll
          for (int tt = 0; tt < T; ++tt) {
            const int k_lo = kw0 + 16 * tt + g;
            sv[tt][0] = (k_lo < lim[0] && k_lo >= llo[0]) ? c[tt][0] * sl2 : NEG_INF;
            sv[tt][1] = (k_lo < lim[1] && k_lo >= llo[1]) ? c[tt][1] * sl2 : NEG_INF;
            sv[tt][2] = (k_lo + 8 < lim[0] && k_lo + 8 >= llo[0]) ? c[tt][2] * sl2 : NEG_INF;
            sv[tt][3] = (k_lo + 8 < lim[1] && k_lo + 8 >= llo[1]) ? c[tt][3] * sl2 : NEG_INF;
            mx0 = fmaxf(mx0, fmaxf(sv[tt][0], sv[tt][2]));
            mx1 = fmaxf(mx1, fmaxf(sv[tt][1], sv[tt][3]));
          }
        }
#pragma unroll
        for (int o = 4; o <= 16; o <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
        }
        const bool up0 = mx0 > m[0] + kRescale;
        const bool up1 = mx1 > m[1] + kRescale;
        if (__any_sync(0xffffffffu, up0 || up1)) {
          const float al0 = up0 ? fast_exp2(m[0] - mx0) : 1.f;  // 0 when m was -inf
          const float al1 = up1 ? fast_exp2(m[1] - mx1) : 1.f;
          if (up0) m[0] = mx0;
          if (up1) m[1] = mx1;
          l[0] *= al0;
          l[1] *= al1;
#pragma unroll
          for (int dt = 0; dt < DS / 16; ++dt) {
            acc[dt][0] *= al0;
            acc[dt][1] *= al1;
            acc[dt][2] *= al0;
            acc[dt][3] *= al1;
          }
        }
        const float ref0 = (m[0] == NEG_INF) ? 0.f : m[0];
        const float ref1 = (m[1] == NEG_INF) ? 0.f : m[1];
        uint32_t pb[T][2];
#pragma unroll
        for (int tt = 0; tt < T; ++tt) {
          const float p0 = fast_exp2(sv[tt][0] - ref0);
          const float p1 = fast_exp2(sv[tt][1] - ref1);
          const float p2 = fast_exp2(sv[tt][2] - ref0);
          const float p3 = fast_exp2(sv[tt][3] - ref1);
          l[0] += p0 + p2;
          l[1] += p1 + p3;
          // P^T (keys x rows) -> B fragment of PV: transpose the two 8x8 halves.
          pb[tt][0] = movmatrix_trans(pack2<Cfg::kBf16Mma>(p0, p1));
          pb[tt][1] = movmatrix_trans(pack2<Cfg::kBf16Mma>(p2, p3));
        }

        // ---- O^T[D x 8] += V^T P^T.  Keys past `ke` may hold stale or
        // uninitialised shared memory: zero them so 0 * NaN cannot occur.
        if constexpr (!Cfg::kFp8) {
#pragma unroll
          for (int dt = 0; dt < DS / 16; ++dt) {
            const int dg = ks0 + dt;  // global 16-dim tile; (dg & 3) == (dt & 3)
            const uint32_t vo = vt + (dg / 4) * Cfg::BLOCK_BYTES + swz<Cfg::SWB>(lrowV, (dt % 4) * 2 + lchkV);
#pragma unroll
            for (int tt = 0; tt < T; ++tt) {
              const int kbt = key0 + rbase + 16 * tt;
              uint32_t a0, a1, a2, a3;
              ldsm_x4_trans(vo + (rbase + 16 * tt) * Cfg::SWB, a0, a1, a2, a3);
              if (kbt + 16 > ke) {
                const int kq = kbt + 2 * t;
                const uint32_t m01 = (kq < ke ? 0x0000ffffu : 0u) | (kq + 1 < ke ? 0xffff0000u : 0u);
                const uint32_t m89 = (kq + 8 < ke ? 0x0000ffffu : 0u) | (kq + 9 < ke ? 0xffff0000u : 0u);
                a0 &= m01; a1 &= m01; a2 &= m89; a3 &= m89;
              }
              mma16816<Cfg::kBf16Mma>(acc[dt], a0, a1, a2, a3, pb[tt][0], pb[tt][1]);
            }
          }
        } else {
          // d = 32u + 4g + e:  e = 0 / 1 -> tile 2u rows g / g+8,
          //                    e = 2 / 3 -> tile 2u+1 rows g / g+8.
#pragma unroll
          for (int tt = 0; tt < T; ++tt) {
            const int kbt = key0 + rbase + 16 * tt;
            const int ra = rbase + 16 * tt + 2 * t;
            const bool tail = kbt + 16 > ke;
            const int kq = kbt + 2 * t;
            const uint32_t z0 = (kq < ke) ? 0xffffffffu : 0u, z1 = (kq + 1 < ke) ? 0xffffffffu : 0u;
            const uint32_t z8 = (kq + 8 < ke) ? 0xffffffffu : 0u, z9 = (kq + 9 < ke) ? 0xffffffffu : 0u;
#pragma unroll
            for (int u = 0; u < DS / 32; ++u) {
              const int byte = 32 * (wd * (DS / 32) + u) + 4 * g;
              const int cb = byte / Cfg::SWB;
              const int inb = byte % Cfg::SWB;
              const uint32_t blk = vt + cb * Cfg::BLOCK_BYTES;
              const uint32_t wsub = static_cast<uint32_t>(inb & 15);
              uint32_t w0 = lds32(blk + swz<Cfg::SWB>(ra, inb >> 4) + wsub);
              uint32_t w1 = lds32(blk + swz<Cfg::SWB>(ra + 1, inb >> 4) + wsub);
              uint32_t w8 = lds32(blk + swz<Cfg::SWB>(ra + 8, inb >> 4) + wsub);
              uint32_t w9 = lds32(blk + swz<Cfg::SWB>(ra + 9, inb >> 4) + wsub);
              if (tail) {
                w0 &= z0; w1 &= z1; w8 &= z8; w9 &= z9;
              }
              uint32_t x0, x1, y0, y1, u0, u1, v0, v1;
              e4m3x4_to_f16x2x2(prmt(w0, w1, 0x5140u), x0, x1);  // d+0, d+1; keys 2t,2t+1
              e4m3x4_to_f16x2x2(prmt(w0, w1, 0x7362u), y0, y1);  // d+2, d+3
              e4m3x4_to_f16x2x2(prmt(w8, w9, 0x5140u), u0, u1);  // keys 2t+8, 2t+9
              e4m3x4_to_f16x2x2(prmt(w8, w9, 0x7362u), v0, v1);
              mma16816<false>(acc[2 * u], x0, x1, u0, u1, pb[tt][0], pb[tt][1]);
              mma16816<false>(acc[2 * u + 1], y0, y1, v0, v1, pb[tt][0], pb[tt][1]);
            }
          }
        }
      }
      __syncwarp();
      // The slot of a pass's last stage is released after the exchange that
      // reuses it (below) when the producer issues ahead.
      if (lane == 0 && !(Cfg::kHoldSlot && s == nst - 1)) mbar_arrive(bar_empty + 8 * buf);
    }
    // ring slot of the epilogue exchange: the last stage's (the producer may
    // already be filling the others with the next pass), or any when the pass
    // had no stage (nothing is then in flight)
    const int xbuf = (nst > 0 ? it + nst - 1 : it) % Cfg::NS;
    it += nst;

    // ------------------------------------------------------------ epilogue
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
      l[0] += __shfl_xor_sync(0xffffffffu, l[0], o);
      l[1] += __shfl_xor_sync(0xffffffffu, l[1], o);
    }
    if constexpr (Cfg::kDirectEpi) {
      // One key warp per row group: its m, l and accumulators are the pass's
      // final ones (the slice warps of a row group hold the same m and l), so
      // each thread scales its own elements and stores them -- rows 2t and
      // 2t+1 of its group, the head dims its accumulator tiles cover.
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int n = pass_base + 8 * wq + 2 * t + e;
        if (!warp_active || n >= row_hi) continue;
        const int tok = n / G;
        const int hq = h * G + n % G;
        const float M = m[e];
        float lsum = M != NEG_INF ? l[e] : 0.f;
        // A single piece writes the output row: its head's sink joins here.
        const bool sink = prow_base < 0 && p.sinks != nullptr;
        const float f = sink ? add_sink(M, __ldg(p.sinks + hq) * 1.4426950408889634f, lsum) : 1.f;
        const float inv = lsum > 0.f ? p.v_scale / lsum : 0.f;
        auto fin = [&](float v) {
          if (M == NEG_INF) v = 0.f;
          if (sink) v *= f;
          return v * inv;
        };
        if (prow_base < 0) {
          const int trow = row0 + tok;
          if (trow >= p.num_tokens) {
            atomicOr(p.plan.err, PA_DEVERR_PLAN_OVERFLOW);
            continue;
          }
          uint16_t* orow = static_cast<uint16_t*>(p.out) + (static_cast<size_t>(trow) * p.Hq + hq) * D;
#pragma unroll
          for (int dt = 0; dt < DS / 16; ++dt) {
            if constexpr (!Cfg::kFp8) {
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const float v = fin(acc[dt][2 * hh + e]);
                const uint32_t pk = p.out_f16 ? pack2<false>(v, 0.f) : pack2<true>(v, 0.f);
                orow[wd * DS + 16 * dt + g + 8 * hh] = static_cast<uint16_t>(pk & 0xffffu);
              }
            } else {  // dims d, d + 1 of the pair hh = 0, 1
              const int d = wd * DS + 32 * (dt / 2) + 4 * g + 2 * (dt % 2);
              const float v0 = fin(acc[dt][e]), v1 = fin(acc[dt][2 + e]);
              *reinterpret_cast<uint32_t*>(orow + d) = p.out_f16 ? pack2<false>(v0, v1) : pack2<true>(v0, v1);
            }
          }
        } else {
          const size_t prow = static_cast<size_t>(prow_base + tok) * p.Hq + hq;
          float* po = p.plan.part_o + prow * D;
#pragma unroll
          for (int dt = 0; dt < DS / 16; ++dt) {
            if constexpr (!Cfg::kFp8) {
              po[wd * DS + 16 * dt + g] = fin(acc[dt][e]);
              po[wd * DS + 16 * dt + g + 8] = fin(acc[dt][2 + e]);
            } else {
              const int d = wd * DS + 32 * (dt / 2) + 4 * g + 2 * (dt % 2);
              *reinterpret_cast<float2*>(po + d) = make_float2(fin(acc[dt][e]), fin(acc[dt][2 + e]));
            }
          }
          if (g == 0 && wd == 0) p.plan.part_lse[prow] = lsum > 0.f ? M + __log2f(lsum) : NEG_INF;
        }
      }
    } else {
    named_barrier_sync(1, Cfg::NCW * 32);  // all stage reads of this pass done

    // exchange area: O [WQ][WK][8][DP], then m and l [WQ][WK][8]
    float* ex_o = Cfg::kHoldSlot ? ex + xbuf * (Cfg::STAGE_BYTES / 4) : ex;
    float* ex_m = ex_o + WQ * Cfg::WK * 8 * Cfg::DP;
    float* ex_l = ex_m + WQ * Cfg::WK * 8;
    const int wslot = (wq * Cfg::WK + wk) * 8;
#pragma unroll
    for (int dt = 0; dt < DS / 16; ++dt) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        int d = wd * DS;  // the slice's dims
        if constexpr (!Cfg::kFp8)
          d += 16 * dt + g + 8 * hh;
        else
          d += 32 * (dt / 2) + 4 * g + 2 * (dt % 2) + hh;
        ex_o[(wslot + 2 * t) * Cfg::DP + d] = acc[dt][2 * hh];
        ex_o[(wslot + 2 * t + 1) * Cfg::DP + d] = acc[dt][2 * hh + 1];
      }
    }
    if (g == 0 && wd == 0) {  // every slice warp holds the same m and l
      ex_m[wslot + 2 * t] = m[0];
      ex_m[wslot + 2 * t + 1] = m[1];
      ex_l[wslot + 2 * t] = l[0];
      ex_l[wslot + 2 * t + 1] = l[1];
    }
    named_barrier_sync(1, Cfg::NCW * 32);

    constexpr int D4 = D / 4;
    for (int u = ct; u < WQ * 8 * D4; u += Cfg::NCW * 32) {
      const int gq = u / (8 * D4);
      const int col = (u / D4) % 8;
      const int d4 = (u % D4) * 4;
      const int n = pass_base + 8 * gq + col;
      if (n >= row_hi) continue;
      float M = NEG_INF;
#pragma unroll
      for (int k = 0; k < Cfg::WK; ++k) M = fmaxf(M, ex_m[(gq * Cfg::WK + k) * 8 + col]);
      float lsum = 0.f, o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
      if (M != NEG_INF) {
#pragma unroll
        for (int k = 0; k < Cfg::WK; ++k) {
          const int ws = (gq * Cfg::WK + k) * 8 + col;
          const float w = fast_exp2(ex_m[ws] - M);
          const float4 v = *reinterpret_cast<const float4*>(ex_o + ws * Cfg::DP + d4);
          lsum += w * ex_l[ws];
          o0 += w * v.x; o1 += w * v.y; o2 += w * v.z; o3 += w * v.w;
        }
      }
      const int tok = n / G;
      const int hq = h * G + n % G;
      // A single piece writes the output row: its head's sink joins here (a
      // request with several pieces gets it in the merge).
      if (prow_base < 0 && p.sinks) {
        const float f = add_sink(M, __ldg(p.sinks + hq) * 1.4426950408889634f, lsum);
        o0 *= f; o1 *= f; o2 *= f; o3 *= f;
      }
      const float inv = lsum > 0.f ? p.v_scale / lsum : 0.f;
      o0 *= inv; o1 *= inv; o2 *= inv; o3 *= inv;
      if (prow_base < 0) {
        const int trow = row0 + tok;
        if (trow >= p.num_tokens) {
          atomicOr(p.plan.err, PA_DEVERR_PLAN_OVERFLOW);
          continue;
        }
        uint2 pk;
        if (p.out_f16) {
          pk.x = pack2<false>(o0, o1);
          pk.y = pack2<false>(o2, o3);
        } else {
          pk.x = pack2<true>(o0, o1);
          pk.y = pack2<true>(o2, o3);
        }
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) +
                                  (static_cast<size_t>(trow) * p.Hq + hq) * D + d4) = pk;
      } else {
        const size_t prow = static_cast<size_t>(prow_base + tok) * p.Hq + hq;
        *reinterpret_cast<float4*>(p.plan.part_o + prow * D + d4) = make_float4(o0, o1, o2, o3);
        if (d4 == 0) p.plan.part_lse[prow] = lsum > 0.f ? M + __log2f(lsum) : NEG_INF;
      }
    }
    fence_proxy_async_smem();  // exchange writes precede the next pass's TMA writes
    if constexpr (Cfg::kHoldSlot) {
      __syncwarp();
      if (nst > 0 && lane == 0) mbar_arrive(bar_empty + 8 * xbuf);  // this warp is done with it
    }
    }  // exchange epilogue
    // Fused merge: the consumers of the CTA that finished a request's last
    // piece (of a group) combine the pieces' partials while the producer
    // issues the next item's first stages.
    if constexpr (D <= 256) {  // wide heads keep the merge kernel (registers)
      if (p.fused && prow_base >= 0 && pass == npass - 1)
        fused_merge<D>(p, r, h, prow_base, row0, L, ct, cw, Cfg::NCW, lane);
    }
    __syncthreads();  // pairs with the producer's end-of-pass barrier
  }
  }  // consumers
  }  // work items

  // Drain: wait (bounded) until the last copy issued into every ring slot has
  // landed, so that none can still be writing shared memory when the CTA
  // exits -- whether or not the pipeline was aborted.
  // Each producer warp drains the stages it issued.
  if (warp < Cfg::NPW && lane == 0) {
    for (int k = (issued > Cfg::NS ? issued - Cfg::NS : 0); k < issued; ++k)
      mbar_wait(bar_full + 8 * (k % Cfg::NS), (k / Cfg::NS) & 1, p.plan.err, p.wait_ns);
  }
  if constexpr (Cfg::kTc) {
    // Every MMA the issuing thread started has completed (a last commit, on a
    // barrier of its own, and a bounded wait) before the tensor memory is
    // released.
    if (warp == Cfg::NPW) {
      const uint32_t bar_drain = bar_full + 16 * Cfg::NS + 48;
      if (lane == 0) {
        tc_commit(bar_drain);
        mbar_wait(bar_drain, 0, p.plan.err, p.wait_ns);
      }
      __syncwarp();
      tc_fence_after();
      tc_dealloc(*reinterpret_cast<volatile uint32_t*>(smem_raw + (base - raw) + Cfg::DATA_BYTES +
                                                       Cfg::TC_TMEM_SLOT),
                 Cfg::TC_COLS);
    }
  }
  // With the merge fused there is no merge kernel to reset the work counter
  // after this grid: the last CTA to finish does (thread 0 made every claim).
  if constexpr (D <= 256)
    if (p.fused && threadIdx.x == 0) cta_finished(p);
}

template <int D, int KVT, int WQ, int KL>
cudaError_t launch_split_cfg(const SplitParams& p, const CUtensorMap& tk,
                             const CUtensorMap& tv, cudaStream_t s) {
  using Cfg = SplitCfg<D, KVT, WQ, KL>;
  auto kern = split_kernel<D, KVT, WQ, KL>;
  // per device: the shared-memory attribute, then CTAs per SM as the
  // occupancy calculator sees the kernel
  static std::atomic<int> state[kMaxDevices];
  int per_sm = 0;
  const cudaError_t e = per_device_once(state, per_sm, [&](int& b) {
    cudaError_t r =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (r == cudaSuccess)
      r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, Cfg::THREADS, Cfg::SMEM_BYTES);
    return r;
  });
  if (e != cudaSuccess) return e;
  SplitParams q = p;
  q.resident = per_sm > 0 && p.sms > 0 ? per_sm * p.sms : 0;
  const unsigned zero_ctas = static_cast<unsigned>((p.num_tokens + kZeroRows - 1) / kZeroRows);
  return launch_pdl(kern, dim3(static_cast<unsigned>(p.C) * p.Hkv + zero_ctas), dim3(Cfg::THREADS),
                    Cfg::SMEM_BYTES, s, tk, tv, q);
}

template <int D, int KL>
cudaError_t launch_split_d(const SplitParams& p, int kv_dtype, int wq,
                           const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s) {
  constexpr int kMaxWq = split_max_row_groups(D);
#define PA_SPLIT_CASE(KVT)                                                               \
  switch (wq) {                                                                          \
    case 1: return launch_split_cfg<D, KVT, 1, KL>(p, tk, tv, s);                     \
    case 2:                                                                              \
      if constexpr (kMaxWq >= 2) return launch_split_cfg<D, KVT, 2, KL>(p, tk, tv, s); \
      return cudaErrorInvalidValue;                                                      \
    case 3:                                                                              \
      if constexpr (kMaxWq >= 3) return launch_split_cfg<D, KVT, 3, KL>(p, tk, tv, s); \
      return cudaErrorInvalidValue;                                                      \
    default:                                                                             \
      if constexpr (kMaxWq >= 4) return launch_split_cfg<D, KVT, 4, KL>(p, tk, tv, s); \
      return cudaErrorInvalidValue;                                                      \
  }
  switch (kv_dtype) {
    case PA_BF16: PA_SPLIT_CASE(PA_BF16)
    case PA_FP16: PA_SPLIT_CASE(PA_FP16)
    default: PA_SPLIT_CASE(PA_FP8_E4M3)
  }
#undef PA_SPLIT_CASE
}

}  // namespace pa
