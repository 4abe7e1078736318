// pa_internal.h -- shared between the C-ABI layer and the kernel translation
// units: the plan's device buffers, kernel parameter blocks, launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace pa {

constexpr int kTile = 256;       // partition tile, tokens
constexpr int kMaxSeqs = 4096;   // planner domain
constexpr int kStageTensorBytes = 16384;  // split kernel: K (or V) bytes per pipeline stage

// Bounded waits inside the kernels give up after this long by default (a plan
// may set another limit) and raise PA_DEVERR_TIMEOUT.
constexpr unsigned long long kWaitLimitNs = 4000000000ull;

constexpr int kMinPieceTiles = 2;  // a slot is cut into pieces of at least this many tiles
constexpr int kWarpMergePieces = 8;  // rows with at most this many pieces are merged by one warp

// Launch set-up that every device needs once: a kernel's function attributes
// (cudaFuncSetAttribute) and its occupancy belong to the device, so launchers
// keep one entry per device ordinal -- 0 until set up, else the value + 1 --
// for the current device.  Concurrent first calls both set up: idempotent.
constexpr int kMaxDevices = 64;
template <typename SetUp>
inline cudaError_t per_device_once(std::atomic<int>* state, int& value, SetUp&& set_up) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int v = state[dev].load(std::memory_order_acquire);
  if (v == 0) {
    int x = 0;
    e = set_up(x);
    if (e != cudaSuccess) return e;
    v = x + 1;
    state[dev].store(v, std::memory_order_release);
  }
  value = v - 1;
  return cudaSuccess;
}

// Device buffers owned by one plan.
//
// The plan's tasks (work_info: one per slot) are what the pages define.  The
// split kernel runs *pieces*: a slot's tile range cut into q >= 1 consecutive
// sub-ranges, q chosen by the planner so that, when the whole grid is one wave,
// no CTA is left with a task much longer than the others (every piece writes
// its own partial; the merge combines them with the request's other partials).
struct PlanDev {
  int4* work;       // [C] (seq, tile_begin, tile_end, seq_ctx); seq = -1 unused
  int2* reduce;     // [n] (first_slot, num_parts)
  int2* snap;       // [n] (context_len, query_len) seen by the last refresh
  unsigned* err;    // sticky PA_DEVERR_* word
  float* part_o;    // [rows_cap][Hq][D] normalised partial outputs
  float* part_lse;  // [rows_cap][Hq] log2-sum-exp of each partial (log2 units)
  int4* pieces;     // [C * Q] in launch order (longest first): {r, first key, end key,
                    // partial row of the piece's token 0, or -1 when the request has
                    // one piece and its CTA writes the output row}
  int2* extra;      // [max_extra] (piece position, row chunk >= 1) for requests whose
                    // query rows exceed one work item
  int* counters;    // [0] extra items, [1] next late piece or extra item (x Hkv; reset by
                    // the planner, and after each decode by the merge kernel or, with the
                    // merge fused, by the split kernel's last CTA), [2] merge rows with more
                    // than kWarpMergePieces pieces, [3] merge rows with 2..kWarpMergePieces
                    // pieces, [4] pieces, [5] split CTAs finished (fused merge only)
  int4* mrows;      // [max_tokens] one entry per row of a request with several pieces:
                    // {r | (pieces - 1) << 12, token, partial row of piece 0, L}
                    // (piece k's partial row is that + k * L); rows with few pieces
                    // first ([0, counters[3])), then rows with many
  int2* preq;       // [n] (first partial row, pieces) of each request (fused merge)
  int* tickets;     // [levels][rows_cap][Hkv] arrival counts of the fused merge's
                    // groups, zero between decode calls (each is reset by the CTA that
                    // takes its last ticket)
};

// Fused merge (decode-only plans): the pieces of a (request, kv head) are
// merged in a tree of fan-in kFusedFanIn -- the CTA that finishes the last
// piece of a group merges the group's partials into one, in place of its first
// -- with one ticket per group and level; kFusedLevels levels cover
// kFusedFanIn^kFusedLevels >= Q * P pieces.
constexpr int kFusedFanIn = 8;
constexpr int kFusedLog2FanIn = 3;
constexpr int kFusedLevels = 7;  // at most: 8^7 > 4 * 65536

// Sizes and offsets of one plan's buffers (256-byte aligned, back to back).
struct PlanLayout {
  long long C;          // capacity: slots of work_info
  int Q;                // at most Q pieces per slot
  long long rows_cap;   // partial rows
  int rpc;              // query rows per split-kernel work item
  long long max_extra;  // extra (piece, row chunk) items
  int fused;            // 1: the split kernel merges the partials (decode-only plans whose
                        // query rows fit one work item); 0: the merge kernel does
  int levels;           // fused merge: tree levels needed for Q * P pieces
  size_t b_work, b_red, b_snap, b_err, b_po, b_pl, b_pieces, b_ext, b_mrow, b_preq, b_tick, total;
};
// `pieces` = false keeps every task whole (Q = 1); `fused` = false keeps the
// separate merge kernel for every plan.
PlanLayout plan_layout(int num_seqs, int Hq, int Hkv, int D, int max_qlen, int max_tokens,
                       int max_partitions, int budget, int sms, bool pieces, bool fused);
// Points the buffers of `l` into [base, base + l.total); the error word and
// the counters share one 256-byte block.
PlanDev carve_plan(char* base, const PlanLayout& l);

struct PlanParams {
  const int* context_lens;
  const int* cu;  // nullable
  int n, Hkv, P, C, kind, max_qlen, max_tokens;
  int Q;          // at most Q pieces per slot
  int window;     // sliding window (0: none): a request's plan starts at its first visible tile
  int G;          // q heads per kv head
  int rpc;        // query rows per split-kernel work item (row chunk)
  int wave;       // CTAs of the decode grid that run at once (0: unknown); a plan of
                  // more (C * Hkv > wave) has its slots cut into pieces
  long long rows_cap;
  long long max_extra;
  PlanDev dev;
};

struct SplitParams {
  PlanDev plan;
  const void* q;
  void* out;
  const int* block_tables;
  const int* context_lens;
  const int* cu;  // nullable
  int num_tokens, num_blocks, Hq, Hkv, G, bs, max_blocks, n;
  int C;            // plan capacity: CTAs [C*Hkv, grid) write zero rows
  int sms;          // multiprocessors of the device
  int resident;     // set by the launcher: CTAs of this grid that run at once (0: all).
                    // CTA b starts on item b (piece b / Hkv, kv head b % Hkv) for b < C*Hkv,
                    // or, when the plan holds more pieces than C, for b < min(resident,
                    // C*Hkv); every later item is taken from the work counter by
                    // whichever CTA is free
  int total_rows;   // num_blocks * Hkv * bs: first out-of-range row of the cache view
  int out_f16;      // q/out element type: 1 = fp16, 0 = bf16
  int rpc;          // query rows per work item (row chunk); a multiple of 8 x row groups
  float scale_log2; // softmax scale * k_scale * log2(e)
  float v_scale;    // 1 for 16-bit caches
  int window;       // sliding window: a row that may see keys [0, K) sees [K - window, K); 0: none
  const float* sinks;  // [Hq] sink logits (scale * q.k units) or null
  int fused;        // 1: merge each request's partials in this kernel (no merge kernel)
  long long rows_cap;  // partial rows of the plan (ticket indexing)
  unsigned long long wait_ns;  // limit of every bounded wait (PA_DEVERR_TIMEOUT after it)
  int skip_stage;   // test hook: when >= 0, every CTA's producer leaves ring stage number
                    // skip_stage un-issued (no copy, no arrival), so the waits on it run out
};

// Head dims the kernels take: 64, and 128 to 1024 in steps of 128.
constexpr bool head_dim_supported(int D) { return D == 64 || (D % 128 == 0 && D >= 128 && D <= 1024); }
// Query-row groups of 8 per pass the split kernel is built with for head_dim D:
// head dims above 256 run one warp per 128- or 256-dim slice, so fewer row
// groups fit.
constexpr int split_max_row_groups(int D) { return D <= 256 ? 4 : (D <= 512 ? 2 : 1); }
// Rows of one TMA box of a KV tile for head_dim D, cache dtype, block size.
int split_box_rows(int D, int kv_dtype, int bs);
// Bytes of one box row (the swizzle span): min(128, D * elem_bytes).
int split_box_row_bytes(int D, int kv_dtype);
// TMA descriptor of a K or V cache view for the split kernel (grouped: K in
// [num_blocks, Hkv, D/16, bs, 16]); false if the driver rejects it.  The one
// encoder every launch path uses, so the boxes and swizzle always match the
// kernel's shared-memory layout.
bool encode_cache_tmap(const void* ptr, int num_blocks, int Hkv, int bs, int D, int dtype,
                       bool grouped, CUtensorMap* out);
// Query-row groups of 8 handled per pass for a plan with this max query length.
int split_row_groups(int max_qlen, int G, int D);
// Upper bound on the extra (slot, row chunk) items a plan with these limits can list.
long long split_max_extra(int G, int rpc, long long rows_cap, int max_tokens, int max_qlen);

struct MergeParams {
  PlanDev plan;
  void* out;
  const int* context_lens;
  const int* cu;  // nullable
  int num_tokens, n, Hq, D, out_f16;
  int grid;       // persistent grid size
  const float* sinks;  // [Hq] sink logits (scale * q.k units) or null
};

// A softmax whose numerator and denominator W are relative to 2^M (log2 units)
// gains a sink logit s2 (log2 units) in its denominator: W becomes the new
// denominator relative to 2^max(M, s2), and the numerator must be multiplied
// by the returned factor.  No-op for s2 = -inf.
__device__ __forceinline__ float add_sink(float M, float s2, float& W) {
  const float NEG_INF = -__int_as_float(0x7f800000);
  if (s2 == NEG_INF) return 1.f;
  const float M2 = fmaxf(M, s2);
  float y, f = 0.f;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(s2 - M2));
  if (M != NEG_INF) asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(f) : "f"(M - M2));
  W = W * f + y;
  return f;
}

// Launches `kernel` with programmatic stream serialization: it may be
// scheduled while the previous kernel on the stream is still running (every
// kernel of this library waits for its predecessor before touching data).
template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, int smem, cudaStream_t s,
                       const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t launch_plan(const PlanParams& p, cudaStream_t s);
cudaError_t launch_merge(const MergeParams& p, cudaStream_t s);
// k_layout: PA_K_ROWS or PA_K_GROUPED (the K cache's layout; V is always rows).
cudaError_t launch_split(const SplitParams& p, int D, int kv_dtype, int row_groups, int k_layout,
                         const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s);
// One translation unit per head_dim and K layout (the _gk ones: grouped K); head
// dims above 256 share one per head_dim for both layouts (k_layout argument).
#define PA_DECLARE_SPLIT(NAME)                                                        \
  cudaError_t NAME(const SplitParams& p, int kv_dtype, int row_groups, const CUtensorMap& tk, \
                   const CUtensorMap& tv, cudaStream_t s);
PA_DECLARE_SPLIT(launch_split_d64)
PA_DECLARE_SPLIT(launch_split_d128)
PA_DECLARE_SPLIT(launch_split_d256)
PA_DECLARE_SPLIT(launch_split_d64_gk)
PA_DECLARE_SPLIT(launch_split_d128_gk)
PA_DECLARE_SPLIT(launch_split_d256_gk)
#define PA_DECLARE_SPLIT_WIDE(NAME)                                                   \
  cudaError_t NAME(const SplitParams& p, int kv_dtype, int row_groups, int k_layout,  \
                   const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s);
PA_DECLARE_SPLIT_WIDE(launch_split_d384)
PA_DECLARE_SPLIT_WIDE(launch_split_d512)
PA_DECLARE_SPLIT_WIDE(launch_split_d640)
PA_DECLARE_SPLIT_WIDE(launch_split_d768)
PA_DECLARE_SPLIT_WIDE(launch_split_d896)
PA_DECLARE_SPLIT_WIDE(launch_split_d1024)
#undef PA_DECLARE_SPLIT_WIDE
#undef PA_DECLARE_SPLIT

}  // namespace pa
