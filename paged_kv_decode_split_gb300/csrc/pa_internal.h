// pa_internal.h -- shared between the C-ABI layer and the kernel translation
// units: the plan's device buffers, kernel parameter blocks, launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

constexpr int kTile = 256;       // partition tile, tokens
constexpr int kMaxSeqs = 4096;   // planner domain
constexpr int kStageTensorBytes = 16384;  // split kernel: K (or V) bytes per pipeline stage

// Device buffers owned by one plan.
struct PlanDev {
  int4* work;       // [C] (seq, tile_begin, tile_end, seq_ctx); seq = -1 unused
  int2* reduce;     // [n] (first_slot, num_parts)
  int* part_row;    // [C] first partial row of the slot's request part; -1 if none
  int2* snap;       // [n] (context_len, query_len) seen by the last refresh
  unsigned* err;    // sticky PA_DEVERR_* word
  float* part_o;    // [rows_cap][Hq][D] normalised partial outputs
  float* part_lse;  // [rows_cap][Hq] log2-sum-exp of each partial (log2 units)
  int* order;       // [C] slots by task length, longest first (launch order)
  int2* extra;      // [max_extra] (slot, row chunk >= 1) of requests with many query rows
  int* counters;    // [0] extra items, [1] next extra item (x Hkv), [2] split CTAs done,
                    // [3] rows to merge
  int4* mrows;      // [max_tokens] one entry per row of a multi-partition request:
                    // {r | (parts - 1) << 12, token, partial row of partition 0, L}
                    // (partition j's partial row is that + j * L)
};

struct PlanParams {
  const int* context_lens;
  const int* cu;  // nullable
  int n, Hkv, P, C, kind, max_qlen, max_tokens;
  int G;          // q heads per kv head
  int rpc;        // query rows per split-kernel work item (row chunk)
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
  int C;            // plan capacity: CTAs [0, C*Hkv) run tasks, the rest write zero rows
  int total_rows;   // num_blocks * Hkv * bs: first out-of-range row of the cache view
  int out_f16;      // q/out element type: 1 = fp16, 0 = bf16
  int rpc;          // query rows per work item (row chunk); a multiple of 8 x row groups
  float scale_log2; // softmax scale * k_scale * log2(e)
  float v_scale;    // 1 for 16-bit caches
};

// Rows of one TMA box of a KV tile for head_dim D, cache dtype, block size.
int split_box_rows(int D, int kv_dtype, int bs);
// Bytes of one box row (the swizzle span): min(128, D * elem_bytes).
int split_box_row_bytes(int D, int kv_dtype);
// Query-row groups of 8 handled per pass for a plan with this max query length.
int split_row_groups(int max_qlen, int G);
// Upper bound on the extra (slot, row chunk) items a plan with these limits can list.
long long split_max_extra(int G, int rpc, long long rows_cap, int max_tokens, int max_qlen);

struct MergeParams {
  PlanDev plan;
  void* out;
  const int* context_lens;
  const int* cu;  // nullable
  int num_tokens, n, Hq, D, out_f16;
  int grid;       // persistent grid size
};

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
cudaError_t launch_split(const SplitParams& p, int C, int D, int kv_dtype, int row_groups,
                         const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s);
cudaError_t launch_split_d64(const SplitParams& p, int C, int kv_dtype, int row_groups,
                             const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s);
cudaError_t launch_split_d128(const SplitParams& p, int C, int kv_dtype, int row_groups,
                              const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s);
cudaError_t launch_split_d256(const SplitParams& p, int C, int kv_dtype, int row_groups,
                              const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s);

}  // namespace pa
