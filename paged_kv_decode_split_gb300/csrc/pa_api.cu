// pa_api.cu -- the C ABI declared in include/pa.h: argument validation (the
// capability gate of "[MiniMax-M3] Route the paged decode to aiter's FlyDSL
// kernel with work planner", review item 5), plan memory, TMA descriptors and
// the kernel launches.  Host code only; every step of the computation runs in
// the kernels of pa_plan.cu, pa_split_d*.cu and pa_merge.cu.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>

#include "../../include/pa.h"
#include "pa_internal.h"
#include "pa_split_cfg.h"

namespace {

struct TmapSlot {
  bool valid = false;
  const void* ptr = nullptr;
  int num_blocks = 0, Hkv = 0, bs = 0, D = 0, dtype = 0, grouped = 0;
  CUtensorMap map;
};

// Current-device guard: the ABI never leaves the caller's current device changed.
struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) return;
    ok = (prev == dev) || (cudaSetDevice(dev) == cudaSuccess);
  }
  ~DeviceGuard() {
    int cur;
    if (ok && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

struct pa_plan {
  int device, n, Hq, Hkv, D, max_qlen, max_tokens, P, W, kind, C, Q, rpc, sms;
  int kv_dtype;  // the cache type the decode calls are expected to read
  int wave;      // CTAs of that decode grid that run at once
  int window;          // sliding window for the next refresh (0: none)
  int fused_ok;   // the layout allows the fused merge (decode-only plan; tickets allocated)
  int fused;      // decode calls merge in the split kernel (no merge kernel launch)
  unsigned long long wait_ns;  // limit of the kernels' bounded waits
  int skip_stage;              // test hook (pa_plan_skip_stage_for_test); -1: off
  int window_planned;  // the window the last refresh planned with
  long long rows_cap, max_extra;
  pa::PlanDev dev;
  void* mem;
  long long bytes;
  int refreshed;  // 0: never; 1: without cu_query_lens; 2: with cu_query_lens
  cudaEvent_t ev_start, ev_stop;      // around the split kernel
  cudaEvent_t ev_call0, ev_call1;     // around the whole decode call
  TmapSlot tmaps[8];
  int tmap_next;
};

namespace pa {

int split_box_row_bytes(int D, int kv_dtype) {
  const int row = D * (kv_dtype == PA_FP8_E4M3 ? 1 : 2);
  return row < 128 ? row : 128;
}

int split_box_rows(int D, int kv_dtype, int bs) {
  // keys per stage: one 16-key tile above head_dim 256
  const int ks = D > 256 ? 16 : kStageTensorBytes / (D * (kv_dtype == PA_FP8_E4M3 ? 1 : 2));
  return bs < ks ? bs : ks;
}

int split_row_groups(int max_qlen, int G, int D) {
  const long long rows = static_cast<long long>(max_qlen) * G;
  int wq = 1;  // long prompts: 8-row work items, spread over the CTAs by work stealing
  if (rows <= 32) wq = static_cast<int>((rows + 7) / 8);
  return wq < split_max_row_groups(D) ? wq : split_max_row_groups(D);
}

long long split_max_extra(int G, int rpc, long long rows_cap, int max_tokens, int max_qlen) {
  if (static_cast<long long>(max_qlen) * G <= rpc) return 0;
  // sum_r T_r (ceil(L_r G / rpc) - 1) <= G / rpc * (sum_{T_r >= 2} T_r L_r + sum_{T_r = 1} L_r)
  // for T_r pieces of request r
  return (static_cast<long long>(G) * (rows_cap + max_tokens) + rpc - 1) / rpc;
}

namespace {
size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
}  // namespace

PlanLayout plan_layout(int num_seqs, int Hq, int Hkv, int D, int max_qlen, int max_tokens,
                       int max_partitions, int budget, int sms, bool pieces, bool fused) {
  PlanLayout l;
  const long long per_head = (static_cast<long long>(budget) + Hkv - 1) / Hkv;
  const long long lo = per_head > num_seqs ? per_head : num_seqs;
  const long long hi = static_cast<long long>(num_seqs) * max_partitions;
  l.C = hi < lo ? hi : lo;
  // Pieces: only decode-only plans whose grid is about one wave (2 CTAs per
  // SM) gain from cutting long slots; elsewhere tasks run whole.
  l.Q = (pieces && max_qlen == 1 && l.C * Hkv <= 4ll * sms) ? 4 : 1;
  long long rows = l.C * max_qlen;
  const long long rows_alt = static_cast<long long>(max_partitions) * max_tokens;
  if (rows_alt < rows) rows = rows_alt;
  if (rows < 1) rows = 1;
  l.rows_cap = rows * l.Q;  // sum_r T_r L_r <= Q sum_r p_r L_r
  const int G = Hq / Hkv;
  l.rpc = 8 * split_row_groups(max_qlen, G, D);
  l.max_extra = split_max_extra(G, l.rpc, l.rows_cap, max_tokens, max_qlen);
  // The split kernel can merge a request's partials itself when every query
  // row of a request (its tokens x G) is in one work item and the head dim is
  // at most 256 (the wide-head kernels are at their register limit and are
  // built without the fused merge).
  l.fused = (fused && static_cast<long long>(max_qlen) * G <= l.rpc && D <= 256) ? 1 : 0;
  l.levels = 0;
  if (l.fused) {
    const long long kmax = static_cast<long long>(l.Q) * max_partitions;
    long long cover = 1;
    while (cover < kmax && l.levels < kFusedLevels) {
      cover *= kFusedFanIn;
      ++l.levels;
    }
    if (l.levels < 1) l.levels = 1;
  }
  const size_t n = static_cast<size_t>(num_seqs);
  l.b_work = up256(static_cast<size_t>(l.C) * sizeof(int4));
  l.b_red = up256(n * sizeof(int2));
  l.b_snap = up256(n * sizeof(int2));
  l.b_err = 256;
  l.b_po = up256(static_cast<size_t>(l.rows_cap) * Hq * D * 4);
  l.b_pl = up256(static_cast<size_t>(l.rows_cap) * Hq * 4);
  l.b_pieces = up256(static_cast<size_t>(l.C) * l.Q * sizeof(int4));
  l.b_ext = up256(static_cast<size_t>(l.max_extra > 0 ? l.max_extra : 1) * sizeof(int2));
  l.b_mrow = up256(static_cast<size_t>(max_tokens) * sizeof(int4));
  l.b_preq = up256(n * sizeof(int2));
  l.b_tick = up256(static_cast<size_t>(l.levels > 0 ? l.levels : 1) * l.rows_cap * Hkv *
                   sizeof(int));
  l.total = l.b_work + l.b_red + l.b_snap + l.b_err + l.b_po + l.b_pl + l.b_pieces + l.b_ext +
            l.b_mrow + l.b_preq + l.b_tick;
  return l;
}

PlanDev carve_plan(char* c, const PlanLayout& l) {
  PlanDev d;
  d.work = reinterpret_cast<int4*>(c);
  c += l.b_work;
  d.reduce = reinterpret_cast<int2*>(c);
  c += l.b_red;
  d.snap = reinterpret_cast<int2*>(c);
  c += l.b_snap;
  d.err = reinterpret_cast<unsigned*>(c);
  d.counters = reinterpret_cast<int*>(c + 16);
  c += l.b_err;
  d.part_o = reinterpret_cast<float*>(c);
  c += l.b_po;
  d.part_lse = reinterpret_cast<float*>(c);
  c += l.b_pl;
  d.pieces = reinterpret_cast<int4*>(c);
  c += l.b_pieces;
  d.extra = reinterpret_cast<int2*>(c);
  c += l.b_ext;
  d.mrows = reinterpret_cast<int4*>(c);
  c += l.b_mrow;
  d.preq = reinterpret_cast<int2*>(c);
  c += l.b_preq;
  d.tickets = reinterpret_cast<int*>(c);
  return d;
}

// TMA view of a cache [num_blocks, Hkv, bs, D] as a 2-D tensor of
// num_blocks*Hkv*bs rows x D elements; boxes of split_box_rows() rows x one
// swizzle span (128 bytes, or 64 for a 64-byte row), swizzled to match the
// split kernel's shared-memory layout.  grouped: a K cache
// [num_blocks, Hkv, D/16, bs, 16] as the 3-D tensor
// {128 bytes, bs * 16 * elem / 128, num_blocks * Hkv * D/16} (innermost first):
// rows of 128 bytes, each 4 (fp8: 8) consecutive keys of one 16-dim group; one
// box is 16 keys of every group of one page and head, 128-byte swizzled.
// Every path that launches the split kernel encodes its maps here.
bool encode_cache_tmap(const void* ptr, int num_blocks, int Hkv, int bs, int D, int dtype,
                       bool grouped, CUtensorMap* out) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const int esz = dtype == PA_FP8_E4M3 ? 1 : 2;
  const int swb = split_box_row_bytes(D, dtype);
  const cuuint32_t rows = static_cast<cuuint32_t>(split_box_rows(D, dtype, bs));
  CUtensorMapDataType dt = dtype == PA_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                           : dtype == PA_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                              : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUresult r;
  if (grouped) {
    const cuuint64_t kpr = 128 / (16 * esz);  // keys per 128-byte row
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(128 / esz), bs / kpr,
                          static_cast<cuuint64_t>(num_blocks) * Hkv * (D / 16)};
    cuuint64_t strides[2] = {128, 128 * (bs / kpr)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / esz), static_cast<cuuint32_t>(16 / kpr),
                         static_cast<cuuint32_t>(D / 16)};
    cuuint32_t estr[3] = {1, 1, 1};
    r = fn(out, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(D),
                          static_cast<cuuint64_t>(num_blocks) * Hkv * bs};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * esz};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(swb / esz), rows};
    cuuint32_t estr[2] = {1, 1};
    r = fn(out, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE,
           swb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS;
}

cudaError_t launch_split(const SplitParams& p, int D, int kv_dtype, int row_groups, int k_layout,
                         const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s) {
  const bool gk = k_layout == PA_K_GROUPED;
  switch (D) {
    case 384: return launch_split_d384(p, kv_dtype, row_groups, k_layout, tk, tv, s);
    case 512: return launch_split_d512(p, kv_dtype, row_groups, k_layout, tk, tv, s);
    case 640: return launch_split_d640(p, kv_dtype, row_groups, k_layout, tk, tv, s);
    case 768: return launch_split_d768(p, kv_dtype, row_groups, k_layout, tk, tv, s);
    case 896: return launch_split_d896(p, kv_dtype, row_groups, k_layout, tk, tv, s);
    case 1024: return launch_split_d1024(p, kv_dtype, row_groups, k_layout, tk, tv, s);
    case 64:
      return (gk ? launch_split_d64_gk : launch_split_d64)(p, kv_dtype, row_groups, tk, tv, s);
    case 128:
      return (gk ? launch_split_d128_gk : launch_split_d128)(p, kv_dtype, row_groups, tk, tv, s);
    default:
      return (gk ? launch_split_d256_gk : launch_split_d256)(p, kv_dtype, row_groups, tk, tv, s);
  }
}

}  // namespace pa

namespace {

// Returns the cached tensor map of this cache view, or encodes one
// (pa::encode_cache_tmap) and keeps it in the plan's small cache.
int make_tmap(pa_plan* plan, const void* ptr, int num_blocks, int Hkv, int bs, int D, int dtype,
              int grouped, CUtensorMap* out) {
  for (auto& s : plan->tmaps) {
    if (s.valid && s.ptr == ptr && s.num_blocks == num_blocks && s.Hkv == Hkv && s.bs == bs &&
        s.D == D && s.dtype == dtype && s.grouped == grouped) {
      *out = s.map;
      return PA_OK;
    }
  }
  CUtensorMap m;
  if (!pa::encode_cache_tmap(ptr, num_blocks, Hkv, bs, D, dtype, grouped != 0, &m))
    return PA_ERR_CUDA;
  TmapSlot& s = plan->tmaps[plan->tmap_next];
  plan->tmap_next = (plan->tmap_next + 1) % 8;
  s.valid = true;
  s.ptr = ptr;
  s.num_blocks = num_blocks;
  s.Hkv = Hkv;
  s.bs = bs;
  s.D = D;
  s.dtype = dtype;
  s.grouped = grouped;
  s.map = m;
  *out = m;
  return PA_OK;
}

}  // namespace

extern "C" {

const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_PLAN_MISMATCH: return "PA_ERR_PLAN_MISMATCH";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_OOM: return "PA_ERR_OOM";
    default: return "PA_ERR_UNKNOWN";
  }
}

int pa_plan_build(pa_plan** plan, int device, int num_seqs, int num_kv_heads, int num_q_heads,
                  int head_dim, int max_query_len, int max_tokens, int max_partitions, int budget,
                  int kind) {
  if (!plan) return PA_ERR_INVALID_ARG;
  *plan = nullptr;
  if (device < 0 || num_seqs < 1 || num_q_heads < 1 || num_kv_heads < 1 || max_query_len < 1 ||
      max_tokens < 1)
    return PA_ERR_INVALID_ARG;
  if (kind != PA_PLAN_PROPORTIONAL && kind != PA_PLAN_UNIFORM) return PA_ERR_INVALID_ARG;
  if (num_seqs > PA_MAX_SEQS) return PA_ERR_UNSUPPORTED;
  if (num_q_heads % num_kv_heads != 0) return PA_ERR_UNSUPPORTED;
  if (!pa::head_dim_supported(head_dim)) return PA_ERR_UNSUPPORTED;
  if (max_partitions <= 0) max_partitions = PA_DEFAULT_MAX_PARTITIONS;
  if (max_partitions > 65536 || budget > (1 << 24)) return PA_ERR_UNSUPPORTED;
  if (static_cast<long long>(max_query_len) * (num_q_heads / num_kv_heads) > (1 << 24) ||
      max_tokens > (1 << 28))
    return PA_ERR_UNSUPPORTED;

  DeviceGuard guard(device);
  if (!guard.ok) return PA_ERR_CUDA;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      sms <= 0)
    return PA_ERR_CUDA;
  if (budget <= 0) budget = 2 * sms;
  const pa::PlanLayout lay = pa::plan_layout(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                             max_query_len, max_tokens, max_partitions, budget, sms,
                                             true, true);
  const size_t total = lay.total;

  pa_plan* pl = new (std::nothrow) pa_plan();
  if (!pl) return PA_ERR_OOM;
  void* mem = nullptr;
  if (cudaMalloc(&mem, total) != cudaSuccess) {
    cudaGetLastError();
    delete pl;
    return PA_ERR_OOM;
  }
  pl->dev = pa::carve_plan(static_cast<char*>(mem), lay);
  if (cudaMemset(pl->dev.err, 0, 64) != cudaSuccess ||
      cudaMemset(pl->dev.tickets, 0, lay.b_tick) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    cudaFree(mem);
    delete pl;
    return PA_ERR_CUDA;
  }
  pl->device = device;
  pl->n = num_seqs;
  pl->Hq = num_q_heads;
  pl->Hkv = num_kv_heads;
  pl->D = head_dim;
  pl->max_qlen = max_query_len;
  pl->max_tokens = max_tokens;
  pl->P = max_partitions;
  pl->W = budget;
  pl->kind = kind;
  pl->C = static_cast<int>(lay.C);
  pl->Q = lay.Q;
  pl->rpc = lay.rpc;
  pl->sms = sms;
  pl->kv_dtype = PA_BF16;
  pl->wave = pa::split_ctas_per_sm(head_dim, PA_BF16, lay.rpc / 8) * sms;
  pl->rows_cap = lay.rows_cap;
  pl->max_extra = lay.max_extra;
  pl->mem = mem;
  pl->bytes = static_cast<long long>(total);
  pl->refreshed = 0;
  pl->ev_start = pl->ev_stop = nullptr;
  pl->window = pl->window_planned = 0;
  pl->ev_call0 = pl->ev_call1 = nullptr;
  pl->tmap_next = 0;
  pl->wait_ns = pa::kWaitLimitNs;
  pl->skip_stage = -1;
  pl->fused_ok = lay.fused;
  pl->fused = 0;  // measured slower than the merge kernel on every batch tried

  *plan = pl;
  return PA_OK;
}

int pa_plan_refresh(pa_plan* plan, const int32_t* context_lens, const int32_t* cu_query_lens,
                    void* stream) {
  if (!plan || !context_lens) return PA_ERR_INVALID_ARG;
  DeviceGuard guard(plan->device);
  if (!guard.ok) return PA_ERR_CUDA;
  pa::PlanParams p;
  p.context_lens = context_lens;
  p.cu = cu_query_lens;
  p.n = plan->n;
  p.Hkv = plan->Hkv;
  p.P = plan->P;
  p.C = plan->C;
  p.Q = plan->Q;
  p.window = plan->window;
  p.kind = plan->kind;
  p.max_qlen = plan->max_qlen;
  p.max_tokens = plan->max_tokens;
  p.G = plan->Hq / plan->Hkv;
  p.rpc = plan->rpc;
  p.wave = plan->wave;
  p.rows_cap = plan->rows_cap;
  p.max_extra = plan->max_extra;
  p.dev = plan->dev;
  if (pa::launch_plan(p, static_cast<cudaStream_t>(stream)) != cudaSuccess) return PA_ERR_CUDA;
  plan->refreshed = cu_query_lens ? 2 : 1;
  plan->window_planned = plan->window;
  return PA_OK;
}

int pa_plan_set_window(pa_plan* plan, int sliding_window) {
  if (!plan || sliding_window < 0) return PA_ERR_INVALID_ARG;
  plan->window = sliding_window;
  return PA_OK;
}

int pa_plan_set_wait_limit(pa_plan* plan, long long wait_limit_ns) {
  if (!plan || wait_limit_ns < 0) return PA_ERR_INVALID_ARG;
  if (wait_limit_ns > 0 && wait_limit_ns < 10000) return PA_ERR_INVALID_ARG;
  plan->wait_ns = wait_limit_ns == 0 ? pa::kWaitLimitNs
                                     : static_cast<unsigned long long>(wait_limit_ns);
  return PA_OK;
}

int pa_plan_set_fused_merge(pa_plan* plan, int enable) {
  if (!plan || (enable != 0 && enable != 1)) return PA_ERR_INVALID_ARG;
  if (enable && !plan->fused_ok) return PA_ERR_UNSUPPORTED;
  plan->fused = enable;
  return PA_OK;
}

int pa_plan_get_fused_merge(const pa_plan* plan, int* enabled) {
  if (!plan || !enabled) return PA_ERR_INVALID_ARG;
  *enabled = plan->fused;
  return PA_OK;
}

int pa_plan_skip_stage_for_test(pa_plan* plan, int stage) {
  if (!plan || stage < -1) return PA_ERR_INVALID_ARG;
  plan->skip_stage = stage;
  return PA_OK;
}

int pa_plan_set_kv_dtype(pa_plan* plan, int kv_dtype) {
  if (!plan || (kv_dtype != PA_BF16 && kv_dtype != PA_FP16 && kv_dtype != PA_FP8_E4M3))
    return PA_ERR_INVALID_ARG;
  plan->kv_dtype = kv_dtype;
  plan->wave = pa::split_ctas_per_sm(plan->D, kv_dtype, plan->rpc / 8) * plan->sms;
  return PA_OK;
}

int pa_decode(pa_plan* plan, const void* q, int q_dtype, int num_tokens, int num_q_heads,
              int head_dim, const void* k_cache, const void* v_cache, int kv_dtype, float k_scale,
              float v_scale, int num_blocks, int num_kv_heads, int block_size,
              const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
              const int32_t* cu_query_lens, int num_seqs, float scale, void* out, void* stream) {
  return pa_decode_ex(plan, q, q_dtype, num_tokens, num_q_heads, head_dim, k_cache, v_cache,
                      kv_dtype, k_scale, v_scale, num_blocks, num_kv_heads, block_size,
                      block_tables, max_blocks_per_seq, context_lens, cu_query_lens, num_seqs,
                      scale, nullptr, PA_K_ROWS, out, stream);
}

int pa_decode_ex(pa_plan* plan, const void* q, int q_dtype, int num_tokens, int num_q_heads,
                 int head_dim, const void* k_cache, const void* v_cache, int kv_dtype,
                 float k_scale, float v_scale, int num_blocks, int num_kv_heads, int block_size,
                 const int32_t* block_tables, int max_blocks_per_seq,
                 const int32_t* context_lens, const int32_t* cu_query_lens, int num_seqs,
                 float scale, const float* sinks, int k_layout, void* out, void* stream) {
  if (!plan) return PA_ERR_INVALID_ARG;
  if (k_layout != PA_K_ROWS && k_layout != PA_K_GROUPED) return PA_ERR_UNSUPPORTED;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return PA_ERR_INVALID_ARG;
  if (num_tokens < 1 || num_blocks < 1 || max_blocks_per_seq < 1) return PA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (q_dtype != PA_BF16 && q_dtype != PA_FP16) return PA_ERR_UNSUPPORTED;
  if (kv_dtype != PA_BF16 && kv_dtype != PA_FP16 && kv_dtype != PA_FP8_E4M3)
    return PA_ERR_UNSUPPORTED;
  if ((kv_dtype == PA_BF16 && q_dtype != PA_BF16) || (kv_dtype == PA_FP16 && q_dtype != PA_FP16))
    return PA_ERR_UNSUPPORTED;
  if (kv_dtype == PA_FP8_E4M3 && (!std::isfinite(k_scale) || !std::isfinite(v_scale)))
    return PA_ERR_INVALID_ARG;
  if (block_size != 16 && block_size != 64 && block_size != 128) return PA_ERR_UNSUPPORTED;
  if (!pa::head_dim_supported(head_dim)) return PA_ERR_UNSUPPORTED;
  if (num_kv_heads < 1 || num_q_heads % num_kv_heads != 0) return PA_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_blocks) * num_kv_heads * block_size >= (1ll << 31))
    return PA_ERR_UNSUPPORTED;
  if (num_seqs != plan->n || num_q_heads != plan->Hq || num_kv_heads != plan->Hkv ||
      head_dim != plan->D)
    return PA_ERR_PLAN_MISMATCH;
  if (plan->refreshed == 0 || (cu_query_lens != nullptr) != (plan->refreshed == 2))
    return PA_ERR_PLAN_MISMATCH;
  if (!cu_query_lens && num_tokens != num_seqs) return PA_ERR_INVALID_ARG;

  DeviceGuard guard(plan->device);
  if (!guard.ok) return PA_ERR_CUDA;
  CUtensorMap tk, tv;
  int st = make_tmap(plan, k_cache, num_blocks, num_kv_heads, block_size, head_dim, kv_dtype,
                     k_layout == PA_K_GROUPED ? 1 : 0, &tk);
  if (st != PA_OK) return st;
  st = make_tmap(plan, v_cache, num_blocks, num_kv_heads, block_size, head_dim, kv_dtype, 0, &tv);
  if (st != PA_OK) return st;

  const bool fp8 = kv_dtype == PA_FP8_E4M3;
  pa::SplitParams sp;
  sp.plan = plan->dev;
  sp.q = q;
  sp.out = out;
  sp.block_tables = block_tables;
  sp.context_lens = context_lens;
  sp.cu = cu_query_lens;
  sp.num_tokens = num_tokens;
  sp.num_blocks = num_blocks;
  sp.Hq = num_q_heads;
  sp.Hkv = num_kv_heads;
  sp.G = num_q_heads / num_kv_heads;
  sp.bs = block_size;
  sp.max_blocks = max_blocks_per_seq;
  sp.n = num_seqs;
  sp.C = plan->C;
  sp.sms = plan->sms;
  sp.resident = 0;
  sp.total_rows = num_blocks * num_kv_heads * block_size;
  sp.out_f16 = q_dtype == PA_FP16 ? 1 : 0;
  sp.rpc = plan->rpc;
  sp.scale_log2 = static_cast<float>(static_cast<double>(scale) * (fp8 ? k_scale : 1.0) *
                                     1.4426950408889634);
  sp.v_scale = fp8 ? v_scale : 1.0f;
  sp.window = plan->window_planned;
  sp.sinks = sinks;
  sp.wait_ns = plan->wait_ns;
  sp.skip_stage = plan->skip_stage;
  sp.fused = plan->fused;
  sp.rows_cap = plan->rows_cap;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int wq = pa::split_row_groups(plan->max_qlen, sp.G, head_dim);
  // Profiling events: inside a stream capture they must be external event
  // records to fire on every replay of the graph.
  auto record = [&](cudaEvent_t e) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return false;
    return (cs == cudaStreamCaptureStatusActive
                ? cudaEventRecordWithFlags(e, s, cudaEventRecordExternal)
                : cudaEventRecord(e, s)) == cudaSuccess;
  };
  if (plan->ev_call0 && !record(plan->ev_call0)) return PA_ERR_CUDA;
  if (plan->ev_start && !record(plan->ev_start)) return PA_ERR_CUDA;
  if (pa::launch_split(sp, head_dim, kv_dtype, wq, k_layout, tk, tv, s) != cudaSuccess)
    return PA_ERR_CUDA;
  if (plan->ev_stop && !record(plan->ev_stop)) return PA_ERR_CUDA;

  if (!plan->fused) {
  pa::MergeParams mp;
  mp.plan = plan->dev;
  mp.out = out;
  mp.context_lens = context_lens;
  mp.cu = cu_query_lens;
  mp.num_tokens = num_tokens;
  mp.n = num_seqs;
  mp.Hq = num_q_heads;
  mp.D = head_dim;
  mp.out_f16 = sp.out_f16;
  mp.sinks = sinks;
  const long long pairs = static_cast<long long>(num_tokens) * num_q_heads;
  mp.grid = static_cast<int>(pairs < 8ll * plan->sms ? pairs : 8ll * plan->sms);
  if (pa::launch_merge(mp, s) != cudaSuccess) return PA_ERR_CUDA;
  }
  if (plan->ev_call1 && !record(plan->ev_call1)) return PA_ERR_CUDA;
  return PA_OK;
}

int pa_plan_info(const pa_plan* plan, int* capacity, int* num_seqs, int* budget,
                 int* max_partitions, int* kind, int* device, long long* device_bytes) {
  if (!plan) return PA_ERR_INVALID_ARG;
  if (capacity) *capacity = plan->C;
  if (num_seqs) *num_seqs = plan->n;
  if (budget) *budget = plan->W;
  if (max_partitions) *max_partitions = plan->P;
  if (kind) *kind = plan->kind;
  if (device) *device = plan->device;
  if (device_bytes) *device_bytes = plan->bytes;
  return PA_OK;
}

int pa_plan_download(const pa_plan* plan, int32_t* work_info, int32_t* reduce_info, int* capacity,
                     void* stream) {
  if (!plan) return PA_ERR_INVALID_ARG;
  if (capacity) *capacity = plan->C;
  DeviceGuard guard(plan->device);
  if (!guard.ok) return PA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (work_info && cudaMemcpyAsync(work_info, plan->dev.work,
                                   static_cast<size_t>(plan->C) * sizeof(int4),
                                   cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return PA_ERR_CUDA;
  if (reduce_info && cudaMemcpyAsync(reduce_info, plan->dev.reduce,
                                     static_cast<size_t>(plan->n) * sizeof(int2),
                                     cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

int pa_plan_read_errors(pa_plan* plan, uint32_t* errors, int clear, void* stream) {
  if (!plan || !errors) return PA_ERR_INVALID_ARG;
  DeviceGuard guard(plan->device);
  if (!guard.ok) return PA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(errors, plan->dev.err, sizeof(unsigned), cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  if (clear && cudaMemsetAsync(plan->dev.err, 0, sizeof(unsigned), s) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

int pa_plan_set_split_events(pa_plan* plan, void* start_event, void* stop_event) {
  if (!plan) return PA_ERR_INVALID_ARG;
  if ((start_event == nullptr) != (stop_event == nullptr)) return PA_ERR_INVALID_ARG;
  plan->ev_start = static_cast<cudaEvent_t>(start_event);
  plan->ev_stop = static_cast<cudaEvent_t>(stop_event);
  return PA_OK;
}

int pa_plan_set_call_events(pa_plan* plan, void* start_event, void* stop_event) {
  if (!plan) return PA_ERR_INVALID_ARG;
  if ((start_event == nullptr) != (stop_event == nullptr)) return PA_ERR_INVALID_ARG;
  plan->ev_call0 = static_cast<cudaEvent_t>(start_event);
  plan->ev_call1 = static_cast<cudaEvent_t>(stop_event);
  return PA_OK;
}

int pa_plan_destroy(pa_plan* plan) {
  if (!plan) return PA_OK;
  int st = PA_OK;
  {
    DeviceGuard guard(plan->device);
    if (!guard.ok || cudaFree(plan->mem) != cudaSuccess) st = PA_ERR_CUDA;
  }
  delete plan;
  return st;
}

}  // extern "C"
