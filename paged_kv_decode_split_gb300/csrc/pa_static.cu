// pa_static.cu -- pa_decode_static: plan + split-KV decode + merge in one call
// that allocates no device memory.
//
// Who needs it: callers that cannot call cudaMalloc at decode time.  A serving
// engine typically hands (almost) all HBM to its own KV-cache pool and caching
// allocator at start-up, so a library allocation either fails outright or
// carves into memory the engine has already promised to its KV pages; an
// embedded runtime may not be allowed to allocate device memory at all once it
// is serving.  Such callers cannot create a pa_plan, whose device buffers come
// from pa_plan_build.
//
// Instead, the plan arrays and the fp32 partial results live in one file-scope
// __device__ array of PA_STATIC_SCRATCH_BYTES.  Every GPU on which this module is
// loaded holds that memory until the process exits.  In host code the array's
// name is only a host-side stand-in, never a device address: the address is
// obtained once per device with cudaGetSymbolAddress, with that device current,
// on the first call made on that device (so that first call should happen
// before any stream capture), and then passed to the kernels as a pointer.
//
// All calls share the one array and it keeps the last call's contents.  Each
// call rewrites the whole plan before using it and clears the error word it
// uses, so nothing stale is read; but calls whose work overlaps on the GPU
// (other streams or other threads) race on the array and must be serialised by the caller.  The tensor maps of
// the caches come from pa::encode_cache_tmap, the encoder pa_decode uses.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/pa.h"
#include "pa_internal.h"
#include "pa_split_cfg.h"

namespace {

__device__ __align__(256) unsigned char g_pa_static_scratch[PA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array on `device` (which must be current).
void* scratch_address(int device) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[device]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pa_static_scratch) != cudaSuccess || !p) return nullptr;
    g_addr[device] = p;
  }
  return g_addr[device];
}

}  // namespace

extern "C" int pa_decode_static(const void* q, int q_dtype, int num_tokens, int num_q_heads,
                                int head_dim, const void* k_cache, const void* v_cache,
                                int kv_dtype, float k_scale, float v_scale, int num_blocks,
                                int num_kv_heads, int block_size, const int32_t* block_tables,
                                int max_blocks_per_seq, const int32_t* context_lens,
                                const int32_t* cu_query_lens, int num_seqs, int max_query_len,
                                int max_partitions, int budget, int kind, float scale, void* out,
                                uint32_t* device_errors, void* stream) {
  // ---- arguments (the same domain as pa_plan_build + pa_decode)
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return PA_ERR_INVALID_ARG;
  if (num_seqs < 1 || num_tokens < 1 || num_blocks < 1 || max_blocks_per_seq < 1 ||
      max_query_len < 1 || num_q_heads < 1 || num_kv_heads < 1)
    return PA_ERR_INVALID_ARG;
  if (kind != PA_PLAN_PROPORTIONAL && kind != PA_PLAN_UNIFORM) return PA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out) |
       reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15u)
    return PA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (q_dtype != PA_BF16 && q_dtype != PA_FP16) return PA_ERR_UNSUPPORTED;
  if (kv_dtype != PA_BF16 && kv_dtype != PA_FP16 && kv_dtype != PA_FP8_E4M3)
    return PA_ERR_UNSUPPORTED;
  if ((kv_dtype == PA_BF16 && q_dtype != PA_BF16) || (kv_dtype == PA_FP16 && q_dtype != PA_FP16))
    return PA_ERR_UNSUPPORTED;
  if (kv_dtype == PA_FP8_E4M3 && (!std::isfinite(k_scale) || !std::isfinite(v_scale)))
    return PA_ERR_INVALID_ARG;
  if (num_seqs > PA_MAX_SEQS || num_q_heads % num_kv_heads != 0) return PA_ERR_UNSUPPORTED;
  if (!pa::head_dim_supported(head_dim)) return PA_ERR_UNSUPPORTED;
  if (block_size != 16 && block_size != 64 && block_size != 128) return PA_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_blocks) * num_kv_heads * block_size >= (1ll << 31))
    return PA_ERR_UNSUPPORTED;
  if (!cu_query_lens && num_tokens != num_seqs) return PA_ERR_INVALID_ARG;
  if (max_partitions <= 0) max_partitions = PA_DEFAULT_MAX_PARTITIONS;
  if (max_partitions > 65536 || budget > (1 << 24)) return PA_ERR_UNSUPPORTED;
  if (static_cast<long long>(max_query_len) * (num_q_heads / num_kv_heads) > (1 << 24))
    return PA_ERR_UNSUPPORTED;

  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices)
    return PA_ERR_CUDA;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      sms <= 0)
    return PA_ERR_CUDA;
  if (budget <= 0) budget = 2 * sms;

  // ---- carve the static array: plan arrays, error word, partial results
  // (cutting long slots into pieces needs more partial rows: drop it first)
  pa::PlanLayout lay = pa::plan_layout(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                       max_query_len, num_tokens, max_partitions, budget, sms, true,
                                       false);
  if (lay.total > PA_STATIC_SCRATCH_BYTES)
    lay = pa::plan_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_query_len,
                          num_tokens, max_partitions, budget, sms, false, false);
  if (lay.total > PA_STATIC_SCRATCH_BYTES)
    return PA_ERR_UNSUPPORTED;  // this batch needs more scratch than the static array holds
  const int G = num_q_heads / num_kv_heads;
  const int wq = pa::split_row_groups(max_query_len, G, head_dim);

  char* base = static_cast<char*>(scratch_address(device));
  if (!base) return PA_ERR_CUDA;
  pa::PlanDev dev = pa::carve_plan(base, lay);
  unsigned* own_err = dev.err;
  dev.err = device_errors ? reinterpret_cast<unsigned*>(device_errors) : own_err;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!device_errors && cudaMemsetAsync(own_err, 0, sizeof(unsigned), s) != cudaSuccess)
    return PA_ERR_CUDA;

  CUtensorMap tk, tv;
  if (!pa::encode_cache_tmap(k_cache, num_blocks, num_kv_heads, block_size, head_dim, kv_dtype,
                             false, &tk) ||
      !pa::encode_cache_tmap(v_cache, num_blocks, num_kv_heads, block_size, head_dim, kv_dtype,
                             false, &tv))
    return PA_ERR_CUDA;

  // ---- plan, split, merge
  pa::PlanParams pp;
  pp.context_lens = context_lens;
  pp.cu = cu_query_lens;
  pp.n = num_seqs;
  pp.Hkv = num_kv_heads;
  pp.P = max_partitions;
  pp.C = static_cast<int>(lay.C);
  pp.Q = lay.Q;
  pp.window = 0;
  pp.kind = kind;
  pp.max_qlen = max_query_len;
  pp.max_tokens = num_tokens;
  pp.G = G;
  pp.rpc = lay.rpc;
  pp.wave = pa::split_ctas_per_sm(head_dim, kv_dtype, wq) * sms;
  pp.rows_cap = lay.rows_cap;
  pp.max_extra = lay.max_extra;
  pp.dev = dev;
  if (pa::launch_plan(pp, s) != cudaSuccess) return PA_ERR_CUDA;

  const bool fp8 = kv_dtype == PA_FP8_E4M3;
  pa::SplitParams sp;
  sp.plan = dev;
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
  sp.C = static_cast<int>(lay.C);
  sp.sms = sms;
  sp.resident = 0;
  sp.total_rows = num_blocks * num_kv_heads * block_size;
  sp.out_f16 = q_dtype == PA_FP16 ? 1 : 0;
  sp.rpc = lay.rpc;
  sp.window = 0;
  sp.sinks = nullptr;
  sp.wait_ns = pa::kWaitLimitNs;
  sp.skip_stage = -1;
  sp.fused = 0;
  sp.rows_cap = lay.rows_cap;
  sp.scale_log2 = static_cast<float>(static_cast<double>(scale) * (fp8 ? k_scale : 1.0) *
                                     1.4426950408889634);
  sp.v_scale = fp8 ? v_scale : 1.0f;
  if (pa::launch_split(sp, head_dim, kv_dtype, wq, PA_K_ROWS, tk, tv, s) != cudaSuccess)
    return PA_ERR_CUDA;

  pa::MergeParams mp;
  mp.plan = dev;
  mp.out = out;
  mp.context_lens = context_lens;
  mp.cu = cu_query_lens;
  mp.num_tokens = num_tokens;
  mp.n = num_seqs;
  mp.Hq = num_q_heads;
  mp.D = head_dim;
  mp.out_f16 = sp.out_f16;
  mp.sinks = nullptr;
  const long long pairs = static_cast<long long>(num_tokens) * num_q_heads;
  mp.grid = static_cast<int>(pairs < 8ll * sms ? pairs : 8ll * sms);
  if (pa::launch_merge(mp, s) != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}
