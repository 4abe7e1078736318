// pa_split_d768.cu -- split-KV decode kernels for head_dim 768 (bf16, fp16 and
// fp8-e4m3 caches; K row-major or grouped; 1 query-row group per pass).
#include "pa_split.cuh"

namespace pa {

cudaError_t launch_split_d768(const SplitParams& p, int kv_dtype, int row_groups, int k_layout,
                                const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s) {
  return k_layout == PA_K_GROUPED ? launch_split_d<768, 1>(p, kv_dtype, row_groups, tk, tv, s)
                                  : launch_split_d<768, 0>(p, kv_dtype, row_groups, tk, tv, s);
}

}  // namespace pa
