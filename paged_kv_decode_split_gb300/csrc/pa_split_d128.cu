// pa_split_d128.cu -- split-KV decode kernels for head_dim 128 (bf16, fp16 and
// fp8-e4m3 caches; 1 to 4 query-row groups per pass).
#include "pa_split.cuh"

namespace pa {

cudaError_t launch_split_d128(const SplitParams& p, int kv_dtype, int row_groups,
                             const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s) {
  return launch_split_d<128, 0>(p, kv_dtype, row_groups, tk, tv, s);
}

}  // namespace pa
