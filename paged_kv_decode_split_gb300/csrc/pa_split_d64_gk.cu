// pa_split_d64_gk.cu -- split-KV decode kernels for head_dim 64 with the K
// cache in the grouped layout [num_blocks, Hkv, 64/16, block_size, 16] (bf16,
// fp16 and fp8-e4m3 caches; 1 to 4 query-row groups per pass).
#include "pa_split.cuh"

namespace pa {

cudaError_t launch_split_d64_gk(const SplitParams& p, int kv_dtype, int row_groups,
                               const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s) {
  return launch_split_d<64, 1>(p, kv_dtype, row_groups, tk, tv, s);
}

}  // namespace pa
