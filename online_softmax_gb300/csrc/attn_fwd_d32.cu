// Instances of the tcgen05 attention kernel for head dimension 32 (key tiles 32, 64, 128;
// f16 and bf16).  One translation unit per head dimension so they compile in parallel.
#include "attn_fwd.cuh"

namespace oattn {
cudaError_t launch_attn_d32(const AttnArgs& a, int block_n, int bf16, cudaStream_t st) {
  return launch_attn_d<32>(a, block_n, bf16, st);
}
}  // namespace oattn
