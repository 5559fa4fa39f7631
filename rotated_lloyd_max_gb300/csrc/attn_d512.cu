// Decode-attention instantiations for head dim 512 (query-head groups of 1, 2, 4, 6, 8) and the
// tensor-core dense-split kernel (groups of 16 query heads).
#include "attn.cuh"
#include "attn_dense512.cuh"

namespace tq {
cudaError_t launch_attn_d512(const AttnParams& p, int GT, dim3 grid, cudaStream_t s) {
  switch (GT) {
    case 1: return attn_launch_t<512, 1>(p, grid, s);
    case 2: return attn_launch_t<512, 2>(p, grid, s);
    case 4: return attn_launch_t<512, 4>(p, grid, s);
    case 6: return attn_launch_t<512, 6>(p, grid, s);
    case 8: return attn_launch_t<512, 8>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}
cudaError_t launch_attn_dense512(const AttnParams& p, dim3 grid, cudaStream_t s) {
  return attn_dense512_launch(p, grid, s);
}
int attn_dense512_smem_bytes() { return attn_dense512_smem(); }
}  // namespace tq
