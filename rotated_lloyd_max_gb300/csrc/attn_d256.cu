// Decode-attention instantiations for head dim 256 (query-head groups of 1, 2, 4, 6, 8).
#include "attn.cuh"

namespace tq {
cudaError_t launch_attn_d256(const AttnParams& p, int GT, dim3 grid, cudaStream_t s) {
  switch (GT) {
    case 1: return attn_launch_t<256, 1>(p, grid, s);
    case 2: return attn_launch_t<256, 2>(p, grid, s);
    case 4: return attn_launch_t<256, 4>(p, grid, s);
    case 6: return attn_launch_t<256, 6>(p, grid, s);
    case 8: return attn_launch_t<256, 8>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace tq
