// Decode-attention instantiations for head dim 128 (query-head groups of 1, 2, 4, 6, 8):
// the general kernel and the warp-local kernel for the compressed splits.
#include "attn_rec.cuh"

namespace tq {
cudaError_t launch_attn_d128(const AttnParams& p, int GT, dim3 grid, cudaStream_t s) {
  switch (GT) {
    case 1: return attn_launch_t<128, 1>(p, grid, s);
    case 2: return attn_launch_t<128, 2>(p, grid, s);
    case 4: return attn_launch_t<128, 4>(p, grid, s);
    case 6: return attn_launch_t<128, 6>(p, grid, s);
    case 8: return attn_launch_t<128, 8>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}
cudaError_t launch_attn_rec_d128(const AttnParams& p, int GT, dim3 grid, cudaStream_t s) {
  switch (GT) {
    case 1: return attn_rec_launch_t<128, 1>(p, grid, s);
    case 2: return attn_rec_launch_t<128, 2>(p, grid, s);
    case 4: return attn_rec_launch_t<128, 4>(p, grid, s);
    case 6: return attn_rec_launch_t<128, 6>(p, grid, s);
    case 8: return attn_rec_launch_t<128, 8>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace tq
