// Tensor-core decode attention, head dim 128, 4-bit keys (values of 1-4 bits).
#include "attn_mma.cuh"

namespace tq {
cudaError_t launch_attn_mma_d128_k4(const AttnParams& p, dim3 grid, cudaStream_t s) {
  switch (p.vb) {
    case 1: return attn_mma_launch_t<128, 4, 1>(p, grid, s);
    case 2: return attn_mma_launch_t<128, 4, 2>(p, grid, s);
    case 3: return attn_mma_launch_t<128, 4, 3>(p, grid, s);
    case 4: return attn_mma_launch_t<128, 4, 4>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace tq
