// tcgen05 decode attention, head dim 512, 2-bit keys (values of 1-4 bits).
#include "attn_umma512.cuh"

namespace tq {
cudaError_t launch_attn_umma512_k2(const AttnParams& p, dim3 grid, cudaStream_t s) {
  switch (p.vb) {
    case 1: return attn_umma512_launch_t<2, 1>(p, grid, s);
    case 2: return attn_umma512_launch_t<2, 2>(p, grid, s);
    case 3: return attn_umma512_launch_t<2, 3>(p, grid, s);
    case 4: return attn_umma512_launch_t<2, 4>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace tq
