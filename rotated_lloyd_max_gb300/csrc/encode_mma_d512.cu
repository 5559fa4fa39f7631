// The tensor-core encoders (encode_mma.cuh) at head dim 512.
#include "encode_mma.cuh"

namespace tq {
cudaError_t launch_encode_mma_d512(const EncodeParams& p, int grid, cudaStream_t s) {
  return encm_dispatch<512>(p, grid, s);
}
}  // namespace tq
