// The tensor-core encoders (encode_mma.cuh) at head dim 256.
#include "encode_mma.cuh"

namespace tq {
cudaError_t launch_encode_mma_d256(const EncodeParams& p, int grid, cudaStream_t s) {
  return encm_dispatch<256>(p, grid, s);
}
}  // namespace tq
