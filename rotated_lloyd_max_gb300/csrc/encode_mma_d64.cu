// The tensor-core encoders (encode_mma.cuh) at head dim 64.
#include "encode_mma.cuh"

namespace tq {
cudaError_t launch_encode_mma_d64(const EncodeParams& p, int grid, cudaStream_t s) {
  return encm_dispatch<64>(p, grid, s);
}
}  // namespace tq
