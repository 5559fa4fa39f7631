// tq_encode's kernels: the tensor-core encoders (encode_mma.cuh) at head
// dim 128, and their dispatch by head dim (64, 256 and 512 in their own
// units).  The CUDA-core encoder of encode_core.cuh serves the eviction.
#include "encode_mma.cuh"

namespace tq {

cudaError_t launch_encode_mma_d64(const EncodeParams& p, int grid, cudaStream_t s);
cudaError_t launch_encode_mma_d256(const EncodeParams& p, int grid, cudaStream_t s);
cudaError_t launch_encode_mma_d512(const EncodeParams& p, int grid, cudaStream_t s);

cudaError_t launch_encode(const EncodeParams& p, int grid, cudaStream_t s) {
  switch (p.c.d) {
    case 64: return launch_encode_mma_d64(p, grid, s);
    case 128: return encm_dispatch<128>(p, grid, s);
    case 256: return launch_encode_mma_d256(p, grid, s);
    case 512: return launch_encode_mma_d512(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tq
