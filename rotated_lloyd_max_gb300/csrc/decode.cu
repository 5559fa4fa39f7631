// Decode records back to f32 head vectors (tq_decode); the per-slot
// arithmetic is in decode_core.cuh.
#include "decode_core.cuh"

namespace tq {

template <int D, int B, bool OUTL>
__global__ void __launch_bounds__(kThreads) decode_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int L = D / 32, VPW = 32 / L, VPC = 4 * VPW;
  __shared__ float lut[16];
  __shared__ int pre[kChunk + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int lg = lane % L, vi = lane / L;
  if (threadIdx.x < 16) lut[threadIdx.x] = p.c.centroids[threadIdx.x & ((1 << B) - 1)];
  // CTA b takes part b % 2^lp (kChunk >> lp slots) of its records; the grid
  // is a multiple of 2^lp
  // (head dim 512 keeps one CTA per record: ptxas 13.0 fails register
  // allocation on its instantiation with a runtime part count)
  const int lp = D >= 512 ? 0 : p.log2_parts;
  const int part = (int)blockIdx.x & ((1 << lp) - 1), per = kChunk >> lp;
  const int64_t n_tasks = p.n_groups * p.chunks_per_group;
  for (int64_t task = blockIdx.x >> lp; task < n_tasks; task += gridDim.x >> lp) {
    const int64_t g = task / p.chunks_per_group;
    const int64_t ci = p.first_chunk + task % p.chunks_per_group;
    const int64_t lo = max(p.first_vec, ci * kChunk + part * per);
    const int64_t hi = min(p.first_vec + p.n_vec, ci * kChunk + (part + 1) * per);
    const uint8_t* rec = p.src + g * p.src_gs + ci * (int64_t)p.c.rec_bytes;
    float* dst_g = p.dst + g * p.dst_gs;
    __syncthreads();  // lut ready; pre[] of the previous task consumed
    if (OUTL) {
      outlier_prefix(rec, p.c, pre);
      __syncthreads();
    }
    for (int base = (int)(lo - ci * kChunk); base < (int)(hi - ci * kChunk); base += VPC) {
      const int slot = base + warp * VPW + vi;
      const bool valid = slot < (int)(hi - ci * kChunk);
      float o[32];
      decode_lane<D, B, OUTL>(p.c, rec, slot, valid, lut, pre, o);
      if (valid) {
        float4* dst = reinterpret_cast<float4*>(dst_g + (ci * kChunk + slot - p.first_vec) * p.dst_vs + lg * 32);
#pragma unroll
        for (int k = 0; k < 8; ++k) dst[k] = make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
      }
    }
  }
}

template <int D, int B, bool OUTL>
static cudaError_t dec_launch(const DecodeParams& p, int grid, cudaStream_t s) {
  decode_kernel<D, B, OUTL><<<grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

#define TQ_CASE(D_, B_)                                                        \
  case D_ * 100 + B_ * 10 + 0: return dec_launch<D_, B_, false>(p, grid, s);   \
  case D_ * 100 + B_ * 10 + 1: return dec_launch<D_, B_, true>(p, grid, s);

cudaError_t launch_decode(const DecodeParams& p, int grid, cudaStream_t s) {
  switch (p.c.d * 100 + p.c.bits * 10 + (p.c.has_outl ? 1 : 0)) {
    TQ_CASE(64, 1) TQ_CASE(64, 2) TQ_CASE(64, 3) TQ_CASE(64, 4)
    TQ_CASE(128, 1) TQ_CASE(128, 2) TQ_CASE(128, 3) TQ_CASE(128, 4)
    TQ_CASE(256, 1) TQ_CASE(256, 2) TQ_CASE(256, 3) TQ_CASE(256, 4)
    TQ_CASE(512, 1) TQ_CASE(512, 2) TQ_CASE(512, 3) TQ_CASE(512, 4)
    default: return cudaErrorInvalidValue;
  }
}
#undef TQ_CASE

}  // namespace tq
