// Gaussian Lloyd-Max table and SplitMix64 sign diagonal, on the device.
//
// One warp; lane k owns centroid k.  The Lloyd iteration for N(0,1)
// ("centroids_gaussian(bits)" in the M4 commits of "v1.3 PPL on vLLM";
// one N(0,1) table per bit width scaled by 1/sqrt(d) per the larql PR #196
// turbo-quant note) alternates
//   t_k = (c_k + c_{k+1}) / 2,
//   c_k = (pdf(t_{k-1}) - pdf(t_k)) / P(t_{k-1} < X <= t_k)
// in fp64 until no centroid moves by more than 1e-14.  Cell masses on the
// positive side are differences of upper tails, on the negative side of the
// distribution function, so mirrored cells evaluate the same expression and
// the table comes out exactly symmetric.
#include "tq_common.cuh"
#include "tq_params.h"

namespace tq {

__device__ __forceinline__ double npdf(double x) {
  return isinf(x) ? 0.0 : exp(-0.5 * x * x) * 0.39894228040143267794;  // 1/sqrt(2 pi)
}
__device__ __forceinline__ double ncdf(double x) { return 0.5 * erfc(-x * 0.70710678118654752440); }
__device__ __forceinline__ double nsf(double x) { return 0.5 * erfc(x * 0.70710678118654752440); }
__device__ __forceinline__ double xpdf(double x) { return isinf(x) ? 0.0 : x * npdf(x); }
__device__ __forceinline__ double cell(double a, double b) {
  return a >= 0.0 ? nsf(a) - nsf(b) : ncdf(b) - ncdf(a);
}
__device__ __forceinline__ double warp_max_d(double v) {
#pragma unroll
  for (int m = 16; m; m >>= 1) v = fmax(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int m = 16; m; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

__global__ void __launch_bounds__(32) codebook_kernel(int bits, int d, uint64_t seed,
                                                      CodebookOut* out) {
  const int k = threadIdx.x;
  const int K = 1 << bits;
  const bool own = k < K;
  double c = own ? (k - 0.5 * (K - 1)) * (4.0 / K) : 0.0;
  double a = 0.0, b = 0.0;
  int it = 0;
  for (it = 1; it <= 100000; ++it) {
    double cn = __shfl_down_sync(0xffffffffu, c, 1);
    double t = 0.5 * (c + cn);
    double tp = __shfl_up_sync(0xffffffffu, t, 1);
    a = (k == 0) ? -INFINITY : tp;
    b = (k == K - 1) ? INFINITY : t;
    double nc = own ? (npdf(a) - npdf(b)) / cell(a, b) : 0.0;
    double moved = warp_max_d(own ? fabs(nc - c) : 0.0);
    c = nc;
    if (moved < 1e-14) break;
  }
  // final boundaries from the final centroids, and the distortion
  {
    double cn = __shfl_down_sync(0xffffffffu, c, 1);
    double t = 0.5 * (c + cn);
    double tp = __shfl_up_sync(0xffffffffu, t, 1);
    a = (k == 0) ? -INFINITY : tp;
    b = (k == K - 1) ? INFINITY : t;
  }
  double D = 0.0;
  if (own) {
    double P = cell(a, b);
    double m2 = P - (xpdf(b) - xpdf(a));
    double m1 = npdf(a) - npdf(b);
    D = m2 - 2.0 * c * m1 + c * c * P;
  }
  D = warp_sum_d(D);
  // f32 table for head dim d, and f32 midpoints of the f32 centroids
  const float c32 = (float)(c / sqrt((double)d));
  const float c32n = __shfl_down_sync(0xffffffffu, c32, 1);
  if (own) out->c[k] = c32;
  if (k + 1 < K) out->t[k] = (float)(0.5 * ((double)c32 + (double)c32n));
  // sign diagonal: s_j = -1 iff the top bit of SplitMix64 output j is set
  for (int w = 0; w < d / 32; ++w) {
    const bool neg = (splitmix64_at(seed, (uint64_t)(w * 32 + k)) >> 63) != 0;
    const uint32_t bitsw = __ballot_sync(0xffffffffu, neg);
    if (k == 0) out->signs[w] = bitsw;
  }
  if (k == 0) {
    out->mse = D;
    out->iters = it;
  }
}

cudaError_t launch_codebook(int bits, int d, uint64_t seed, void* scratch, cudaStream_t s) {
  codebook_kernel<<<1, 32, 0, s>>>(bits, d, seed, (CodebookOut*)scratch);
  return cudaGetLastError();
}

}  // namespace tq
