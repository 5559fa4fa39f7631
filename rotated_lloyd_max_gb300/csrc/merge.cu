// a10: merge of the split-K partials and the single inverse transform.
//
// Each split left (m_s, l_s, acc_s) in the log2 domain.  With M = max m_s and
// w_s = 2^(m_s - M):  out = [ s_v . H(sum_{compressed s} w_s acc_s)/sqrt(d)
//                              + sum_{dense s} w_s acc_s ] / sum_s w_s l_s.
// One warp per (layer, batch, query head); a lane owns d/32 consecutive
// coordinates, so the inverse FWHT is in-register stages plus five shuffle
// stages.  An empty context (every l_s = 0) writes a zero row.
#include "tq_common.cuh"
#include "tq_params.h"

namespace tq {

template <int D>
__global__ void __launch_bounds__(kThreads) merge_kernel(const __grid_constant__ MergeParams p) {
  constexpr int R = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= p.rows) return;
  const float* ml = p.ws_ml + row * p.S * 2;
  const float* acc = p.ws_acc + row * p.S * D;
  float* out = p.out + row * D + lane * R;
  float M = -INFINITY;
  for (int s = lane; s < p.S; s += 32)
    if (ml[2 * s + 1] > 0.f) M = fmaxf(M, ml[2 * s]);
  M = warp_max(M);
  if (M == -INFINITY) {
#pragma unroll
    for (int r = 0; r < R; ++r) out[r] = 0.f;
    return;
  }
  float W = 0.f;
  for (int s = lane; s < p.S; s += 32)
    if (ml[2 * s + 1] > 0.f) W += ml[2 * s + 1] * exp2f(ml[2 * s] - M);
  W = warp_sum(W);
  float ar[R], at[R];
#pragma unroll
  for (int r = 0; r < R; ++r) ar[r] = at[r] = 0.f;
  for (int s = 0; s < p.S; ++s) {
    const float ls = ml[2 * s + 1];
    if (!(ls > 0.f)) continue;
    const float w = exp2f(ml[2 * s] - M);
    const float* a = acc + (int64_t)s * D + lane * R;
    float x[R];
#pragma unroll
    for (int r = 0; r < R; r += 2) {
      const float2 v = *reinterpret_cast<const float2*>(a + r);
      x[r] = v.x;
      x[r + 1] = v.y;
    }
    if (s < p.Sc) {
#pragma unroll
      for (int r = 0; r < R; ++r) ar[r] = fmaf(w, x[r], ar[r]);
    } else {
#pragma unroll
      for (int r = 0; r < R; ++r) at[r] = fmaf(w, x[r], at[r]);
    }
  }
  if (p.Sc > 0) {
    fwht_regs<R>(ar);
    fwht_lanes<R>(ar, lane, 32);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int j = lane * R + r;
      const float f = ((p.vsign[j >> 5] >> (j & 31)) & 1u) ? -p.inv_sqrt_d : p.inv_sqrt_d;
      ar[r] *= f;
    }
  }
  const float invW = 1.0f / W;
#pragma unroll
  for (int r = 0; r < R; r += 2)
    *reinterpret_cast<float2*>(out + r) = make_float2((ar[r] + at[r]) * invW, (ar[r + 1] + at[r + 1]) * invW);
}

cudaError_t launch_merge(const MergeParams& p, int D, cudaStream_t s) {
  const int grid = (p.rows + 3) / 4;
  switch (D) {
    case 64: merge_kernel<64><<<grid, kThreads, 0, s>>>(p); break;
    case 128: merge_kernel<128><<<grid, kThreads, 0, s>>>(p); break;
    case 256: merge_kernel<256><<<grid, kThreads, 0, s>>>(p); break;
    case 512: merge_kernel<512><<<grid, kThreads, 0, s>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_attn_d64(const AttnParams& p, int GT, dim3 grid, cudaStream_t s);
cudaError_t launch_attn_d128(const AttnParams& p, int GT, dim3 grid, cudaStream_t s);
cudaError_t launch_attn_d256(const AttnParams& p, int GT, dim3 grid, cudaStream_t s);
cudaError_t launch_attn_d512(const AttnParams& p, int GT, dim3 grid, cudaStream_t s);

cudaError_t launch_attn(const AttnParams& p, int D, int GT, dim3 grid, cudaStream_t s) {
  switch (D) {
    case 64: return launch_attn_d64(p, GT, grid, s);
    case 128: return launch_attn_d128(p, GT, grid, s);
    case 256: return launch_attn_d256(p, GT, grid, s);
    case 512: return launch_attn_d512(p, GT, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tq
