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
  // One CTA per (layer, batch, query head).  Split weights first (warp 0),
  // then every thread sums its coordinates over all splits with independent
  // loads, then warp 0 applies the inverse transform to the compressed part.
  constexpr int R = D / 32;
  __shared__ float w_s[1024];
  __shared__ float acc_c[D];
  __shared__ float acc_t[D];
  __shared__ float s_W;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const float* ml = p.ws_ml + row * p.S * 2;
  const float* acc = p.ws_acc + row * p.S * D;
  float* out = p.out + row * D;
  if (warp == 0) {
    float M = -INFINITY;
    for (int s = lane; s < p.S; s += 32)
      if (ml[2 * s + 1] > 0.f) M = fmaxf(M, ml[2 * s]);
    M = warp_max(M);
    float W = 0.f;
    for (int s = lane; s < p.S; s += 32) {
      const float ls = ml[2 * s + 1];
      const float w = (ls > 0.f) ? exp2f(ml[2 * s] - M) : 0.f;
      w_s[s] = w;
      W += w * ls;
    }
    W = warp_sum(W);
    if (lane == 0) s_W = W;
  }
  __syncthreads();
  const float W = s_W;
  for (int j = tid; j < D; j += kThreads) {
    float c0 = 0.f, c1 = 0.f, t0 = 0.f, t1 = 0.f;
    int s = 0;
    for (; s + 1 < p.Sc; s += 2) {
      const float w0 = w_s[s], w1 = w_s[s + 1];
      const float a0 = w0 > 0.f ? acc[(int64_t)s * D + j] : 0.f;
      const float a1 = w1 > 0.f ? acc[(int64_t)(s + 1) * D + j] : 0.f;
      c0 = fmaf(w0, a0, c0);
      c1 = fmaf(w1, a1, c1);
    }
    for (; s < p.Sc; ++s) {
      const float w0 = w_s[s];
      c0 = fmaf(w0, w0 > 0.f ? acc[(int64_t)s * D + j] : 0.f, c0);
    }
    for (; s + 1 < p.S; s += 2) {
      const float w0 = w_s[s], w1 = w_s[s + 1];
      const float a0 = w0 > 0.f ? acc[(int64_t)s * D + j] : 0.f;
      const float a1 = w1 > 0.f ? acc[(int64_t)(s + 1) * D + j] : 0.f;
      t0 = fmaf(w0, a0, t0);
      t1 = fmaf(w1, a1, t1);
    }
    for (; s < p.S; ++s) {
      const float w0 = w_s[s];
      t0 = fmaf(w0, w0 > 0.f ? acc[(int64_t)s * D + j] : 0.f, t0);
    }
    acc_c[j] = c0 + c1;
    acc_t[j] = t0 + t1;
  }
  __syncthreads();
  if (warp != 0) return;
  if (!(W > 0.f)) {  // empty context: zero row
    for (int j = lane; j < D; j += 32) out[j] = 0.f;
    return;
  }
  float ar[R];
#pragma unroll
  for (int r = 0; r < R; ++r) ar[r] = acc_c[lane * R + r];
  if (p.Sc > 0) {
    fwht_regs<R>(ar);
    fwht_lanes<R>(ar, lane, 32);
  }
  const float invW = 1.0f / W;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int j = lane * R + r;
    const float f = ((p.vsign[j >> 5] >> (j & 31)) & 1u) ? -p.inv_sqrt_d : p.inv_sqrt_d;
    const float x = p.Sc > 0 ? ar[r] * f : 0.f;
    out[j] = (x + acc_t[j]) * invW;
  }
}

cudaError_t launch_merge(const MergeParams& p, int D, cudaStream_t s) {
  const int grid = p.rows;
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

cudaError_t launch_attn_rec_d64(const AttnParams& p, int GT, dim3 grid, cudaStream_t s);
cudaError_t launch_attn_rec_d128(const AttnParams& p, int GT, dim3 grid, cudaStream_t s);

cudaError_t launch_attn_rec(const AttnParams& p, int D, int GT, dim3 grid, cudaStream_t s) {
  switch (D) {
    case 64: return launch_attn_rec_d64(p, GT, grid, s);
    case 128: return launch_attn_rec_d128(p, GT, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

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
