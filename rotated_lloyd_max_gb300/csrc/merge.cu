// Merge of the split-K partials and the single inverse transform.
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
  // One CTA per (layer, batch, query head).  Warp 0 turns the splits' (m, l)
  // into weights; then warp w sums splits w, w+4, ... with a lane holding d/32
  // consecutive coordinates (several vector loads in flight), the four warps'
  // sums meet in shared memory, and warp 0 applies the inverse transform.
  constexpr int R = D / 32;
  __shared__ float w_s[1024];
  __shared__ __align__(16) float part[2][4][D];
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
  float c[R], t[R];
#pragma unroll
  for (int r = 0; r < R; ++r) c[r] = t[r] = 0.f;
  auto add_split = [&](int s, float (&dst)[R]) {
    const float w = w_s[s];
    if (!(w > 0.f)) return;
    const float* a = acc + (int64_t)s * D + lane * R;
#pragma unroll
    for (int r = 0; r < R; r += 2) {
      const float2 v = *reinterpret_cast<const float2*>(a + r);
      dst[r] = fmaf(w, v.x, dst[r]);
      dst[r + 1] = fmaf(w, v.y, dst[r + 1]);
    }
  };
#pragma unroll 4
  for (int s = warp; s < p.Sc; s += 4) add_split(s, c);
#pragma unroll 4
  for (int s = p.Sc + ((warp - p.Sc) & 3); s < p.S; s += 4) add_split(s, t);
#pragma unroll
  for (int r = 0; r < R; ++r) {
    part[0][warp][lane * R + r] = c[r];
    part[1][warp][lane * R + r] = t[r];
  }
  __syncthreads();
  if (warp != 0) return;
  if (p.status && *reinterpret_cast<const volatile int*>(p.status) != 0) {  // failed launch: NaN row
    for (int j = lane; j < D; j += 32) out[j] = __int_as_float(0x7fc00000);
    return;
  }
  if (!(W > 0.f)) {  // empty context: zero row
    for (int j = lane; j < D; j += 32) out[j] = 0.f;
    return;
  }
  float ar[R], at[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int j = lane * R + r;
    ar[r] = (part[0][0][j] + part[0][1][j]) + (part[0][2][j] + part[0][3][j]);
    at[r] = (part[1][0][j] + part[1][1][j]) + (part[1][2][j] + part[1][3][j]);
  }
  if (p.Sc > 0) {
    fwht_regs<R>(ar);
    fwht_lanes<R>(ar, lane, 32);
  }
  const float invW = 1.0f / W;
#pragma unroll
  for (int r = 0; r < R; r += 2) {
    const int j = lane * R + r;
    const float f0 = ((p.vsign[j >> 5] >> (j & 31)) & 1u) ? -p.inv_sqrt_d : p.inv_sqrt_d;
    const float f1 = ((p.vsign[(j + 1) >> 5] >> ((j + 1) & 31)) & 1u) ? -p.inv_sqrt_d : p.inv_sqrt_d;
    const float x0 = p.Sc > 0 ? ar[r] * f0 : 0.f, x1 = p.Sc > 0 ? ar[r + 1] * f1 : 0.f;
    *reinterpret_cast<float2*>(out + j) = make_float2((x0 + at[r]) * invW, (x1 + at[r + 1]) * invW);
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

#define TQ_MMA_DECL(D_, K_) cudaError_t launch_attn_mma_d##D_##_k##K_(const AttnParams& p, dim3 grid, cudaStream_t s);
TQ_MMA_DECL(64, 1)
TQ_MMA_DECL(64, 2)
TQ_MMA_DECL(64, 3)
TQ_MMA_DECL(64, 4)
TQ_MMA_DECL(128, 1)
TQ_MMA_DECL(128, 2)
TQ_MMA_DECL(128, 3)
TQ_MMA_DECL(128, 4)
#undef TQ_MMA_DECL

cudaError_t launch_attn_mma(const AttnParams& p, int D, dim3 grid, cudaStream_t s) {
  switch (D * 10 + p.kb) {
    case 641: return launch_attn_mma_d64_k1(p, grid, s);
    case 642: return launch_attn_mma_d64_k2(p, grid, s);
    case 643: return launch_attn_mma_d64_k3(p, grid, s);
    case 644: return launch_attn_mma_d64_k4(p, grid, s);
    case 1281: return launch_attn_mma_d128_k1(p, grid, s);
    case 1282: return launch_attn_mma_d128_k2(p, grid, s);
    case 1283: return launch_attn_mma_d128_k3(p, grid, s);
    case 1284: return launch_attn_mma_d128_k4(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_attn_mma512_k1(const AttnParams& p, dim3 grid, cudaStream_t s);
cudaError_t launch_attn_mma512_k2(const AttnParams& p, dim3 grid, cudaStream_t s);
cudaError_t launch_attn_mma512_k3(const AttnParams& p, dim3 grid, cudaStream_t s);
cudaError_t launch_attn_mma512_k4(const AttnParams& p, dim3 grid, cudaStream_t s);

cudaError_t launch_attn_umma512_k1(const AttnParams& p, dim3 grid, cudaStream_t s);
cudaError_t launch_attn_umma512_k2(const AttnParams& p, dim3 grid, cudaStream_t s);
cudaError_t launch_attn_umma512_k3(const AttnParams& p, dim3 grid, cudaStream_t s);
cudaError_t launch_attn_umma512_k4(const AttnParams& p, dim3 grid, cudaStream_t s);

cudaError_t launch_attn_umma512(const AttnParams& p, dim3 grid, cudaStream_t s) {
  switch (p.kb) {
    case 1: return launch_attn_umma512_k1(p, grid, s);
    case 2: return launch_attn_umma512_k2(p, grid, s);
    case 3: return launch_attn_umma512_k3(p, grid, s);
    case 4: return launch_attn_umma512_k4(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_attn_mma512(const AttnParams& p, dim3 grid, cudaStream_t s) {
  switch (p.kb) {
    case 1: return launch_attn_mma512_k1(p, grid, s);
    case 2: return launch_attn_mma512_k2(p, grid, s);
    case 3: return launch_attn_mma512_k3(p, grid, s);
    case 4: return launch_attn_mma512_k4(p, grid, s);
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
