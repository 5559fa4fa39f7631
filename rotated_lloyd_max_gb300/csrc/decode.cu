// Decode records back to f32 head vectors ("v1.3 PPL on vLLM", M5 commit:
// dequantise through the centroid table, replace outlier coordinates by their
// stored values, inverse WHT, rescale by the norm):
//   xhat = n * s . H(yhat) / sqrt(d).
// Same thread mapping as the encoder: L = d/32 lanes per vector, 32
// consecutive coordinates per lane, in-register + shuffle FWHT stages.
#include "tq_common.cuh"
#include "tq_params.h"

namespace tq {

// Adding and subtracting 1.5 * 2^9 rounds an f32 of magnitude below 2^9 to
// the nearest multiple of 2^-14.
constexpr float kSplitMagic = 768.0f;

template <int D, int B, bool OUTL>
__global__ void __launch_bounds__(kThreads) decode_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int L = D / 32, VPW = 32 / L, VPC = 4 * VPW, RB = D * B / 8;
  __shared__ float lut[16];
  __shared__ int pre[kChunk + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int lg = lane % L, vi = lane / L;
  if (threadIdx.x < 16) lut[threadIdx.x] = p.c.centroids[threadIdx.x & ((1 << B) - 1)];
  const uint32_t sbits = p.c.signs[lg];
  const float scale = p.c.inv_sqrt_d;
  const int64_t n_tasks = p.n_groups * p.chunks_per_group;
  for (int64_t task = blockIdx.x; task < n_tasks; task += gridDim.x) {
    const int64_t g = task / p.chunks_per_group;
    const int64_t ci = p.first_chunk + task % p.chunks_per_group;
    const int64_t lo = max(p.first_vec, ci * kChunk), hi = min(p.first_vec + p.n_vec, (ci + 1) * kChunk);
    const uint8_t* rec = p.src + g * p.src_gs + ci * (int64_t)p.c.rec_bytes;
    float* dst_g = p.dst + g * p.dst_gs;
    __syncthreads();  // lut ready; pre[] of the previous task consumed
    if (OUTL && warp == 0) {
      int run = 0;
      for (int k0 = 0; k0 < kChunk; k0 += 32) {
        const int v = rec[p.c.off_count + k0 + lane];
        int inc = v;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
          int o = __shfl_up_sync(0xffffffffu, inc, m);
          if (lane >= m) inc += o;
        }
        pre[k0 + lane] = run + inc - v;
        run += __shfl_sync(0xffffffffu, inc, 31);
      }
      if (lane == 0) pre[kChunk] = run;
    }
    if (OUTL) __syncthreads();
    for (int base = (int)(lo - ci * kChunk); base < (int)(hi - ci * kChunk); base += VPC) {
      const int slot = base + warp * VPW + vi;
      const bool valid = slot < (int)(hi - ci * kChunk);
      float x[32];
      uint32_t w[B];
#pragma unroll
      for (int q = 0; q < B; ++q) w[q] = 0u;
      float n = 0.f;
      if (valid) {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(rec + (size_t)slot * RB + lg * 4 * B);
#pragma unroll
        for (int q = 0; q < B; ++q) w[q] = src[q];
        n = reinterpret_cast<const float*>(rec + p.c.off_norm)[slot];
      }
#pragma unroll
      for (int r = 0; r < 32; ++r) {
        const int bit = r * B;
        uint32_t code = w[bit >> 5] >> (bit & 31);
        if ((bit & 31) + B > 32) code |= w[(bit >> 5) + 1] << (32 - (bit & 31));
        x[r] = lut[code & ((1u << B) - 1u)];
      }
      if (OUTL && valid) {
        const int e0 = pre[slot], e1 = min(e0 + rec[p.c.off_count + slot], p.c.cap);
        const uint32_t* ent = reinterpret_cast<const uint32_t*>(rec + p.c.off_entries);
        for (int e = e0; e < e1; ++e) {
          const uint32_t v = ent[e];
          const int idx = (int)(v & 0xFFFFu);
          if ((idx >> 5) == lg) {
            const float val = bf16_to_f32((uint16_t)(v >> 16));
#pragma unroll
            for (int r = 0; r < 32; ++r) x[r] = (r == (idx & 31)) ? val : x[r];
          }
        }
      }
      // Split transform: yhat = hi + lo with hi on the 2^-14 grid (|yhat| <= 1,
      // so every partial sum of at most 512 hi values is an integer multiple of
      // 2^-14 below 2^9 and exact in f32) and lo = yhat - hi exact; H(hi) is
      // exact and H(lo), at most 2^-15 d, carries f32 rounding only relative to
      // its own small size.
      float lo[32];
#pragma unroll
      for (int r = 0; r < 32; ++r) {
        const float h = (x[r] + kSplitMagic) - kSplitMagic;
        lo[r] = x[r] - h;
        x[r] = h;
      }
      fwht_regs<32>(x);
      fwht_lanes<32>(x, lane, L);
      fwht_regs<32>(lo);
      fwht_lanes<32>(lo, lane, L);
      if (valid) {
        // n * (H(hi) + H(lo)) / sqrt(d) rounded once: f = n / sqrt(d) is carried
        // as fh + fl (fl: the product's rounding error plus n times the error
        // of the f32 constant 1/sqrt(d)), and the small terms fh * H(lo) and
        // fl * H(hi) enter the last fused multiply-add of fh * H(hi).
        const float fh = n * scale;
        const float fl = fmaf(n, scale, -fh) + n * p.c.inv_sqrt_d_lo;
        float4* dst = reinterpret_cast<float4*>(dst_g + (ci * kChunk + slot - p.first_vec) * p.dst_vs + lg * 32);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          float o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = 4 * k + e;
            const float v = fmaf(fh, x[r], fmaf(fh, lo[r], fl * x[r]));
            o[e] = ((sbits >> r) & 1u) ? -v : v;
          }
          dst[k] = make_float4(o[0], o[1], o[2], o[3]);
        }
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
