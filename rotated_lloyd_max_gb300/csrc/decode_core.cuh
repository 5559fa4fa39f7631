// Decode of record slots back to f32 head vectors ("v1.3 PPL on vLLM", M5
// commit: dequantise through the centroid table, replace outlier coordinates
// by their stored values, inverse WHT, rescale by the stored scale):
//   xhat = n * s . H(yhat) / sqrt(d).
// Shared by the decode kernel (decode.cu) and the deep rollback (rollback.cu).
// Thread mapping as in the encoders: L = d/32 lanes per vector, 32
// consecutive coordinates per lane, in-register + shuffle FWHT stages.
#pragma once

#include "tq_common.cuh"
#include "tq_params.h"

namespace tq {

// Adding and subtracting 1.5 * 2^9 rounds an f32 of magnitude below 2^9 to
// the nearest multiple of 2^-14.
constexpr float kSplitMagic = 768.0f;

// Exclusive prefix of a record's outlier counts (pre[slot], pre[128] = total),
// by warp 0 of the CTA; the caller synchronises before reading it.
__device__ __forceinline__ void outlier_prefix(const uint8_t* rec, const CodecDev& c, int* pre) {
  if ((threadIdx.x >> 5) == 0) {
    const int lane = threadIdx.x & 31;
    int run = 0;
#pragma unroll
    for (int k0 = 0; k0 < kChunk; k0 += 32) {
      const int v = rec[c.off_count + k0 + lane];
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
}

// The lane's 32 decoded coordinates (32 lg .. 32 lg + 31) of slot `slot` of
// the record at `rec`, signs and scale applied.  All L lanes of the vector
// call it (the transform's lane stages shuffle), valid or not; an invalid
// slot reads nothing.  lut: the codec's centroids; pre: outlier_prefix.
template <int D, int B, bool OUTL>
__device__ __forceinline__ void decode_lane(const CodecDev& c, const uint8_t* rec, int slot, bool valid,
                                            const float* lut, const int* pre, float (&o)[32]) {
  constexpr int L = D / 32, RB = D * B / 8;
  const int lane = threadIdx.x & 31, lg = lane % L;
  const uint32_t sbits = c.signs[lg];
  float x[32];
  uint32_t w[B];
#pragma unroll
  for (int q = 0; q < B; ++q) w[q] = 0u;
  float n = 0.f;
  if (valid) {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(rec + (size_t)slot * RB + lg * 4 * B);
#pragma unroll
    for (int q = 0; q < B; ++q) w[q] = src[q];
    n = reinterpret_cast<const float*>(rec + c.off_norm)[slot];
  }
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    const int bit = r * B;
    uint32_t code = w[bit >> 5] >> (bit & 31);
    if ((bit & 31) + B > 32) code |= w[(bit >> 5) + 1] << (32 - (bit & 31));
    x[r] = lut[code & ((1u << B) - 1u)];
  }
  if (OUTL && valid) {
    const int e0 = pre[slot], e1 = min(e0 + rec[c.off_count + slot], c.cap);
    const uint32_t* ent = reinterpret_cast<const uint32_t*>(rec + c.off_entries);
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
  // n * (H(hi) + H(lo)) / sqrt(d) rounded once: f = n / sqrt(d) is carried
  // as fh + fl (fl: the product's rounding error plus n times the error of
  // the f32 constant 1/sqrt(d)), and the small terms fh * H(lo) and
  // fl * H(hi) enter the last fused multiply-add of fh * H(hi).
  const float fh = n * c.inv_sqrt_d;
  const float fl = fmaf(n, c.inv_sqrt_d, -fh) + n * c.inv_sqrt_d_lo;
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    const float v = fmaf(fh, x[r], fmaf(fh, lo[r], fl * x[r]));
    o[r] = ((sbits >> r) & 1u) ? -v : v;
  }
}

}  // namespace tq
