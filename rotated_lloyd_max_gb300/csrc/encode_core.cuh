// The CUDA-core encoder's device code, used by the eviction kernels
// (evict.cu; tq_encode runs the tensor-core encoders of encode_mma.cuh):
// encode bf16 head vectors into 128-token records.
//
// Per vector ("v1.3 PPL on vLLM", M4 Phase A/B commits: rotate = H.D.x,
// per-row scale, Lloyd-Max argmin, outliers; larql PR #196 turbo-quant note:
// N(0,1) table scaled by 1/sqrt(d)):
//   n = ||x||;  w = H(s . x) (unnormalised FWHT);  y = w / (n sqrt(d));
//   code_j = #{k : y_j > t_k};  outlier_j = |y_j| > T/sqrt(d), value bf16(y_j).
// Thread mapping: a vector is spread over L = d/32 lanes, each holding 32
// consecutive coordinates (64 B of bf16, four 16-byte loads), so the first five
// FWHT stages run in registers and log2(L) stages via warp shuffles; the 32
// codes of a lane are exactly b 32-bit words of the packed row.
// A CTA (4 warps) owns one record at a time and walks its 128 slots in passes
// of 4*32/L vectors; with outliers, each pass is followed by a CTA-wide prefix
// sum so that entries land in (slot, index) order.
#pragma once

#include "tq_common.cuh"
#include "tq_params.h"

#include <algorithm>

namespace tq {

template <int D, int B, bool OUTL>
struct Enc {
  static constexpr int L = D / 32;       // lanes per vector
  static constexpr int VPW = 32 / L;     // vectors per warp pass
  static constexpr int VPC = 4 * VPW;    // vectors per CTA pass
  static constexpr int HALF = 1 << (B - 1);
  static constexpr int NPOS = HALF - 1;  // boundaries strictly above zero
  static constexpr int RB = D * B / 8;   // packed row bytes
};

struct EncSmem {
  int cnt[kChunk];
  int off[kChunk];
  int running;
};

// Per-thread constants of the encoder: the signs of the lane's 32
// coordinates as XOR masks on packed bf16 pairs (bits 15 and 31), and the
// positive decision boundaries.
template <int D, int B, bool OUTL>
struct EncLane {
  using E = Enc<D, B, OUTL>;
  int lane, warp, lg, vi;
  uint32_t smask[16];
  float tpos[E::NPOS > 0 ? E::NPOS : 1];
  __device__ __forceinline__ explicit EncLane(const CodecDev& c) {
    lane = threadIdx.x & 31;
    warp = threadIdx.x >> 5;
    lg = lane % E::L;
    vi = lane / E::L;
    const uint32_t sb = c.signs[lg];
#pragma unroll
    for (int k = 0; k < 16; ++k) smask[k] = (((sb >> (2 * k)) & 1u) << 15) | (((sb >> (2 * k + 1)) & 1u) << 31);
#pragma unroll
    for (int k = 0; k < E::NPOS; ++k) tpos[k] = c.boundaries[E::HALF + k];
  }
};

// The 16-point transform over the lane index of a d-512 vector (16 lanes x 32
// coordinates) through shared memory instead of 128 shuffles per lane: the
// lanes write their rows, lane l' takes coordinate pair (2 l', 2 l' + 1) of
// all 16 rows, applies the butterflies in registers and writes the pair back,
// and every lane reads its row again.  Rows are padded to 36 floats (row
// writes and pair reads both at the minimum number of wavefronts); the
// buffer holds the warp's two vectors.
constexpr int kTRow = 36, kTVec = 16 * kTRow + 4;
__device__ __forceinline__ void fwht16_lanes_smem(float (&x)[32], float* tb, int lane) {
  float* base = tb + (lane >> 4) * kTVec;
  float* row = base + (lane & 15) * kTRow;
  const int pc = 2 * (lane & 15);
#pragma unroll
  for (int k = 0; k < 8; ++k)
    *reinterpret_cast<float4*>(row + 4 * k) = make_float4(x[4 * k], x[4 * k + 1], x[4 * k + 2], x[4 * k + 3]);
  __syncwarp();
  float2 y[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) y[i] = *reinterpret_cast<const float2*>(base + i * kTRow + pc);
#pragma unroll
  for (int m = 1; m < 16; m <<= 1)
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (!(i & m)) {
        const float2 a = y[i], b = y[i | m];
        y[i] = add2(a, b);
        y[i | m] = fma2(b, f2(-1.f, -1.f), a);
      }
#pragma unroll
  for (int i = 0; i < 16; ++i) *reinterpret_cast<float2*>(base + i * kTRow + pc) = y[i];
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float4 v = *reinterpret_cast<const float4*>(row + 4 * k);
    x[4 * k] = v.x;
    x[4 * k + 1] = v.y;
    x[4 * k + 2] = v.z;
    x[4 * k + 3] = v.w;
  }
  __syncwarp();  // the buffer is written again for the warp's next vectors
}

// The lane's 32 bf16 coordinates of a vector (zeros for an invalid slot).
__device__ __forceinline__ void enc_load(const uint16_t* rowp, bool valid, uint4 (&w)[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) w[k] = make_uint4(0u, 0u, 0u, 0u);
  if (valid) {
    const uint4* src = reinterpret_cast<const uint4*>(rowp);
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = __ldg(src + k);
  }
}

// Encode one vector spread over the L lanes of a group: norm, FWHT, codes,
// packed store, and (OUTL) the outlier mask and the lane's unnormalised
// transform values x with inv = 1/(n sqrt(d)), so that y = x * inv.
//
// The decisions compare the unnormalised transform w_j against the
// boundaries scaled by sigma = n sqrt(d) (y_j > t_k  <=>  w_j > t_k sigma):
// the two forms differ only within about one f32 ulp of a boundary.  A code
// is the mirror of the count of positive boundaries below |w_j|:
// HALF + cnt for w_j > 0, HALF - 1 - cnt otherwise (w = 0 gives HALF - 1,
// the code of y = 0).
// With a scale mode other than the norm, the stored f32 is the mode's scale
// (vector_scale) from ||chat||^2 and <chat, y>, chat_j = cent[code_j] or, at
// an outlier coordinate, the stored bf16 value.
template <int D, int B, bool OUTL, bool SCALE>
__device__ __forceinline__ void enc_vector(const CodecDev& c, const EncLane<D, B, OUTL>& ln,
                                           const float2* cells, float* tb, const uint4 (&w)[4], bool valid,
                                           uint8_t* rec, int slot, float (&x)[32], float& inv, uint32_t& omask,
                                           const float* cent) {
  using E = Enc<D, B, OUTL>;
  {
    const uint32_t* ww = reinterpret_cast<const uint32_t*>(w);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint32_t v = ww[k] ^ ln.smask[k];
      x[2 * k] = __uint_as_float(v << 16);
      x[2 * k + 1] = __uint_as_float(v & 0xFFFF0000u);
    }
  }
  // ||x||^2 by a pairwise tree (squares of bf16 values are exact in f32)
  float2 sq[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float2 a = f2(x[4 * k], x[4 * k + 1]), b2 = f2(x[4 * k + 2], x[4 * k + 3]);
    sq[k] = fma2(a, a, mul2(b2, b2));
  }
#pragma unroll
  for (int h = 4; h; h >>= 1)
#pragma unroll
    for (int k = 0; k < h; ++k) sq[k] = add2(sq[k], sq[k + h]);
  float ss = sq[0].x + sq[0].y;
#pragma unroll
  for (int m = 1; m < E::L; m <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
  const float n = sqrtf(ss);
  const float sigma = n * c.sqrt_d;
  inv = n > 0.f ? 1.0f / sigma : 0.f;
  float T[E::NPOS > 0 ? E::NPOS : 1];
#pragma unroll
  for (int k = 0; k < E::NPOS; ++k) T[k] = ln.tpos[k] * sigma;
  const float Tout = OUTL ? c.thr_out * sigma : 0.f;

  fwht_regs<32>(x);
  if constexpr (D == 512) {
    fwht16_lanes_smem(x, tb, ln.lane);
  } else {
    fwht_lanes<32>(x, ln.lane, E::L);
  }

  uint32_t wd[B];
#pragma unroll
  for (int q = 0; q < B; ++q) wd[q] = 0u;
  omask = 0u;
  const float zscale = n > 0.f ? kCellScale / sigma : 0.f;  // z = 128 y
  float cc = 0.f, cx = 0.f;  // scale modes: the lane's parts of ||chat||^2 and <chat, x>
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    const float aw = fabsf(x[r]);
    uint32_t code;
    if constexpr (B >= 3) {  // decision cells (shared table)
      const float z = x[r] * zscale;
      const uint32_t ci = __float_as_uint(z + 8388736.0f) & 0x1FFu;  // round(z) + 128 (2^23 + 128 magic)
      code = cell_count(cells, ci) + (__float_as_uint(cell_boundary(cells, ci) - z) >> 31);  // + (z > boundary)
    } else {
      uint32_t msum = 0u;  // -(number of positive boundaries below |w|)
#pragma unroll
      for (int k = 0; k < E::NPOS; ++k) msum += mask_gt(aw, T[k]);
      code = ((uint32_t)E::HALF - msum) ^ (mask_le(x[r], 0.f) & ((1u << B) - 1u));
    }
    const int bit = r * B;
    wd[bit >> 5] += code << (bit & 31);
    if ((bit & 31) + B > 32) wd[(bit >> 5) + 1] += code >> (32 - (bit & 31));
    if (OUTL) omask |= mask_gt(aw, Tout) & (1u << r);
    if constexpr (SCALE) {
      float cj = cent[code & ((1u << B) - 1u)];
      if (OUTL && ((omask >> r) & 1u)) cj = bf16_to_f32(f32_to_bf16_rne(x[r] * inv));
      cc = fmaf(cj, cj, cc);
      cx = fmaf(cj, x[r], cx);
    }
  }
  float stored = n;
  if constexpr (SCALE) {
#pragma unroll
    for (int m = 1; m < E::L; m <<= 1) {
      cc += __shfl_xor_sync(0xffffffffu, cc, m);
      cx += __shfl_xor_sync(0xffffffffu, cx, m);
    }
    stored = vector_scale(c.scale_mode, n, cc, cx * inv);
  }
  if (valid) {
    uint8_t* dstrow = rec + (size_t)slot * E::RB + ln.lg * 4 * B;
    if constexpr (B == 4) {
      *reinterpret_cast<uint4*>(dstrow) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
    } else if constexpr (B == 2) {
      *reinterpret_cast<uint2*>(dstrow) = make_uint2(wd[0], wd[1]);
    } else {
#pragma unroll
      for (int q = 0; q < B; ++q) reinterpret_cast<uint32_t*>(dstrow)[q] = wd[q];
    }
    if (ln.lg == 0) reinterpret_cast<float*>(rec + c.off_norm)[slot] = stored;
  } else {
    omask = 0u;
  }
}

// Outlier entries of one pass, in (slot, index) order: per-vector counts, a
// CTA prefix sum over the pass (continuing the record's running total), then
// each lane writes its entries.  All 128 threads must call it.
template <int D, int B>
__device__ __forceinline__ void enc_outliers(const CodecDev& c, const EncLane<D, B, true>& ln,
                                             const float (&x)[32], float inv, uint32_t omask, bool valid,
                                             uint8_t* rec, int slot, int pslot, EncSmem* sm) {
  using E = Enc<D, B, true>;
  const int lane = ln.lane, lg = ln.lg;
  const int lc = __popc(omask);
  int incl = lc;
#pragma unroll
  for (int m = 1; m < E::L; m <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, m, E::L);
    if (lg >= m) incl += o;
  }
  const int excl = incl - lc;  // entries in lanes before this one
  const int vtot = __shfl_sync(0xffffffffu, incl, E::L - 1, E::L);
  const int nslot = min(vtot, 255);
  if (lg == 0) sm->cnt[pslot] = valid ? nslot : 0;
  __syncthreads();
  if (ln.warp == 0) {
    int run = sm->running;
    for (int k0 = 0; k0 < E::VPC; k0 += 32) {
      const int v = (k0 + lane < E::VPC) ? sm->cnt[k0 + lane] : 0;
      int inc = v;
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, inc, m);
        if (lane >= m) inc += o;
      }
      if (k0 + lane < E::VPC) sm->off[k0 + lane] = run + inc - v;
      run += __shfl_sync(0xffffffffu, inc, 31);
    }
    __syncwarp();
    if (lane == 0) sm->running = run;
  }
  __syncthreads();
  if (valid) {
    const int off = sm->off[pslot];
    const int stored = max(0, min(nslot, c.cap - off));
    uint32_t* ent = reinterpret_cast<uint32_t*>(rec + c.off_entries);
    int k = excl;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      if ((omask >> r) & 1u) {
        if (k < stored) {
          const uint32_t idx = (uint32_t)(lg * 32 + r);
          const uint32_t v = f32_to_bf16_rne(x[r] * inv);
          ent[off + k] = idx | (v << 16);
        }
        ++k;
      }
    }
    if (lg == 0) rec[c.off_count + slot] = (uint8_t)stored;
  }
  // the next pass rewrites cnt[] only before its first barrier and off[] only
  // after it, so no barrier is needed here
}

// Encode slots [s_begin, s_end) of the record at `rec`, one pass of VPC
// vectors at a time with the next pass's loads in flight; row(slot) gives the
// bf16 source of a slot.  Must be called by all 128 threads of the CTA.
template <int D, int B, bool OUTL, bool SCALE, class RowFn>
__device__ __forceinline__ void encode_record(const CodecDev& c, const float2* cells, const float* cent, float* tb,
                                              RowFn row, uint8_t* rec, int s_begin, int s_end, EncSmem* sm) {
  using E = Enc<D, B, OUTL>;
  const EncLane<D, B, OUTL> ln(c);
  if (OUTL && threadIdx.x == 0) sm->running = 0;
  if (OUTL) __syncthreads();
  const int pslot = ln.warp * E::VPW + ln.vi;  // slot index within a pass
  uint4 wn[4];
  enc_load(row(s_begin + pslot) + ln.lg * 32, s_begin + pslot < s_end, wn);
  for (int base = s_begin; base < s_end; base += E::VPC) {
    const int slot = base + pslot;
    const bool valid = slot < s_end;
    uint4 w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = wn[k];
    const int nslot = slot + E::VPC;
    enc_load(row(nslot) + ln.lg * 32, nslot < s_end, wn);
    float x[32];
    float inv;
    uint32_t omask;
    enc_vector<D, B, OUTL, SCALE>(c, ln, cells, tb, w, valid, rec, slot, x, inv, omask, cent);
    if constexpr (OUTL) enc_outliers<D, B>(c, ln, x, inv, omask, valid, rec, slot, pslot, sm);
  }
}


#define TQ_DISPATCH_DBO(FN, D_, B_, O_, ...)                                      \
  do {                                                                           \
    switch (D_ * 100 + B_ * 10 + (O_ ? 1 : 0)) {                                 \
      case 6410: return FN<64, 1, false>(__VA_ARGS__);                           \
      case 6411: return FN<64, 1, true>(__VA_ARGS__);                            \
      case 6420: return FN<64, 2, false>(__VA_ARGS__);                           \
      case 6421: return FN<64, 2, true>(__VA_ARGS__);                            \
      case 6430: return FN<64, 3, false>(__VA_ARGS__);                           \
      case 6431: return FN<64, 3, true>(__VA_ARGS__);                            \
      case 6440: return FN<64, 4, false>(__VA_ARGS__);                           \
      case 6441: return FN<64, 4, true>(__VA_ARGS__);                            \
      case 12810: return FN<128, 1, false>(__VA_ARGS__);                         \
      case 12811: return FN<128, 1, true>(__VA_ARGS__);                          \
      case 12820: return FN<128, 2, false>(__VA_ARGS__);                         \
      case 12821: return FN<128, 2, true>(__VA_ARGS__);                          \
      case 12830: return FN<128, 3, false>(__VA_ARGS__);                         \
      case 12831: return FN<128, 3, true>(__VA_ARGS__);                          \
      case 12840: return FN<128, 4, false>(__VA_ARGS__);                         \
      case 12841: return FN<128, 4, true>(__VA_ARGS__);                          \
      case 25610: return FN<256, 1, false>(__VA_ARGS__);                         \
      case 25611: return FN<256, 1, true>(__VA_ARGS__);                          \
      case 25620: return FN<256, 2, false>(__VA_ARGS__);                         \
      case 25621: return FN<256, 2, true>(__VA_ARGS__);                          \
      case 25630: return FN<256, 3, false>(__VA_ARGS__);                         \
      case 25631: return FN<256, 3, true>(__VA_ARGS__);                          \
      case 25640: return FN<256, 4, false>(__VA_ARGS__);                         \
      case 25641: return FN<256, 4, true>(__VA_ARGS__);                          \
      case 51210: return FN<512, 1, false>(__VA_ARGS__);                         \
      case 51211: return FN<512, 1, true>(__VA_ARGS__);                          \
      case 51220: return FN<512, 2, false>(__VA_ARGS__);                         \
      case 51221: return FN<512, 2, true>(__VA_ARGS__);                          \
      case 51230: return FN<512, 3, false>(__VA_ARGS__);                         \
      case 51231: return FN<512, 3, true>(__VA_ARGS__);                          \
      case 51240: return FN<512, 4, false>(__VA_ARGS__);                         \
      case 51241: return FN<512, 4, true>(__VA_ARGS__);                          \
      default: return cudaErrorInvalidValue;                                     \
    }                                                                            \
  } while (0)

}  // namespace tq
