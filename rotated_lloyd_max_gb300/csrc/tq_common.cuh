// Device-side helpers shared by the sm_103a kernels of the codec and the
// decode attention (bf16 unpacking, packed-f32 math, Walsh-Hadamard stages,
// SplitMix64, cp.async staging).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/tq.h"
#include "tq_params.h"

namespace tq {

constexpr int kChunk = TQ_CHUNK;
constexpr int kThreads = 128;  // every kernel here runs 4-warp CTAs

// ---------------------------------------------------------------- bf16 / f32
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// Round-to-nearest-even f32 -> bf16 bits (finite inputs).
__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

// Packed pair helpers (sm_100+ f32x2 FMA / add).
__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

// ------------------------------------------------------------ Walsh-Hadamard
// In-register butterflies over the index bits of an array of R values
// (Sylvester order, unnormalised): stage H pairs (i, i + H) for i & H == 0.
// Written as compile-time recursion so every index is a constant and the
// array stays in registers.
template <int R, int H>
__device__ __forceinline__ void fwht_stage(float (&x)[R]) {
  if constexpr (H == 1) {
#pragma unroll
    for (int i = 0; i < R; i += 2) {
      const float a = x[i], b = x[i + 1];
      x[i] = a + b;
      x[i + 1] = a - b;
    }
  } else {
#pragma unroll
    for (int i = 0; i < R; i += 2 * H) {
#pragma unroll
      for (int j = 0; j < H; j += 2) {
        const float2 a = f2(x[i + j], x[i + j + 1]), b = f2(x[i + j + H], x[i + j + H + 1]);
        const float2 s = add2(a, b);
        const float2 d = fma2(b, f2(-1.f, -1.f), a);
        x[i + j] = s.x;
        x[i + j + 1] = s.y;
        x[i + j + H] = d.x;
        x[i + j + H + 1] = d.y;
      }
    }
  }
  if constexpr (2 * H < R) fwht_stage<R, 2 * H>(x);
}

template <int R>
__device__ __forceinline__ void fwht_regs(float (&x)[R]) {
  if constexpr (R > 1) fwht_stage<R, 1>(x);
}

// Butterflies across lanes: lane bit `m` (1, 2, 4, ...) carries an index bit
// above the in-register ones; the lane with the bit set keeps a - b.
template <int R>
__device__ __forceinline__ void fwht_lanes(float (&x)[R], int lane, int lanes_per_vec) {
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    if (m >= lanes_per_vec) break;
    const float sg = (lane & m) ? -1.f : 1.f;
    const float2 sg2 = f2(sg, sg);
#pragma unroll
    for (int r = 0; r < R; r += 2) {
      float p0 = __shfl_xor_sync(0xffffffffu, x[r], m);
      float p1 = __shfl_xor_sync(0xffffffffu, x[r + 1], m);
      float2 v = fma2(f2(x[r], x[r + 1]), sg2, f2(p0, p1));
      x[r] = v.x;
      x[r + 1] = v.y;
    }
  }
}

// 0xFFFFFFFF if a > b, else 0 (an f32 compare that yields an integer mask).
__device__ __forceinline__ uint32_t mask_gt(float a, float b) {
  uint32_t r;
  asm("set.gt.u32.f32 %0, %1, %2;" : "=r"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ uint32_t mask_le(float a, float b) {
  uint32_t r;
  asm("set.le.u32.f32 %0, %1, %2;" : "=r"(r) : "f"(a), "f"(b));
  return r;
}

// Byte offset of record c of stream (b, h) within its layer's record array:
// contiguous [B][Hkv][rec_cap] records, or, with a block table, block
// table[b][c] of a pool of rec_cap blocks of Hkv records each.  A table entry
// outside the pool is clamped into it (a wrong table reads a wrong record,
// never out of bounds).
__device__ __forceinline__ int64_t rec_offset(const int32_t* table, int table_stride, int rec_cap, int Hkv, int b,
                                              int h, int c, int rec_bytes) {
  if (table) {
    const int blk = min(max(__ldg(table + (int64_t)b * table_stride + c), 0), rec_cap - 1);
    return ((int64_t)blk * Hkv + h) * rec_bytes;
  }
  return (((int64_t)b * Hkv + h) * rec_cap + c) * rec_bytes;
}

// n / f.d for a FastDiv (tq_params.h)
__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv& f) {
  const uint32_t t = __umulhi(n, f.m);
  return (t + ((n - t) >> f.s1)) >> f.s2;
}

// ------------------------------------------------------------- SplitMix64
__device__ __forceinline__ uint64_t splitmix64_at(uint64_t seed, uint64_t k) {
  // output k (0-based) of SplitMix64 seeded with `seed`
  uint64_t z = seed + (k + 1) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// ------------------------------------------------------------- cp.async
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// Cooperative async copy of `bytes` (multiple of 16) by the whole CTA.
__device__ __forceinline__ void cta_copy_async(void* smem, const void* gmem, int bytes) {
  char* s = (char*)smem;
  const char* g = (const char*)gmem;
  for (int off = threadIdx.x * 16; off < bytes; off += kThreads * 16) cp_async16(s + off, g + off);
}

// ------------------------------------------------------------- reductions
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

// Code r (0..31) of a 32-code run packed LSB-first into B words, with a
// run-time index.
template <int B>
__device__ __forceinline__ uint32_t code_at(const uint32_t (&w)[B], int r) {
  const int bit = r * B;
  const int wi = bit >> 5, sh = bit & 31;
  uint32_t lo = w[0], hi = B > 1 ? w[1] : 0u;
#pragma unroll
  for (int k = 1; k < B; ++k)
    if (wi == k) { lo = w[k]; hi = (k + 1 < B) ? w[k + 1] : 0u; }
  uint64_t v = ((uint64_t)hi << 32) | lo;
  return (uint32_t)(v >> sh) & ((1u << B) - 1u);
}

// Decision cells (the d-128 encoder at b >= 2, the CUDA-core encoder at b >= 3): with z = y * 128 (y the normalised rotated value, |y| <= 1)
// and i = round(z) + 128, cell i covers z in [i - 128.5, i - 127.5) and
// holds (count of boundaries below the cell, the boundary inside it x 128 or
// +huge); boundaries are >= 1.4/128 apart for b <= 4 at every head dim up to
// 512 (the closest pair, around 0 at b = 4, is 0.258/sqrt(d) apart), so a cell holds
// at most one.  |y| <= 1 keeps i in 0..256.  code = count + (z > boundary): the same code as
// #{k : y > t_k} except within a couple of f32 ulp of a boundary.
constexpr int kCells = 512;  // index masked to 9 bits: every value reads a cell (257.. = top cell's law)
constexpr float kCellScale = 128.f;
// z + 2^16 + 128.5 rounds to the 2^-7 grid, so that bits 7..15 of the sum are
// floor of the rounded z + 128.5: the SHIFTED cell index, already times 128
constexpr float kCellMagicShifted = 65664.5f;

// SPLIT: the table's two planes (boundaries as f32, counts as bytes) in the
// storage of kCells float2 (the CUDA-core encoder, whose crowded lookups
// spread over more banks as 4- and 1-byte loads); otherwise float2 entries
// (boundary, count as int bits), one 8-byte load per lookup.
// SHIFTED: cells moved down by 1/256, [i - 128.5 - 2^-8, i - 127.5 - 2^-8),
// the cells of the index floor(z + 128.5) taken on the 2^-7 grid of an add
// to 2^16 (kCellMagicShifted), whose bits 7..15 are the index itself.
template <bool SPLIT = false, bool SHIFTED = false>
__device__ __forceinline__ void build_cells(const CodecDev& c, float2* cells) {
  const int nb = (1 << c.bits) - 1;
  constexpr float sh = SHIFTED ? 0.00390625f : 0.f;
  for (int i = threadIdx.x; i < kCells; i += kThreads) {
    const float lo = ((float)(i - 128) - 0.5f - sh) / kCellScale, hi = ((float)(i - 128) + 0.5f - sh) / kCellScale;
    int below = 0;
    float inside = 3.0e38f;
    for (int k = 0; k < nb; ++k) {
      const float t = c.boundaries[k];
      if (t < lo) ++below;
      else if (t < hi) inside = t * kCellScale;
    }
    const float bnd = inside;
    if constexpr (SPLIT) {
      float* bt = reinterpret_cast<float*>(cells);
      bt[i] = bnd;
      reinterpret_cast<uint8_t*>(bt + kCells)[i] = (uint8_t)below;
    } else {
      cells[i] = make_float2(bnd, __int_as_float(below));
    }
  }
}
// lookups in the SPLIT layout
__device__ __forceinline__ float cell_boundary(const float2* cells, uint32_t i) {
  return reinterpret_cast<const float*>(cells)[i];
}
__device__ __forceinline__ uint32_t cell_count(const float2* cells, uint32_t i) {
  return reinterpret_cast<const uint8_t*>(reinterpret_cast<const float*>(cells) + kCells)[i];
}

// Per-vector scale of a record's "norm" field (tq_scale_mode): n = ||x||,
// cc = ||chat||^2 and cy = <chat, y> of the dequantised rotated vector chat
// (turboquant_plus commit log, the EDEN-scale commits and their Appendix A
// note).  A zero vector stores 0.
__device__ __forceinline__ float vector_scale(int mode, float n, float cc, float cy) {
  if (!(n > 0.f)) return 0.f;
  if (mode == TQ_SCALE_MATCHED_NORM) return n / sqrtf(cc);
  if (mode == TQ_SCALE_INNER_PRODUCT) return n / cy;
  if (mode == TQ_SCALE_LEAST_SQUARES) return n * cy / cc;
  return n;
}

// Logit soft cap (arc PR #98, softcapping fix: cap * tanh(s / cap) on the
// scaled logit, before it is stored and before the running maximum) in the
// log2 domain of the attention kernels: with t = s * log2(e) and
// C = cap * log2(e), log2(e) * cap * tanh(s / cap) = C * tanh(t / C).  A
// masked slot (-inf) stays masked.  Callers test C > 0 (a launch-uniform
// branch) before calling.
__device__ __forceinline__ float soft_cap(float t, float C, float iC) {
  return t > -INFINITY ? C * tanhf(t * iC) : t;
}

}  // namespace tq
