// tq_encode's kernels: encode with the Hadamard transform on the tensor
// cores, at every head dim (128 first; the others below).
//
// Same codes as the CUDA-core encoder (n = ||x||; w = H(s . x), the
// unnormalised Sylvester transform; y = w / (n sqrt(d)); code_j = #{k : y_j > t_k},
// taken from a table of decision cells; outliers |y_j| > T / sqrt(d), value
// bf16(y_j)), computed as
// H128 = H8 (x) H16 over a split of the 7 index bits: a coordinate is
//   c = 32 t + 4 kb + 2 h + e      (t, kb, h, e: 2, 3, 1, 1 bits).
// Stage 1 applies the 16-point transform over the bits (e, h, t) of every
// block kb as one bf16 mma.sync (16 vectors x 16 coordinates x 16 outputs;
// bf16 inputs and +-1 entries are exact, products are exact, sums are f32);
// stage 2 applies the 8-point transform over kb in registers.  With
//   fragment column 2t'+e+8h  <->  input coordinate 32 t' + 4 kb + 2 h + e,
//   output column 2t''+e' of n-tile nt <-> output coordinate 32 t'' + 4 J + 2 nt + e',
// lane (g, t) loads its vectors' coordinates 32 t .. 32 t + 31 with four
// 16-byte loads straight into the A fragments, and after stage 2 holds the
// same 32 coordinates of the output: its 32 codes are b words of the packed
// row, as in the CUDA-core encoder.  A warp encodes 16 vectors at a time
// (rows g and g + 8 of the MMA tile).
//
// Head dims 256 and 512 (R = d/128 quarters of 128 coordinates): with the
// Sylvester ordering H_d = H_R (x) H128 over the top log2 R index bits, so the
// 16 rows of an MMA tile hold quarters rather than whole vectors -- d 256: rows
// g and g + 8 are the halves of vector g (8 vectors per tile); d 512: rows g
// and g + 8 are quarters (g >> 2) and 2 + (g >> 2) of vector g & 3 (4 vectors
// per tile).  Each quarter is transformed as above, then the quarter
// butterflies follow: between the lane's two rows, and at d 512 between lanes
// g and g ^ 4 (lane ^ 16) by shuffles.  A lane ends with 64 outputs of one
// vector (two runs of 32 coordinates), as many as at d 128.
// Head dim 64: a 128-coordinate row holds two vectors (coordinate bit 6, the
// high bit of t, picks the vector), and the 16-point stage leaves that bit
// alone (its matrix is H8 (x) I2 over (e, h, t & 1) and t >> 1), so a tile
// carries 32 vectors and lane (g, t) ends with 32 outputs of vector
// (row, t >> 1); a vector's lanes are pairs (t, t ^ 1) rather than quads.
//
// A CTA of 16 warps (12 at d 256/512, whose lanes also hold the signs of two
// quarters) owns an SM.  Its decision-cell table is replicated 16 times, copy
// j in bank pair j, and lane l reads copy l % 16: the lookups of a half-warp
// (one shared-memory wavefront) never conflict, whatever cells the 16
// coordinates fall in.
#pragma once

#include <cuda_bf16.h>

#include <algorithm>

#include "tq_common.cuh"
#include "tq_params.h"

namespace tq {

__device__ __forceinline__ void mma_bf16_e(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// bf16 +-1 pair of the permuted H16: entry (input in4, output out4) is
// (-1)^popcount(in4 & out4), in4 = e | h<<1 | t'<<2, out4 = e' | nt<<1 | t''<<2.
// (BLOCK, head dim 64) zero where bit 3 of in4 and out4 (t' >> 1, t'' >> 1:
// the vector of the row) differ.
template <bool BLOCK = false>
__device__ __forceinline__ uint32_t h16_pair(int in4a, int in4b, int out4) {
  const int m = BLOCK ? 7 : 15;  // the vector bit never enters the sign
  uint32_t lo = (__popc(in4a & out4 & m) & 1) ? 0xBF80u : 0x3F80u;
  uint32_t hi = (__popc(in4b & out4 & m) & 1) ? 0xBF80u : 0x3F80u;
  if (BLOCK && ((in4a ^ out4) & 8)) lo = 0u;
  if (BLOCK && ((in4b ^ out4) & 8)) hi = 0u;
  return lo | (hi << 16);
}

// Tile geometry of head dim D: R quarters per vector, VT vectors per 16-row
// tile, TPR tiles per 128-slot record; RB bytes per packed row.
template <int D, int B>
struct EncM {
  static constexpr int R = D >= 128 ? D / 128 : 1;
  static constexpr int VT = D == 64 ? 32 : 16 / R;
  static constexpr int TPR = kChunk / VT;
  static constexpr int RB = D * B / 8;
};

// The rows of tile `tile` a lane (g, t) works on: the slots of its vectors
// in rows g and g + 8 and the quarters of them it holds.
struct EncRows {
  int slot_a, slot_b, qa, qb;
};
template <int D>
__device__ __forceinline__ EncRows enc_rows(int tile, int g, int t) {
  if constexpr (D == 64) return {32 * tile + 2 * g + (t >> 1), 32 * tile + 16 + 2 * g + (t >> 1), 0, 0};
  else if constexpr (D == 128) return {16 * tile + g, 16 * tile + g + 8, 0, 0};
  else if constexpr (D == 256) return {8 * tile + g, 8 * tile + g, 0, 1};
  else return {4 * tile + (g & 3), 4 * tile + (g & 3), g >> 2, 2 + (g >> 2)};
}
// Element offset of a lane's 32 coordinates within its vector.
template <int D>
__device__ __forceinline__ int enc_col(int q, int t) { return D == 64 ? 32 * (t & 1) : 128 * q + 32 * t; }

// Lane state shared by the kernels: sign masks of the lane's 32 coordinates
// in each of its rows (XOR on packed bf16 pairs; one set at d 128, where both
// rows hold the same coordinates) and the H16 fragments.
template <int D, int B>
struct EncMLane {
  int lane, warp, g, t;
  uint32_t cell_lane;  // byte offset of this lane's copy within a replicated cell
  uint32_t smask[D <= 128 ? 1 : 2][16];
  uint32_t hb[2][2];  // [n-tile][b0, b1]
  __device__ __forceinline__ explicit EncMLane(const CodecDev& c) {
    lane = threadIdx.x & 31;
    warp = threadIdx.x >> 5;
    g = lane >> 2;
    t = lane & 3;
    cell_lane = (uint32_t)(lane & 15) * 8u;
    const EncRows rw = enc_rows<D>(0, g, t);
#pragma unroll
    for (int s = 0; s < (D <= 128 ? 1 : 2); ++s) {
      const uint32_t sb = c.signs[enc_col<D>(s ? rw.qb : rw.qa, t) / 32];
#pragma unroll
      for (int k = 0; k < 16; ++k)
        smask[s][k] = (((sb >> (2 * k)) & 1u) << 15) | (((sb >> (2 * k + 1)) & 1u) << 31);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int out4 = (g & 1) | (nt << 1) | ((g >> 1) << 2);
      hb[nt][0] = h16_pair<D == 64>(0 | (t << 2), 1 | (t << 2), out4);
      hb[nt][1] = h16_pair<D == 64>(2 | (t << 2), 3 | (t << 2), out4);
    }
  }
};

// cp.async staging of 16-row tiles: a lane copies its own 64 bytes of
// rows g and g + 8 and later reads back exactly those, so no other lane is
// involved; its 4 chunks sit at swizzled positions so that the 16-byte reads
// of a quarter-warp (g in {2q, 2q+1}, t in 0..3) hit 8 different bank groups.
struct EncTile {
  uint4 row[16][16];  // [tile row][16-byte chunk]
};
__device__ __forceinline__ int encm_chunk(int g, int t, int k) { return 4 * t + (k ^ (t >> 1) ^ ((g & 1) << 1)); }

__device__ __forceinline__ void encm_issue(EncTile& tile, int g, int t, const uint16_t* ra, bool va,
                                           const uint16_t* rb, bool vb) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (va) cp_async16(&tile.row[g][encm_chunk(g, t, k)], ra + 8 * k);
    if (vb) cp_async16(&tile.row[g + 8][encm_chunk(g, t, k)], rb + 8 * k);
  }
}

__device__ __forceinline__ void encm_read(const EncTile& tile, int r, int g, int t, bool valid,
                                          const uint32_t (&smask)[16], uint32_t (&w)[16]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint4 v = valid ? tile.row[r][encm_chunk(g, t, k)] : make_uint4(0u, 0u, 0u, 0u);
    w[4 * k] = v.x ^ smask[4 * k];
    w[4 * k + 1] = v.y ^ smask[4 * k + 1];
    w[4 * k + 2] = v.z ^ smask[4 * k + 2];
    w[4 * k + 3] = v.w ^ smask[4 * k + 3];
  }
}

// A predicated 4-byte global store (no branch around it).
__device__ __forceinline__ void st_global_if(bool p, uint32_t* dst, uint32_t v) {
  asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %0, 0;\n @q st.global.u32 [%1], %2;\n}\n" ::"r"((uint32_t)p),
               "l"(dst), "r"(v)
               : "memory");
}

// a * a + c with a bf16 operand (the low or the high half of w), rounded once
// to f32 (the square of a bf16 value is exact in f32)
__device__ __forceinline__ float sq_add_lo(uint32_t w, float c) {
  float d;
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n fma.rn.f32.bf16 %0, lo, lo, %2;\n}\n" : "=f"(d) : "r"(w), "f"(c));
  return d;
}
__device__ __forceinline__ float sq_add_hi(uint32_t w, float c) {
  float d;
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n fma.rn.f32.bf16 %0, hi, hi, %2;\n}\n" : "=f"(d) : "r"(w), "f"(c));
  return d;
}

__device__ __forceinline__ void st_global_u8_if(bool p, uint8_t* dst, uint32_t v) {
  asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %0, 0;\n @q st.global.u8 [%1], %2;\n}\n" ::"r"((uint32_t)p),
               "l"(dst), "r"(v)
               : "memory");
}

// Sum of squares of 32 bf16 coordinates (exact squares, pairwise f32 tree:
// pair k holds a^2 + b^2 of words 2k (a) and 2k + 1 (b), element by element).
__device__ __forceinline__ float encm_sq(const uint32_t (&w)[16]) {
  float2 sq[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    sq[k].x = sq_add_lo(w[2 * k], sq_add_lo(w[2 * k + 1], 0.f));
    sq[k].y = sq_add_hi(w[2 * k], sq_add_hi(w[2 * k + 1], 0.f));
  }
#pragma unroll
  for (int h = 4; h; h >>= 1)
#pragma unroll
    for (int k = 0; k < h; ++k) sq[k] = add2(sq[k], sq[k + h]);
  return sq[0].x + sq[0].y;
}

// The full transform of two vectors (rows g, g + 8): wa, wb hold the lane's
// loaded words; on return xa, xb hold the lane's 32 output coordinates.
template <int D, int B>
__device__ __forceinline__ void encm_transform(const EncMLane<D, B>& ln, const uint32_t (&wa)[16],
                                               const uint32_t (&wb)[16], float (&xa)[32], float (&xb)[32]) {
  float cc[8][2][4];
#pragma unroll
  for (int kb = 0; kb < 8; ++kb)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) cc[kb][nt][e] = 0.f;
      mma_bf16_e(cc[kb][nt], wa[2 * kb], wb[2 * kb], wa[2 * kb + 1], wb[2 * kb + 1], ln.hb[nt][0], ln.hb[nt][1]);
    }
  // 8-point transform over kb, on (element 0, 1) and (2, 3) pairs
#pragma unroll
  for (int m = 1; m < 8; m <<= 1)
#pragma unroll
    for (int kb = 0; kb < 8; ++kb)
      if (!(kb & m))
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const float2 a = f2(cc[kb][nt][e], cc[kb][nt][e + 1]);
            const float2 b = f2(cc[kb | m][nt][e], cc[kb | m][nt][e + 1]);
            const float2 s = add2(a, b);
            const float2 d = fma2(b, f2(-1.f, -1.f), a);
            cc[kb][nt][e] = s.x;
            cc[kb][nt][e + 1] = s.y;
            cc[kb | m][nt][e] = d.x;
            cc[kb | m][nt][e + 1] = d.y;
          }
#pragma unroll
  for (int J = 0; J < 8; ++J)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        xa[4 * J + 2 * nt + e] = cc[J][nt][e];
        xb[4 * J + 2 * nt + e] = cc[J][nt][2 + e];
      }
}

// warps per CTA at most (one CTA per SM): 16, or 12 at d 256/512 (two sets of
// sign masks per lane); small encodes run 6-warp CTAs so that two fit an SM
template <int D>
constexpr int enc_warps() { return D <= 128 ? 16 : 12; }
constexpr int kEncWarpsSmall = 6;
constexpr int kCellCopies = 16;

// Shared memory of both kernels: the replicated decision cells (cell i, copy
// j at float2 index 16 i + j), the centroids, then two tile buffers per warp
// (as many warps as the launch has).
struct EncMSmem {
  float2 cells[kCells * kCellCopies];
  float cent[32];
  EncTile tiles[1][2];  // [warps][2] in the launch's dynamic shared memory
};
constexpr int enc_smem_bytes(int warps) { return (int)(sizeof(EncMSmem) + (warps - 1) * 2 * sizeof(EncTile)); }

// Cell (i128 >> 7) & 511 as seen by a lane (its copy: bank pair lane % 16);
// i128 is the cell index times 128 in bits 7..15 (other bits ignored).
__device__ __forceinline__ float2 encm_cell(const unsigned char* cells, uint32_t i128, uint32_t cell_lane) {
  return *reinterpret_cast<const float2*>(cells + ((i128 & ((uint32_t)(kCells - 1) << 7)) | cell_lane));
}

// The table, built once per CTA: plain cells into a scratch tile first, then
// each cell copied 16 times.
__device__ __forceinline__ void encm_build(const CodecDev& c, EncMSmem& sm) {
  float2* plain = reinterpret_cast<float2*>(&sm.tiles[0][0]);
  static_assert(sizeof(EncTile) >= kCells * sizeof(float2), "scratch tile holds the plain table");
  if (threadIdx.x < kThreads) build_cells<false, true>(c, plain);
  if (threadIdx.x < 16) sm.cent[threadIdx.x] = c.centroids[threadIdx.x];
  __syncthreads();
  for (int i = threadIdx.x; i < kCells * kCellCopies; i += blockDim.x) sm.cells[i] = plain[i / kCellCopies];
  __syncthreads();
}

// Codes of the lane's 32 coordinates of one vector (x: unnormalised
// transform, scale = 128 / (n sqrt(d)) or 0 for a zero vector), packed
// LSB-first into B words; (OUTL) the outlier mask |y| > T / sqrt(d).
// (SCALE) the lane's parts of ||chat||^2 and <chat, x> over its coordinates,
// chat_j = cent[code_j] or, at an outlier coordinate, the stored bf16 value.
// (OUTL) also the lane's 32 values y = x * inv as bf16 into its chunks of a
// tile row (srow: its 4 chunks, swizzled by sw as in encm_chunk).
template <int B, bool OUTL, bool SCALE = false>
__device__ __forceinline__ void encm_quantize(const float (&x)[32], const unsigned char* cells, uint32_t cell_lane,
                                              float scale,
                                              float thr_out, uint32_t (&wd)[B], uint32_t& omask,
                                              const float* cent = nullptr, float* cc = nullptr,
                                              float* cx = nullptr, uint4* srow = nullptr, int sw = 0,
                                              float inv_y = 0.f) {
#pragma unroll
  for (int q = 0; q < B; ++q) wd[q] = 0u;
  omask = 0u;
  // the outlier test compares |x| against the threshold scaled once per
  // vector (|z| = |x| scale > T 128  <=>  |x| > T 128 / scale); a zero vector
  // (scale 0) has x = 0 and no outliers
  const float inv = scale > 0.f ? 1.0f / scale : 0.f;
  const float Tox = OUTL ? (scale > 0.f ? thr_out * kCellScale * inv : INFINITY) : 0.f;
  uint32_t yw[4];
#pragma unroll
  for (int r = 0; r < 32; r += 2) {
    if constexpr (OUTL) {
      const float2 yv = mul2(f2(x[r], x[r + 1]), f2(inv_y, inv_y));
      const __nv_bfloat162 h = __floats2bfloat162_rn(yv.x, yv.y);
      yw[(r >> 1) & 3] = *reinterpret_cast<const uint32_t*>(&h);
      if ((r & 7) == 6) srow[(r >> 3) ^ sw] = make_uint4(yw[0], yw[1], yw[2], yw[3]);
    }
    uint32_t code[2];
    if constexpr (B == 1) {
      // the one boundary is 0: code 1 for x > 0
#pragma unroll
      for (int k = 0; k < 2; ++k) code[k] = 1u - (mask_le(x[r + k], 0.f) & 1u);
    } else {
      const float2 z = mul2(f2(x[r], x[r + 1]), f2(scale, scale));
      const float2 u = add2(z, f2(kCellMagicShifted, kCellMagicShifted));  // the shifted cell index x 128
      const float2 e0 = encm_cell(cells, __float_as_uint(u.x), cell_lane);
      const float2 e1 = encm_cell(cells, __float_as_uint(u.y), cell_lane);
      // count below the cell + (z > the cell's boundary): the sign bit of boundary - z
      // (+0 when equal, so a tie takes the lower code)
      code[0] = (uint32_t)__float_as_int(e0.y) + (__float_as_uint(e0.x - z.x) >> 31);
      code[1] = (uint32_t)__float_as_int(e1.y) + (__float_as_uint(e1.x - z.y) >> 31);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int bit = (r + k) * B;
      wd[bit >> 5] += code[k] << (bit & 31);
      if ((bit & 31) + B > 32) wd[(bit >> 5) + 1] += code[k] >> (32 - (bit & 31));
      if (OUTL) omask += mask_gt(fabsf(x[r + k]), Tox) * (0u - (1u << (r + k)));  // distinct bits: + is |
      if constexpr (SCALE) {
        float cj = cent[code[k]];
        if (OUTL && ((omask >> (r + k)) & 1u)) cj = bf16_to_f32(f32_to_bf16_rne(x[r + k] * (scale * (1.f / kCellScale))));
        *cc = fmaf(cj, cj, *cc);
        *cx = fmaf(cj, x[r + k], *cx);
      }
    }
  }
}

template <int B>
__device__ __forceinline__ void encm_store_row(uint8_t* row, const uint32_t (&wd)[B]) {
  if constexpr (B == 4) {
    *reinterpret_cast<uint4*>(row) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
  } else if constexpr (B == 2) {
    *reinterpret_cast<uint2*>(row) = make_uint2(wd[0], wd[1]);
  } else {
#pragma unroll
    for (int q = 0; q < B; ++q) reinterpret_cast<uint32_t*>(row)[q] = wd[q];
  }
}

// (d 128) The stored scales of the vectors of a lane's two rows from the quad
// sums of ||chat||^2 and <chat, x> (z = 128 / (n sqrt(d)), so <chat, y> = <chat, x> z / 128).
__device__ __forceinline__ void encm_scales(int mode, float na, float nb, float za, float zb, float cca, float cxa,
                                            float ccb, float cxb, float& sa, float& sb) {
#pragma unroll
  for (int m = 1; m < 4; m <<= 1) {
    cca += __shfl_xor_sync(0xffffffffu, cca, m);
    cxa += __shfl_xor_sync(0xffffffffu, cxa, m);
    ccb += __shfl_xor_sync(0xffffffffu, ccb, m);
    cxb += __shfl_xor_sync(0xffffffffu, cxb, m);
  }
  sa = vector_scale(mode, na, cca, cxa * (za * (1.f / kCellScale)));
  sb = vector_scale(mode, nb, ccb, cxb * (zb * (1.f / kCellScale)));
}

// Norms of the lane's vectors: d 64 one per row and pair, d 128 one per row
// (quad sums), otherwise one
// per vector over its rows (quad sums, at d 512 also over lane ^ 16).  Every
// lane of a vector ends with the same value (f32 addition commutes).
template <int D, int R>
__device__ __forceinline__ void encm_norms(const uint32_t (&wa)[16], const uint32_t (&wb)[16], float& na,
                                           float& nb) {
  float sa = encm_sq(wa), sb = encm_sq(wb);
  if constexpr (R == 1) {
    sa += __shfl_xor_sync(0xffffffffu, sa, 1);
    sb += __shfl_xor_sync(0xffffffffu, sb, 1);
    if constexpr (D == 128) {  // at d 64 a vector's lanes are a pair
      sa += __shfl_xor_sync(0xffffffffu, sa, 2);
      sb += __shfl_xor_sync(0xffffffffu, sb, 2);
    }
    na = sqrtf(sa);
    nb = sqrtf(sb);
  } else {
    float s = sa + sb;
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    if constexpr (R == 4) s += __shfl_xor_sync(0xffffffffu, s, 16);
    na = nb = sqrtf(s);
  }
}

// The quarter butterflies of H_d = H_R (x) H128 (Sylvester order: quarter q
// = index bits 7 and up): xa, xb hold the H128 outputs of the lane's rows.
// d 256: rows = quarters 0, 1 -> (xa + xb, xa - xb).  d 512: rows = quarters
// (g >> 2), 2 + (g >> 2): the same over bit 8 in the lane, then over bit 7
// with lane ^ 16 (the lane of bit 7 = 0 adds its partner's value, the other
// subtracts its own from it).  The rows then hold the same quarters of the
// output.
template <int R>
__device__ __forceinline__ void encm_quarters(int g, float (&xa)[32], float (&xb)[32]) {
  if constexpr (R >= 2) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const float2 a = f2(xa[i], xa[i + 1]), b = f2(xb[i], xb[i + 1]);
      const float2 s = add2(a, b), d = fma2(b, f2(-1.f, -1.f), a);
      xa[i] = s.x;
      xa[i + 1] = s.y;
      xb[i] = d.x;
      xb[i + 1] = d.y;
    }
  }
  if constexpr (R == 4) {
    const float sg = (g >> 2) ? -1.f : 1.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float pa = __shfl_xor_sync(0xffffffffu, xa[i], 16);
      const float pb = __shfl_xor_sync(0xffffffffu, xb[i], 16);
      xa[i] = fmaf(sg, xa[i], pa);
      xb[i] = fmaf(sg, xb[i], pb);
    }
  }
}

// The stored scales (scale modes) from the lane's parts of ||chat||^2 and
// <chat, x> (z = 128 / (n sqrt(d)), so <chat, y> = <chat, x> z / 128): per
// row at d 128, per vector otherwise.
template <int D, int R>
__device__ __forceinline__ void encm_scales_r(int mode, float na, float nb, float za, float zb, float cca,
                                              float cxa, float ccb, float cxb, float& sa, float& sb) {
  if constexpr (D == 64) {  // pair sums
    cca += __shfl_xor_sync(0xffffffffu, cca, 1);
    cxa += __shfl_xor_sync(0xffffffffu, cxa, 1);
    ccb += __shfl_xor_sync(0xffffffffu, ccb, 1);
    cxb += __shfl_xor_sync(0xffffffffu, cxb, 1);
    sa = vector_scale(mode, na, cca, cxa * (za * (1.f / kCellScale)));
    sb = vector_scale(mode, nb, ccb, cxb * (zb * (1.f / kCellScale)));
  } else if constexpr (R == 1) {
    encm_scales(mode, na, nb, za, zb, cca, cxa, ccb, cxb, sa, sb);
  } else {
    float cc = cca + ccb, cx = cxa + cxb;
#pragma unroll
    for (int m = 1; m < 4; m <<= 1) {
      cc += __shfl_xor_sync(0xffffffffu, cc, m);
      cx += __shfl_xor_sync(0xffffffffu, cx, m);
    }
    if constexpr (R == 4) {
      cc += __shfl_xor_sync(0xffffffffu, cc, 16);
      cx += __shfl_xor_sync(0xffffffffu, cx, 16);
    }
    sa = sb = vector_scale(mode, na, cc, cx * (za * (1.f / kCellScale)));
  }
}

// Byte offset of a lane's 32 codes (coordinates enc_col ..) within a packed row.
template <int D, int B>
__device__ __forceinline__ int encm_run_bytes(int q, int t) { return enc_col<D>(q, t) / 8 * B; }

// Encode without outliers: every (group, record, tile) is a task of one warp;
// warps stride over the tasks with the next task's rows in flight (cp.async,
// two buffers per warp).
template <int D, int B, bool SCALE>
__global__ void __launch_bounds__(32 * enc_warps<D>(), 1) encode_mma_kernel(const __grid_constant__ EncodeParams p) {
  using E = EncM<D, B>;
  constexpr int R = E::R, TPR = E::TPR;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  EncMSmem& sm = *reinterpret_cast<EncMSmem*>(smem_raw);
  encm_build(p.c, sm);
  const unsigned char* cells = reinterpret_cast<const unsigned char*>(sm.cells);
  const float* cent = sm.cent;
  EncTile (*tiles)[2] = sm.tiles;
  const int W = blockDim.x >> 5;  // warps in this CTA
  const EncMLane<D, B> ln(p.c);
  const int64_t per_group = p.chunks_per_group * TPR;
  const int64_t n_tasks = p.n_groups * per_group;
  const int64_t v_end = p.first_vec + p.n_vec;
  struct Task {
    int64_t grp, chunk, ta, tb;
    EncRows rw;
    bool va, vb;
  };
  auto locate = [&](int64_t task) {
    Task k;
    int64_t r;
    if (p.small_tasks) {  // 32-bit multiply-shift division instead of a 64-bit divide
      const uint32_t rec = (uint32_t)task / (uint32_t)TPR, grp = fast_div(rec, p.cpg);
      k.grp = grp;
      r = (int64_t)((uint32_t)task - grp * (uint32_t)per_group);
    } else {
      k.grp = task / per_group;
      r = task % per_group;
    }
    k.chunk = p.first_chunk + r / TPR;
    k.rw = enc_rows<D>((int)(r % TPR), ln.g, ln.t);
    k.ta = k.chunk * kChunk + k.rw.slot_a;
    k.tb = k.chunk * kChunk + k.rw.slot_b;
    k.va = task < n_tasks && k.ta >= p.first_vec && k.ta < v_end;
    k.vb = task < n_tasks && k.tb >= p.first_vec && k.tb < v_end;
    return k;
  };
  auto issue = [&](const Task& k, int buf) {
    const uint16_t* src = p.src + k.grp * p.src_gs;
    encm_issue(tiles[ln.warp][buf], ln.g, ln.t,
               src + (k.va ? k.ta - p.first_vec : 0) * p.src_vs + enc_col<D>(k.rw.qa, ln.t), k.va,
               src + (k.vb ? k.tb - p.first_vec : 0) * p.src_vs + enc_col<D>(k.rw.qb, ln.t), k.vb);
    cp_async_commit();
  };
  const int64_t stride = (int64_t)gridDim.x * W;
  int64_t task = (int64_t)blockIdx.x * W + ln.warp;
  Task cur = locate(task);
  issue(cur, 0);
  for (int it = 0; task < n_tasks; task += stride, ++it) {
    const Task nxt = locate(task + stride);
    issue(nxt, (it + 1) & 1);
    cp_async_wait<1>();  // this lane's copies of the current tile are in
    uint32_t wa[16], wb[16];
    encm_read(tiles[ln.warp][it & 1], ln.g, ln.g, ln.t, cur.va, ln.smask[0], wa);
    encm_read(tiles[ln.warp][it & 1], ln.g + 8, ln.g, ln.t, cur.vb, ln.smask[R == 1 ? 0 : 1], wb);
    float na, nb;
    encm_norms<D, R>(wa, wb, na, nb);
    float xa[32], xb[32];
    encm_transform<D, B>(ln, wa, wb, xa, xb);
    encm_quarters<R>(ln.g, xa, xb);
    uint8_t* rec = p.dst + cur.grp * p.dst_gs + cur.chunk * (int64_t)p.c.rec_bytes;
    uint32_t wd[B], om;
    const float za = na > 0.f ? kCellScale / (na * p.c.sqrt_d) : 0.f;
    const float zb = nb > 0.f ? kCellScale / (nb * p.c.sqrt_d) : 0.f;
    float cca = 0.f, cxa = 0.f, ccb = 0.f, cxb = 0.f;
    encm_quantize<B, false, SCALE>(xa, cells, ln.cell_lane, za, 0.f, wd, om, cent, &cca, &cxa);
    if (cur.va) encm_store_row<B>(rec + (size_t)cur.rw.slot_a * E::RB + encm_run_bytes<D, B>(cur.rw.qa, ln.t), wd);
    encm_quantize<B, false, SCALE>(xb, cells, ln.cell_lane, zb, 0.f, wd, om, cent, &ccb, &cxb);
    if (cur.vb) encm_store_row<B>(rec + (size_t)cur.rw.slot_b * E::RB + encm_run_bytes<D, B>(cur.rw.qb, ln.t), wd);
    float sca = na, scb = nb;
    if constexpr (SCALE) encm_scales_r<D, R>(p.c.scale_mode, na, nb, za, zb, cca, cxa, ccb, cxb, sca, scb);
    if ((D == 64 ? (ln.t & 1) : ln.t) == 0) {  // one lane per vector writes its scale
      float* nrm = reinterpret_cast<float*>(rec + p.c.off_norm);
      if constexpr (R == 1) {
        if (cur.va) nrm[cur.rw.slot_a] = sca;
        if (cur.vb) nrm[cur.rw.slot_b] = scb;
      } else {
        if (cur.va && (R == 2 || ln.g < 4)) nrm[cur.rw.slot_a] = sca;
      }
    }
    cur = nxt;
  }
  cp_async_wait<0>();
}

// Encode with outliers: a warp owns a whole record and encodes its tiles in
// slot order (the next tile, of this record or the warp's next one, in
// flight through cp.async as in the kernel above).  Entries land in (slot,
// index) order without any CTA barrier: a row's lanes take their places by a
// prefix over the vector's lanes (a quad, a pair at d 64), a vector's rows
// (quarters) in coordinate order, a tile's
// vectors by a warp prefix, and a running warp-uniform offset carries the
// record's entry count from tile to tile.
template <int D, int B, bool SCALE>
__global__ void __launch_bounds__(32 * enc_warps<D>(), 1) encode_mma_outl_kernel(const __grid_constant__ EncodeParams p) {
  using E = EncM<D, B>;
  constexpr int R = E::R, TPR = E::TPR;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  EncMSmem& sm = *reinterpret_cast<EncMSmem*>(smem_raw);
  encm_build(p.c, sm);
  const unsigned char* cells = reinterpret_cast<const unsigned char*>(sm.cells);
  const float* cent = sm.cent;
  EncTile (*tiles)[2] = sm.tiles;
  const int W = blockDim.x >> 5;  // warps in this CTA
  const EncMLane<D, B> ln(p.c);
  const int64_t n_tasks = p.n_groups * p.chunks_per_group;
  const int64_t v_end = p.first_vec + p.n_vec;
  const int64_t warps = (int64_t)gridDim.x * W;
  // unit u of this warp: record task warp_id + (u / TPR) * warps, tile u % TPR
  struct Unit {
    int64_t task, grp, chunk, ta, tb;
    int tile;
    EncRows rw;
    bool va, vb;
  };
  const int64_t wid = (int64_t)blockIdx.x * W + ln.warp;
  auto locate = [&](int64_t u) {
    Unit k;
    k.task = wid + (u / TPR) * warps;
    k.tile = (int)(u % TPR);
    if (p.small_tasks) {  // 32-bit multiply-shift division instead of a 64-bit divide
      const uint32_t grp = fast_div((uint32_t)k.task, p.cpg);
      k.grp = grp;
      k.chunk = p.first_chunk + ((uint32_t)k.task - grp * (uint32_t)p.chunks_per_group);
    } else {
      k.grp = k.task / p.chunks_per_group;
      k.chunk = p.first_chunk + k.task % p.chunks_per_group;
    }
    k.rw = enc_rows<D>(k.tile, ln.g, ln.t);
    k.ta = k.chunk * kChunk + k.rw.slot_a;
    k.tb = k.chunk * kChunk + k.rw.slot_b;
    k.va = k.task < n_tasks && k.ta >= p.first_vec && k.ta < v_end;
    k.vb = k.task < n_tasks && k.tb >= p.first_vec && k.tb < v_end;
    return k;
  };
  auto issue = [&](const Unit& k, int buf) {
    const uint16_t* src = p.src + k.grp * p.src_gs;
    encm_issue(tiles[ln.warp][buf], ln.g, ln.t,
               src + (k.va ? k.ta - p.first_vec : 0) * p.src_vs + enc_col<D>(k.rw.qa, ln.t), k.va,
               src + (k.vb ? k.tb - p.first_vec : 0) * p.src_vs + enc_col<D>(k.rw.qb, ln.t), k.vb);
    cp_async_commit();
  };
  Unit cur = locate(0);
  issue(cur, 0);
  int run = 0;  // entries of the current record written so far (warp-uniform)
  for (int64_t u = 0; cur.task < n_tasks; ++u) {
    const Unit nxt = locate(u + 1);
    issue(nxt, (int)((u + 1) & 1));
    if (cur.tile == 0) run = 0;
    cp_async_wait<1>();  // this lane's copies of the current tile are in
    EncTile& tl = tiles[ln.warp][u & 1];
    uint8_t* rec = p.dst + cur.grp * p.dst_gs + cur.chunk * (int64_t)p.c.rec_bytes;
    const bool va = cur.va, vb = cur.vb;
    uint32_t wa[16], wb[16];
    encm_read(tl, ln.g, ln.g, ln.t, va, ln.smask[0], wa);
    encm_read(tl, ln.g + 8, ln.g, ln.t, vb, ln.smask[R == 1 ? 0 : 1], wb);
    float na, nb;
    encm_norms<D, R>(wa, wb, na, nb);
    float xa[32], xb[32];
    encm_transform<D, B>(ln, wa, wb, xa, xb);
    encm_quarters<R>(ln.g, xa, xb);
    uint32_t wd[B], oma, omb;
    const float za = na > 0.f ? kCellScale / (na * p.c.sqrt_d) : 0.f;
    const float zb = nb > 0.f ? kCellScale / (nb * p.c.sqrt_d) : 0.f;
    float cca = 0.f, cxa = 0.f, ccb = 0.f, cxb = 0.f;
    // the quantiser also keeps the lane's y values as bf16 (the stored
    // outlier value) in its own chunks of the tile buffer it has just read,
    // for the entry writes below
    const int sw = (ln.t >> 1) ^ ((ln.g & 1) << 1);
    encm_quantize<B, true, SCALE>(xa, cells, ln.cell_lane, za, p.c.thr_out, wd, oma, cent, &cca, &cxa,
                                  &tl.row[ln.g][4 * ln.t], sw, na > 0.f ? 1.0f / (na * p.c.sqrt_d) : 0.f);
    if (va) encm_store_row<B>(rec + (size_t)cur.rw.slot_a * E::RB + encm_run_bytes<D, B>(cur.rw.qa, ln.t), wd);
    if (!va) oma = 0u;
    encm_quantize<B, true, SCALE>(xb, cells, ln.cell_lane, zb, p.c.thr_out, wd, omb, cent, &ccb, &cxb,
                                  &tl.row[ln.g + 8][4 * ln.t], sw, nb > 0.f ? 1.0f / (nb * p.c.sqrt_d) : 0.f);
    if (vb) encm_store_row<B>(rec + (size_t)cur.rw.slot_b * E::RB + encm_run_bytes<D, B>(cur.rw.qb, ln.t), wd);
    if (!vb) omb = 0u;
    float sca = na, scb = nb;
    if constexpr (SCALE) encm_scales_r<D, R>(p.c.scale_mode, na, nb, za, zb, cca, cxa, ccb, cxb, sca, scb);
    if ((D == 64 ? (ln.t & 1) : ln.t) == 0) {  // one lane per vector writes its scale
      float* nrm = reinterpret_cast<float*>(rec + p.c.off_norm);
      if constexpr (R == 1) {
        if (va) nrm[cur.rw.slot_a] = sca;
        if (vb) nrm[cur.rw.slot_b] = scb;
      } else {
        if (va && (R == 2 || ln.g < 4)) nrm[cur.rw.slot_a] = sca;
      }
    }
    // entries before this lane within its row's vector (prefix over the
    // VL lanes of the vector: a quad, a pair at d 64), a in the low and b in
    // the high half-word (at most 128 per row)
    constexpr int VL = D == 64 ? 2 : 4;
    const int ca = __popc(oma), cb = __popc(omb);
    uint32_t qp = (uint32_t)ca | ((uint32_t)cb << 16);
#pragma unroll
    for (int m = 1; m < VL; m <<= 1) {
      const uint32_t o = __shfl_up_sync(0xffffffffu, qp, m, VL);
      if ((ln.t & (VL - 1)) >= m) qp += o;
    }
    const int ia = (int)(qp & 0xFFFFu), ib = (int)(qp >> 16);
    const uint32_t qs = __shfl_sync(0xffffffffu, qp, VL - 1, VL);
    const int nsa = (int)(qs & 0xFFFFu), nsb = (int)(qs >> 16);
    // record-list positions of the lane's first row-a and row-b entries and,
    // for the lane that writes it, a vector's stored count
    int pos_a, pos_b, cnt_a = 0, cnt_b = 0;
    if constexpr (R == 1) {
      // the tile's vectors in slot order (those of the a rows, then those of
      // the b rows): an inclusive prefix over the vectors' lane groups, whose
      // lanes all hold the group's sums
      uint32_t wp = qs;
#pragma unroll
      for (int m = VL; m < 32; m <<= 1) {
        const uint32_t o = __shfl_up_sync(0xffffffffu, wp, m);
        if (ln.lane >= m) wp += o;
      }
      const uint32_t tot = __shfl_sync(0xffffffffu, wp, 31);
      const int tot_a = (int)(tot & 0xFFFFu), tot_b = (int)(tot >> 16);
      const int off_a = run + (int)(wp & 0xFFFFu) - nsa, off_b = run + tot_a + (int)(wp >> 16) - nsb;
      run += tot_a + tot_b;
      pos_a = off_a + ia - ca;
      pos_b = off_b + ib - cb;
      cnt_a = max(0, min(nsa, p.c.cap - off_a));
      cnt_b = max(0, min(nsb, p.c.cap - off_b));
    } else if constexpr (R == 2) {
      // vector g: its first half's entries (row a), then its second half's
      const int vt = nsa + nsb;
      int wp = vt;
#pragma unroll
      for (int m = 4; m < 32; m <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, wp, m);
        if (ln.lane >= m) wp += o;
      }
      const int tot = __shfl_sync(0xffffffffu, wp, 31);
      const int off_v = run + wp - vt;
      run += tot;
      pos_a = off_v + ia - ca;
      pos_b = off_v + nsa + ib - cb;
      cnt_a = max(0, min(vt, p.c.cap - off_v));
    } else {
      // vector g & 3: quarters 0 and 2 in quad g & 3, 1 and 3 in quad (g & 3) + 4
      // (lane ^ 16), entries in quarter order
      const int pa = __shfl_xor_sync(0xffffffffu, nsa, 16), pb = __shfl_xor_sync(0xffffffffu, nsb, 16);
      const bool hi = ln.g >= 4;
      const int vt = nsa + nsb + pa + pb;
      int wp = vt;  // prefix over the tile's 4 vectors, in each half of the warp
#pragma unroll
      for (int m = 4; m < 16; m <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, wp, m);
        if ((ln.lane & 15) >= m) wp += o;
      }
      const int tot = __shfl_sync(0xffffffffu, wp, 15);
      const int off_v = run + wp - vt;
      run += tot;
      pos_a = off_v + (hi ? pa : 0) + ia - ca;
      pos_b = off_v + (hi ? pa + nsa + pb : nsa + pa) + ib - cb;
      cnt_a = max(0, min(vt, p.c.cap - off_v));
    }
    // entry writes: per row, a warp-uniform number of rounds (the most
    // entries a lane holds), in each of which every lane writes its next
    // entry, if it has one and it is within the capacity: predicated
    // stores, no divergent loop
    uint32_t* ent = reinterpret_cast<uint32_t*>(rec + p.c.off_entries);
    const uint32_t swz = (uint32_t)sw << 4;  // the chunk swizzle in bytes
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      const int c = v ? cb : ca;
      int pos = v ? pos_b : pos_a;
      uint32_t om = v ? omb : oma;
      const uint32_t idx0 = (uint32_t)enc_col<D>(v ? cur.rw.qb : cur.rw.qa, ln.t);
      // the lane's stashed values of this row: value j at byte (2 j) ^ swz of its 64 bytes
      const unsigned char* sv = reinterpret_cast<const unsigned char*>(&tl.row[v ? ln.g + 8 : ln.g][4 * ln.t]);
      const int rounds = (int)__reduce_max_sync(0xffffffffu, (unsigned)c);
      for (int i = 0; i < rounds; ++i) {
        const uint32_t r = (uint32_t)(__ffs(om) - 1) & 31u;  // a lane without entries left reads value 31, unused
        om &= om - 1;
        const uint32_t val = *reinterpret_cast<const uint16_t*>(sv + ((2u * r) ^ swz));
        st_global_if(i < c && pos < p.c.cap, ent + pos, (idx0 + r) | (val << 16));
        ++pos;
      }
    }
    if ((D == 64 ? (ln.t & 1) : ln.t) == 0) {  // one lane per vector writes its stored count
      if constexpr (R == 1) {
        st_global_u8_if(va, rec + p.c.off_count + cur.rw.slot_a, (uint32_t)cnt_a);
        st_global_u8_if(vb, rec + p.c.off_count + cur.rw.slot_b, (uint32_t)cnt_b);
      } else {
        st_global_u8_if(va && (R == 2 || ln.g < 4), rec + p.c.off_count + cur.rw.slot_a, (uint32_t)cnt_a);
      }
    }
    cur = nxt;
  }
  cp_async_wait<0>();
}

// `grid` is 8 CTAs per SM; these kernels run one CTA per SM of up to 16
// (d 128) or 12 warps (all of its registers and most of its shared memory),
// so one wave (grid / 8) of persistent CTAs, whose warps then prefetch their
// next task.  An encode of fewer than 4 tile tasks per such warp runs 6-warp
// CTAs instead (112 KB, two per SM), so that another encode on a concurrent
// stream (a small cache's K and V) shares the SMs rather than waiting for them
// (Qwen2-shaped encode phase: 27.5 us with 4-warp CTAs, 26.4 us with 6).
template <int D, int B, bool SCALE>
static cudaError_t encm_launch(const EncodeParams& p, int grid, cudaStream_t s) {
  using E = EncM<D, B>;
  constexpr int WMAX = enc_warps<D>();
  grid = std::max(1, grid / 8);
  const int64_t tiles = p.n_groups * p.chunks_per_group * E::TPR;
  const int W = tiles < 4LL * WMAX * grid ? kEncWarpsSmall : WMAX;
  const int smem = enc_smem_bytes(W);
  if (p.c.has_outl) {
    const int64_t tasks = (p.n_groups * p.chunks_per_group + W - 1) / W;  // a warp per record
    cudaError_t e = cudaFuncSetAttribute(encode_mma_outl_kernel<D, B, SCALE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, enc_smem_bytes(WMAX));
    if (e != cudaSuccess) return e;
    encode_mma_outl_kernel<D, B, SCALE><<<(int)std::min<int64_t>(tasks, grid), 32 * W, smem, s>>>(p);
  } else {
    const int64_t tasks = (tiles + W - 1) / W;
    cudaError_t e = cudaFuncSetAttribute(encode_mma_kernel<D, B, SCALE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         enc_smem_bytes(WMAX));
    if (e != cudaSuccess) return e;
    encode_mma_kernel<D, B, SCALE><<<(int)std::min<int64_t>(tasks, grid), 32 * W, smem, s>>>(p);
  }
  return cudaGetLastError();
}

template <int D>
cudaError_t encm_dispatch(const EncodeParams& p, int grid, cudaStream_t s) {
  const bool sc = p.c.scale_mode != TQ_SCALE_NORM;
  switch (p.c.bits) {
    case 1: return sc ? encm_launch<D, 1, true>(p, grid, s) : encm_launch<D, 1, false>(p, grid, s);
    case 2: return sc ? encm_launch<D, 2, true>(p, grid, s) : encm_launch<D, 2, false>(p, grid, s);
    case 3: return sc ? encm_launch<D, 3, true>(p, grid, s) : encm_launch<D, 3, false>(p, grid, s);
    case 4: return sc ? encm_launch<D, 4, true>(p, grid, s) : encm_launch<D, 4, false>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tq
