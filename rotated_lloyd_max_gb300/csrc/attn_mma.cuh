// Decode attention on the tensor cores over the compressed records
// (head dims 64 and 128, up to 8 query heads of one kv head per CTA).
//
// Same quantities as the warp-local kernel (q~ = H(s_k . q)/sqrt(d) once per
// CTA; a token scores n_i * q~ . c[codes]; values accumulate p_i n_i c[codes]
// in the rotated basis, inverted once by the merge), but both contractions
// run as mma.sync.m16n8k16 (f16 operands, f32 accumulation):
//   scores   C[token][head]  = K~[token][coord] . Q~^T[coord][head]
//   values   O^T[coord][head] += V~^T[coord][token] . P'^T[token][head]
// with the query heads (<= 8) as the MMA's n dimension.  f16 alone does not
// hold an f32 centroid or q~ to the attention tolerance, so every operand is
// split x = hi + lo (two f16, 22 significant bits) and a product is the three
// MMAs hi.hi + hi.lo + lo.hi.  Centroids enter scaled by 2^16, q~ by a per-head
// power of two and P' by a per-warp power of two, so that no f16 part is
// subnormal or out of range; the scales are undone in f32.
//
// Dequantisation is one 64-bit shared-memory load per PAIR of codes from a
// pair table (entry = hi pair, lo pair), replicated so that lane j of a
// half-warp only ever touches bank pair j (conflict-free at any index).
// Fragment coordinates are permuted so that a lane's codes are a contiguous
// bit run of a packed row:
//   score A (tokens x coords), k-step kk: fragment column 2t+e <-> coordinate
//     (d/4) t + 4 kk + e, column 2t+8+e <-> (d/4) t + 4 kk + 2 + e;
//   value A (coords x tokens), m-tile mc: fragment row g <-> coordinate
//     (d/8) g + 2 mc, row g+8 <-> (d/8) g + 2 mc + 1.
// (g = lane / 4, t = lane % 4: the mma.sync fragment coordinates.)
//
// A warp owns 32 of a record's 128 tokens (two m-tiles) end to end; records
// are staged with cp.async in a two-deep ring, one CTA barrier per record;
// the online softmax is warp-local (the running max moves only when a logit
// passes it by 2^8).
// Outlier side lists (OUTL, the sparse-V route of such codecs): a CTA is
// three 4-warp groups (one CTA per SM holding one copy of the pair tables;
// 4-bit keys take 32 KB), each group with its own staging ring and barrier
// over every third record of the split.  A record is staged with its per-slot
// counts and the first entries of its list (the rest, rarely any, are read
// from global memory).  The MMAs score the centroids; lane l then takes the
// entries (slot, j, value) of the warp's token l, four at a time with their
// loads independent, adding (value - c[code_j]) q~_h[j] for every head (q~
// by coordinate, one 128-bit load) before the sums move to the lanes whose
// score fragments hold the token.  For the values the same lane adds
// (value - c[code_j]) 2^16 P'(token, h) to a per-warp shared buffer over
// (head, coordinate) in the accumulator's units, in fixed point through
// shared integer atomics; the owning lanes fold it into their accumulator
// fragments during the next record (folding right after the value MMAs
// stalls on their results), with 64-bit accesses laid out across all banks.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <type_traits>

#include "attn.cuh"

namespace tq {

__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (x0, x1) -> f16 pairs hi = f16(x), lo = f16(x - hi); x0 in the low half.
__device__ __forceinline__ void split_f16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 hf = __half22float2(h);
  const __half2 r = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&r);
}

// floor(log2 x) for a normal positive float (-127 for zero).
__device__ __forceinline__ int exp_of(float x) { return (int)((__float_as_uint(x) >> 23) & 0xFFu) - 127; }
// 2^e as a float, e clamped to the normal range.
__device__ __forceinline__ float pow2i(int e) {
  e = max(-126, min(127, e));
  return __uint_as_float((uint32_t)(e + 127) << 23);
}

// NB bits of a packed row starting at bit `off` (NB, off multiples of 32 when
// ALIGNED), as ceil(NB/32) words, LSB-first.  The unaligned form reads one
// word past the run: callers keep that inside the staged record.
template <int NB, bool ALIGNED>
__device__ __forceinline__ void load_run(const unsigned char* row, int off, uint32_t (&w)[(NB + 31) / 32]) {
  constexpr int NW = (NB + 31) / 32;
  const uint32_t* r = reinterpret_cast<const uint32_t*>(row) + (off >> 5);
  if constexpr (ALIGNED && NW == 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(r);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if constexpr (ALIGNED && NW == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(r);
    w[0] = v.x; w[1] = v.y;
  } else if constexpr (ALIGNED) {
#pragma unroll
    for (int i = 0; i < NW; ++i) w[i] = r[i];
  } else {
    const int sh = off & 31;
    uint32_t tmp[NW + 1];
#pragma unroll
    for (int i = 0; i <= NW; ++i) tmp[i] = r[i];
#pragma unroll
    for (int i = 0; i < NW; ++i) w[i] = __funnelshift_r(tmp[i], tmp[i + 1], sh);
  }
}

// Shared-memory byte offset of the pair-table entry named by the W-bit field
// at bit `off` of a word run: field * 128 + lane_off (lane_off < 128), i.e.
// the field moved to bit 7 and or-ed with the lane's bank-pair offset.
template <int NW>
__device__ __forceinline__ uint32_t pair_off(const uint32_t (&w)[NW], int off, int W, uint32_t lane_off) {
  const int wi = off >> 5, sh = off & 31;
  uint32_t v;
  if (sh + W <= 32 || wi + 1 >= NW) v = sh >= 7 ? (w[wi] >> (sh - 7)) : (w[wi] << (7 - sh));
  else v = __funnelshift_r(w[wi], w[wi + 1], sh - 7);
  return (v & (((1u << W) - 1u) << 7)) | lane_off;
}

// 3-bit codes -> one code per nibble (8 codes of a 24-bit field -> 32 bits).
__device__ __forceinline__ uint32_t spread3(uint32_t x) {
  x &= 0xFFFFFFu;
  x = (x & 0xFFFu) | ((x << 4) & 0xFFF0000u);
  x = (x & 0x003F003Fu) | ((x << 2) & 0x3F003F00u);
  x = (x & 0x07070707u) | ((x << 1) & 0x70707070u);
  return x;
}

// Code of coordinate j of a packed row (BITS-bit fields, LSB-first); a 3-bit
// field may straddle two words (the second read stays inside the staged record).
template <int BITS>
__device__ __forceinline__ uint32_t row_code(const unsigned char* row, int j) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(row);
  const int bit = j * BITS;
  if constexpr (BITS == 3) return __funnelshift_r(w[bit >> 5], w[(bit >> 5) + 1], bit & 31) & 7u;
  else return (w[bit >> 5] >> (bit & 31)) & ((1u << BITS) - 1u);
}

// Side-list entries of the warp's 32 slots of a staged record (per-slot
// counts at `counts`): lane l gets (offset of slot 32 w + l's first entry) << 8
// | its count.
__device__ __forceinline__ int slot_entries(const unsigned char* counts, int warp, int lane) {
  const int c = counts[32 * warp + lane];
  int pre = 0;
  for (int s = lane; s < 32 * warp; s += 32) pre += counts[s];
  const int base = (int)__reduce_add_sync(0xffffffffu, (unsigned)pre);
  int inc = c;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, inc, m);
    if (lane >= m) inc += o;
  }
  return ((base + inc - c) << 8) | c;
}

constexpr int kMmaHeads = 8;  // query heads per CTA at most
// Barrier of the 4 warps of group grp < 3 (named barriers 1-3; 0 is __syncthreads).
__device__ __forceinline__ void group_sync(int grp) {
  if (grp == 0) asm volatile("bar.sync 1, 128;\n" ::: "memory");
  else if (grp == 1) asm volatile("bar.sync 2, 128;\n" ::: "memory");
  else asm volatile("bar.sync 3, 128;\n" ::: "memory");
}

template <int D>
struct MCfg {
  static constexpr int KS = D / 16;  // score k-steps = value m-tiles
  static constexpr int KR = D / 4;   // coordinates of a lane's score run
  static constexpr int VR = D / 8;   // coordinates of a lane group's value run
};

// Value pair-table index width: 2b bits, or two nibbles for b = 3.
template <int VB>
struct VIdx {
  static constexpr int FW = (VB == 3) ? 4 : VB;   // field width after spreading
  static constexpr int ENTRIES = (VB == 3) ? 120 : (1 << (2 * VB));
};

// Pair-index words for the value fragments of tokens (t0, t1): ze holds, per
// 2*FW-bit field m, (code(t0, 2m) | code(t1, 2m) << FW); zo the same for the
// odd coordinates.
template <int VB, int NW>
__device__ __forceinline__ void v_pair_words(const uint32_t (&r0)[NW], const uint32_t (&r1)[NW],
                                             uint32_t (&ze)[(VB == 3) ? 2 * NW : NW],
                                             uint32_t (&zo)[(VB == 3) ? 2 * NW : NW]) {
  if constexpr (VB == 3) {
    // spread to nibbles first (NW words of 3-bit codes hold at most 16 codes)
    constexpr int NS = 2 * NW;
    uint32_t s0[NS], s1[NS];
    s0[0] = spread3(r0[0]);
    s1[0] = spread3(r1[0]);
    if constexpr (NS > 1) {
      s0[1] = spread3(NW > 1 ? __funnelshift_r(r0[0], r0[1], 24) : (r0[0] >> 24));
      s1[1] = spread3(NW > 1 ? __funnelshift_r(r1[0], r1[1], 24) : (r1[0] >> 24));
    }
#pragma unroll
    for (int i = 2; i < NS; ++i) { s0[i] = 0u; s1[i] = 0u; }
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      ze[i] = (s0[i] & 0x0F0F0F0Fu) | ((s1[i] << 4) & 0xF0F0F0F0u);
      zo[i] = ((s0[i] >> 4) & 0x0F0F0F0Fu) | (s1[i] & 0xF0F0F0F0u);
    }
  } else {
    constexpr uint32_t M = VB == 4 ? 0x0F0F0F0Fu : VB == 2 ? 0x33333333u : 0x55555555u;
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      ze[i] = (r0[i] & M) | ((r1[i] << VB) & ~M);
      zo[i] = ((r0[i] >> VB) & M) | (r1[i] & ~M);
    }
  }
}

// The CTA's warps' (m, l, acc) of a split -> the split's partial in the
// workspace.  acc is in the value-fragment layout (coordinate (d/8) g + 2 mc
// (+1 for elements 2, 3), head 2t (+1 for odd elements)), scaled by 1/un.
// mainb (the staging rings, free by now) holds the warps' partials.
template <int D>
__device__ __forceinline__ void mma_split_merge(const AttnParams& p, unsigned char* mainb, float* wml,
                                                const float (&acc)[D / 16][4], float un, float m0, float m1,
                                                float l0, float l1, int GT, int64_t qh0, int split) {
  constexpr int KS = D / 16, VR = D / 8;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t = lane & 3;
  const int NW = blockDim.x >> 5;
#pragma unroll
  for (int m = 4; m < 32; m <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, m);
    l1 += __shfl_xor_sync(0xffffffffu, l1, m);
  }
  __syncwarp();
  cp_async_wait<0>();
  __syncthreads();  // all tokens consumed: the staging rings become the merge buffer
  // merge buffer [warps][8 heads][D + D/8]: element (h, j) of a warp at
  // h (D + D/8) + j + 4 (j / 32) + h / 2, so that a warp's 32 fragment stores
  // (j = (d/8) g + const, h = 2t + const) hit 32 different banks
  float* red = reinterpret_cast<float*>(mainb);
  constexpr int RS = D + D / 8;
  auto red_at = [&](int w, int h, int j) { return w * 8 * RS + h * RS + j + 4 * (j >> 5) + (h >> 1); };
#pragma unroll
  for (int mc = 0; mc < KS; ++mc)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = VR * g + 2 * mc + (e >> 1), h = 2 * t + (e & 1);
      red[red_at(warp, h, j)] = acc[mc][e] * un;
    }
  if (g == 0) {
    wml[(warp * 2) * 8 + 2 * t] = m0;
    wml[(warp * 2) * 8 + 2 * t + 1] = m1;
    wml[(warp * 2 + 1) * 8 + 2 * t] = l0;
    wml[(warp * 2 + 1) * 8 + 2 * t + 1] = l1;
  }
  __syncthreads();
  for (int idx = tid; idx < GT * D; idx += blockDim.x) {
    const int h = idx / D, j = idx % D;
    float M = -INFINITY;
    for (int w = 0; w < NW; ++w) M = fmaxf(M, wml[(w * 2) * 8 + h]);
    float v = 0.f, L = 0.f;
    for (int w = 0; w < NW; ++w) {
      const float mw = wml[(w * 2) * 8 + h];
      const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
      v = fmaf(f, red[red_at(w, h, j)], v);
      L = fmaf(f, wml[(w * 2 + 1) * 8 + h], L);
    }
    p.ws_acc[((qh0 + h) * p.S + split) * D + j] = v;
    if (j == 0) {
      float* ml = p.ws_ml + ((qh0 + h) * p.S + split) * 2;
      ml[0] = M;
      ml[1] = L;
    }
  }
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (x0, x1) -> three bf16 pairs whose sum is x to 24 significant bits.
__device__ __forceinline__ void split3_bf16x2(float x0, float x1, uint32_t (&w)[3]) {
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    w[k] = *reinterpret_cast<const uint32_t*>(&h);
    const float2 hf = __bfloat1622float2(h);
    x0 -= hf.x;
    x1 -= hf.y;
  }
}

// Dense split (tail ring tokens or a bf16 layer) of the tensor-core kernel:
// the bf16 keys and values are exact MMA operands, and so is q (not rotated
// here), so a score is one bf16 MMA per k-step; the probabilities are split
// into three bf16 parts for the value MMAs.  Same fragment coordinate
// permutations as the compressed path; a warp takes 16-token tiles.
template <int D>
__device__ __noinline__ void mma_dense_split(const AttnParams& p, unsigned char* mainb, float* wml, int l, int b,
                                             int kvh, int GT, int h0, int64_t qh0, int lb, int split) {
  constexpr int KS = D / 16, KR = D / 4, VR = D / 8;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, t = lane & 3;
  const int len = min(p.tail_len ? p.tail_len[lb] : 0, p.tail_cap);
  const int t_begin = (split - p.Sc) * p.tps;
  const int t_end = min(t_begin + p.tps, len);
  if (t_begin >= t_end) {
    if (threadIdx.x < GT) {
      float* ml = p.ws_ml + ((qh0 + threadIdx.x) * p.S + split) * 2;
      ml[0] = -INFINITY;
      ml[1] = 0.f;
    }
    return;
  }
  const int n = t_end - t_begin;
  const int cap = p.tail_cap;
  const int tstart = p.tail_start ? ((p.tail_start[lb] % cap) + cap) % cap : 0;
  const int first = (tstart + t_begin) % cap;
  const uint16_t* kt0 = p.ktail + l * p.tail_ls + (int64_t)(b * p.Hkv + kvh) * cap * D;
  const uint16_t* vt0 = p.vtail + l * p.tail_ls + (int64_t)(b * p.Hkv + kvh) * cap * D;
  auto slot = [&](int i) { int s = first + i; return s >= cap ? s - cap : s; };  // i < n <= cap

  // query fragments: head g (zero beyond GT), coordinates (d/4) t + 4 kk + {0,1} / {2,3}
  uint32_t bq[KS][2];
  {
    const uint16_t* qp = p.q + l * p.q_ls + b * p.q_bs + (int64_t)(h0 + min(g, GT - 1)) * D + KR * t;
#pragma unroll
    for (int kk = 0; kk < KS; kk += 2) {
      const uint4 w = *reinterpret_cast<const uint4*>(qp + 4 * kk);
      bq[kk][0] = g < GT ? w.x : 0u;
      bq[kk][1] = g < GT ? w.y : 0u;
      bq[kk + 1][0] = g < GT ? w.z : 0u;
      bq[kk + 1][1] = g < GT ? w.w : 0u;
    }
  }
  const bool hv0 = 2 * t < GT, hv1 = 2 * t + 1 < GT;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // (dense tokens are never skipped by sparse-V)
  float acc[KS][4];
#pragma unroll
  for (int mc = 0; mc < KS; ++mc)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[mc][e] = 0.f;

  const int ntile = (n + 15) / 16;
  for (int tile = warp; tile < ntile; tile += 4) {
    const int tb = tile * 16;
    // keys of tokens g, g + 8 (lane t's 32 coordinates), values of tokens
    // 2t, 2t+1, 2t+8, 2t+9 (lane group g's 16 coordinates); zero past the end
    uint32_t kw[2][KR / 2];
    uint32_t vw[4][VR / 2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int i = tb + g + 8 * r;
      const uint4* src = reinterpret_cast<const uint4*>(kt0 + (int64_t)slot(min(i, n - 1)) * D + KR * t);
#pragma unroll
      for (int k = 0; k < KR / 8; ++k) {
        const uint4 v = i < n ? __ldg(src + k) : make_uint4(0u, 0u, 0u, 0u);
        kw[r][4 * k] = v.x; kw[r][4 * k + 1] = v.y; kw[r][4 * k + 2] = v.z; kw[r][4 * k + 3] = v.w;
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = tb + 2 * t + (r & 1) + 8 * (r >> 1);
      const uint4* src = reinterpret_cast<const uint4*>(vt0 + (int64_t)slot(min(i, n - 1)) * D + VR * g);
#pragma unroll
      for (int k = 0; k < VR / 8; ++k) {
        const uint4 v = i < n ? __ldg(src + k) : make_uint4(0u, 0u, 0u, 0u);
        vw[r][4 * k] = v.x; vw[r][4 * k + 1] = v.y; vw[r][4 * k + 2] = v.z; vw[r][4 * k + 3] = v.w;
      }
    }
    // scores
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      const uint32_t a[4] = {kw[0][2 * kk], kw[1][2 * kk], kw[0][2 * kk + 1], kw[1][2 * kk + 1]};
      mma_bf16(sc, a, bq[kk][0], bq[kk][1]);
    }
    const bool va = tb + g < n, vb = tb + g + 8 < n;
    sc[0] = (hv0 && va) ? sc[0] * p.sscale : -INFINITY;
    sc[1] = (hv1 && va) ? sc[1] * p.sscale : -INFINITY;
    sc[2] = (hv0 && vb) ? sc[2] * p.sscale : -INFINITY;
    sc[3] = (hv1 && vb) ? sc[3] * p.sscale : -INFINITY;
    if (p.scap > 0.f) {
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[e] = soft_cap(sc[e], p.scap, p.iscap);
    }
    // online softmax (lazy rescale)
    const bool need = (sc[0] > m0 + 8.f) | (sc[2] > m0 + 8.f) | (sc[1] > m1 + 8.f) | (sc[3] > m1 + 8.f);
    if (__any_sync(0xffffffffu, need)) {
      float x0 = fmaxf(sc[0], sc[2]), x1 = fmaxf(sc[1], sc[3]);
#pragma unroll
      for (int m = 4; m < 32; m <<= 1) {
        x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, m));
        x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, m));
      }
      const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
      const float a0 = n0 == -INFINITY ? 1.f : exp2f(m0 - n0);
      const float a1 = n1 == -INFINITY ? 1.f : exp2f(m1 - n1);
      m0 = n0;
      m1 = n1;
      l0 *= a0;
      l1 *= a1;
#pragma unroll
      for (int mc = 0; mc < KS; ++mc) {
        acc[mc][0] *= a0;
        acc[mc][1] *= a1;
        acc[mc][2] *= a0;
        acc[mc][3] *= a1;
      }
    }
    const float p0 = sc[0] == -INFINITY ? 0.f : exp2f(sc[0] - m0);
    const float p1 = sc[1] == -INFINITY ? 0.f : exp2f(sc[1] - m1);
    const float p2 = sc[2] == -INFINITY ? 0.f : exp2f(sc[2] - m0);
    const float p3 = sc[3] == -INFINITY ? 0.f : exp2f(sc[3] - m1);
    l0 += p0 + p2;
    l1 += p1 + p3;
    // P^T fragments (three bf16 parts): tokens 2t, 2t+1 / 2t+8, 2t+9 of head g
    uint32_t tw[3], bw[3];
    split3_bf16x2(p0, p1, tw);
    split3_bf16x2(p2, p3, bw);
    const int sa = 4 * (2 * t) + (g >> 1), sb = sa + 4;
    const uint32_t sel = (g & 1) ? 0x7632u : 0x5410u;
    uint32_t pb0[3], pb1[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      pb0[k] = __byte_perm(__shfl_sync(0xffffffffu, tw[k], sa), __shfl_sync(0xffffffffu, tw[k], sb), sel);
      pb1[k] = __byte_perm(__shfl_sync(0xffffffffu, bw[k], sa), __shfl_sync(0xffffffffu, bw[k], sb), sel);
    }
    // values: rows g / g + 8 <-> coordinates (d/8) g + 2 mc / + 1
#pragma unroll
    for (int mc = 0; mc < KS; ++mc) {
      const uint32_t a[4] = {__byte_perm(vw[0][mc], vw[1][mc], 0x5410), __byte_perm(vw[0][mc], vw[1][mc], 0x7632),
                             __byte_perm(vw[2][mc], vw[3][mc], 0x5410), __byte_perm(vw[2][mc], vw[3][mc], 0x7632)};
#pragma unroll
      for (int k = 0; k < 3; ++k) mma_bf16(acc[mc], a, pb0[k], pb1[k]);
    }
  }
  mma_split_merge<D>(p, mainb, wml, acc, 1.f, m0, m1, l0, l1, GT, qh0, split);
}

template <int D, int KB, int VB, bool OUTL>
__global__ void __launch_bounds__(OUTL ? kMmaOutlGroups * kThreads : kThreads, OUTL ? 1 : 4)
    attn_mma_kernel(const __grid_constant__ AttnParams p) {
  using C = MCfg<D>;
  constexpr int KS = C::KS, KR = C::KR, VR = C::VR;
  constexpr int KNB = KR * KB, VNB = VR * VB;
  constexpr int KNW = (KNB + 31) / 32, VNW = (VNB + 31) / 32;
  constexpr bool KAL = (KNB % 32) == 0, VAL = (VNB % 32) == 0;
  constexpr int FW = VIdx<VB>::FW;
  constexpr int ZW = (VB == 3) ? 2 * VNW : VNW;
  constexpr int EK = 1 << (2 * KB), EV = VIdx<VB>::ENTRIES;
  constexpr int KP_OFF = 0, VP_OFF = EK * 128;  // pair tables at fixed offsets (immediate addressing)
  extern __shared__ __align__(128) unsigned char sm[];
  // q~ (f32): coordinate c of head h at h*4*ST + (c / KR)*ST + c % KR with
  // ST = max(KR, 32) + 1, so the 32 lanes' runs start in 32 different banks
  float* qf = reinterpret_cast<float*>(sm + p.sm_q);
  constexpr int QST = (MCfg<D>::KR > 32 ? MCfg<D>::KR : 32) + 1;
  auto qidx = [](int h, int c) { return h * 4 * QST + (c / MCfg<D>::KR) * QST + (c % MCfg<D>::KR); };
  float* wml = reinterpret_cast<float*>(sm + p.sm_red);   // [warps][2][8]
  uint4* qfrag = reinterpret_cast<uint4*>(sm + p.sm_logit);  // [KS][32 lanes] (hi b0, hi b1, lo b0, lo b1)
  uint2* cent = reinterpret_cast<uint2*>(sm + p.sm_slot); // [32] (hi|lo f16) of K then V centroids x 2^16
  unsigned char* mainb = sm + p.sm_main;
  // (OUTL) f32 centroids, K then V; q~ by coordinate [D][8 heads]; value
  // corrections [warp][head][D + 8]
  float* kcf = reinterpret_cast<float*>(sm + p.sm_lut);
  float* vcf = kcf + 16;
  const float4* qi4 = reinterpret_cast<const float4*>(sm + p.sm_qi);
  int* corr = reinterpret_cast<int*>(sm + p.sm_corr);
  // corrections of (head h, coordinate j) at h CST + j + 2 (j / 16): a fold's
  // 64-bit accesses (j = 16 g + 2 mc + {0, 1}, h = 2 t + const) then cover 32
  // different banks (CST = 8 mod 32)
  constexpr int CST = D == 128 ? 168 : 72;
  auto cj = [](int j) { return j + 2 * (j >> 4); };

  // (OUTL) The CTA is one or more groups of 4 warps (blockDim.x / 128).  Each
  // group stages and scores its own records of the split (records grp,
  // grp + NG, ...) with its own two-deep ring and barrier; the pair tables,
  // q~ and the query fragments are shared.  Otherwise one group.
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int NW = OUTL ? (int)(blockDim.x >> 5) : 4, NG = NW >> 2;
  const int grp = warp >> 2, wg = warp & 3, gtid = tid & 127;
  const int g = lane >> 2, t = lane & 3;
  const int l = blockIdx.z;
  int rem = blockIdx.y;
  const int hg = rem % p.n_hg;
  rem /= p.n_hg;
  const int kvh = rem % p.Hkv, b = rem / p.Hkv;
  const int split = blockIdx.x + p.split_base;
  const int GT = p.G / p.n_hg;
  const int h0 = kvh * p.G + hg * GT;
  const int lb = l * p.B + b;
  const int64_t qh0 = (int64_t)lb * p.Hq + h0;
  if (split >= p.Sc) {  // dense tokens (tail ring or bf16 layer); such launches run one group
    mma_dense_split<D>(p, sm + p.sm_main, reinterpret_cast<float*>(sm + p.sm_red), l, b, kvh, GT, h0, qh0, lb,
                       split);
    return;
  }
  const int nch = min(p.n_chunks[lb], p.rec_limit);
  const int c_begin = split * p.cps;
  const int c_end = min(c_begin + p.cps, nch);
  if (c_begin >= c_end) {
    if (tid < GT) {
      float* ml = p.ws_ml + ((qh0 + tid) * p.S + split) * 2;
      ml[0] = -INFINITY;
      ml[1] = 0.f;
    }
    return;
  }
  const int n = c_end - c_begin;
  const int ng = n > grp ? (n - grp + NG - 1) / NG : 0;  // this group's records
  // record c of this unit (contiguous, or through the block table)
  const uint8_t* kl0 = p.krec + l * p.krec_ls;
  const uint8_t* vl0 = p.shared_kv ? kl0 : p.vrec + l * p.vrec_ls;
  auto krec_at = [&](int64_t c) {
    return kl0 + rec_offset(p.table, p.table_stride, p.rec_cap, p.Hkv, b, kvh, (int)c, p.krec_bytes);
  };
  auto vrec_at = [&](int64_t c) {
    return vl0 + rec_offset(p.table, p.table_stride, p.rec_cap, p.Hkv, b, kvh, (int)c, p.vrec_bytes);
  };
  auto rec_of = [&](int i) { return (int64_t)c_begin + grp + (int64_t)NG * i; };
  auto stage = [&](int i) { return mainb + (2 * grp + (i & 1)) * p.sm_stage; };
  auto group_copy = [&](unsigned char* s, const uint8_t* gsrc, int bytes) {
    for (int off = gtid * 16; off < bytes; off += 128 * 16) cp_async16(s + off, gsrc + off);
  };
  auto issue_main = [&](int i) {
    if (i < ng) {
      const int64_t c = rec_of(i);
      group_copy(stage(i), krec_at(c), p.k_main);
      if (!p.shared_kv) group_copy(stage(i) + p.k_main, vrec_at(c), p.v_main);
    }
    cp_async_commit();
  };
  issue_main(0);

  // ---- q~ = H(s_k . q)/sqrt(d) of the CTA's heads (rows >= GT are zero)
  for (int hh = warp; hh < 8; hh += NW) {
    constexpr int R = D / 32;
    float x[R];
    if (hh < GT) {
      const uint16_t* qp = p.q + l * p.q_ls + b * p.q_bs + (int64_t)(h0 + hh) * D + lane * R;
#pragma unroll
      for (int r = 0; r < R; r += 2) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(qp + r);
        x[r] = bf16_lo(w);
        x[r + 1] = bf16_hi(w);
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int j = lane * R + r;
        if ((p.ksign[j >> 5] >> (j & 31)) & 1u) x[r] = -x[r];
      }
      fwht_regs<R>(x);
      fwht_lanes<R>(x, lane, 32);
#pragma unroll
      for (int r = 0; r < R; ++r) x[r] *= inv_sqrt_dim<D>();
    } else {
#pragma unroll
      for (int r = 0; r < R; ++r) x[r] = 0.f;
    }
#pragma unroll
    for (int r = 0; r < R; ++r) qf[qidx(hh, lane * R + r)] = x[r];
    if (OUTL && p.kout) {
      float* qi = reinterpret_cast<float*>(sm + p.sm_qi);
#pragma unroll
      for (int r = 0; r < R; ++r) qi[(lane * R + r) * 8 + hh] = x[r];
    }
  }
  // f16 halves of every centroid x 2^16: cent[i] = (hi, lo) of K centroid i,
  // cent[16 + i] of V centroid i
  if (tid < 32) {
    if constexpr (OUTL) kcf[tid] = tid < 16 ? p.kc[tid] : p.vc[tid - 16];
    const float v = (tid < 16 ? p.kc[tid] : p.vc[tid - 16]) * 65536.f;
    const __half h = __float2half_rn(v);
    const __half r = __float2half_rn(v - __half2float(h));
    cent[tid] = make_uint2(__half_as_ushort(h), __half_as_ushort(r));
  }
  __syncthreads();  // q~ and the centroid halves complete
  // pair tables: entry e at byte e*128 + (lane % 16)*8 holds (hi pair, lo pair)
  // of its two centroids (first in the low half)
  for (int i = tid; i < EK * 16; i += blockDim.x) {
    const int e = i >> 4;
    const uint2 a = cent[e & ((1 << KB) - 1)], c = cent[e >> KB];
    *reinterpret_cast<uint2*>(sm + KP_OFF + i * 8) = make_uint2(__byte_perm(a.x, c.x, 0x5410), __byte_perm(a.y, c.y, 0x5410));
  }
  for (int i = tid; i < EV * 16; i += blockDim.x) {
    const int e = i >> 4;
    const int c0 = e & ((1 << FW) - 1), c1 = e >> FW;
    uint2 v = make_uint2(0u, 0u);
    if (c0 < (1 << VB) && c1 < (1 << VB)) {
      const uint2 a = cent[16 + c0], c = cent[16 + c1];
      v = make_uint2(__byte_perm(a.x, c.x, 0x5410), __byte_perm(a.y, c.y, 0x5410));
    }
    *reinterpret_cast<uint2*>(sm + VP_OFF + i * 8) = v;
  }

  // ---- query fragments: head g, coordinates (d/4) t + 4 kk + {0,1} / {2,3},
  // scaled by 2^s_g so that the largest |q~| of the head is in [2^13, 2^14);
  // stored per lane in shared memory (read once per k-step for both m-tiles).
  // Packed (at most 4 heads per CTA): column g < 4 holds the hi part of head
  // g and column g + 4 its lo part, so that one MMA forms hi.hi and hi.lo
  // (and a second lo.hi and lo.lo): two MMAs per product instead of three,
  // the halves summed across lanes t and t ^ 2; a lane's heads are then
  // 2 (t & 1), 2 (t & 1) + 1.
  const bool pk = GT <= 4;
  const int th = pk ? (t & 1) : t;  // the lane's head pair in the score fragments
  float fq0, fq1;  // 2^-(s_h + 16) for the lane's score heads 2th, 2th+1
  {
    const int hq = pk ? (g & 3) : g;
    const float* qrow = qf + qidx(hq, KR * t);
    float mx = 0.f;
#pragma unroll
    for (int j = 0; j < KR; ++j) mx = fmaxf(mx, fabsf(qrow[j]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const int s = mx > 0.f ? 13 - exp_of(mx) : 0;
    const float sc = pow2i(s);
    for (int kk = warp; kk < KS; kk += NW) {
      uint4 f;
      split_f16x2(qrow[4 * kk] * sc, qrow[4 * kk + 1] * sc, f.x, f.z);
      split_f16x2(qrow[4 * kk + 2] * sc, qrow[4 * kk + 3] * sc, f.y, f.w);
      if (pk && g >= 4) {
        f.x = f.z;
        f.y = f.w;
      }
      qfrag[kk * 32 + lane] = f;
    }
    const int s0 = __shfl_sync(0xffffffffu, s, 4 * (2 * th));
    const int s1 = __shfl_sync(0xffffffffu, s, 4 * (2 * th + 1));
    fq0 = pow2i(-s0 - 16);
    fq1 = pow2i(-s1 - 16);
  }
  const bool hv0 = 2 * th < GT, hv1 = 2 * th + 1 < GT;
  const uint32_t loff = (lane & 15) * 8;
  auto kpair_at = [&](uint32_t o) { return *reinterpret_cast<const uint2*>(sm + KP_OFF + o); };
  auto vpair_at = [&](uint32_t o) { return *reinterpret_cast<const uint2*>(sm + VP_OFF + o); };

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  // sparse-V: exact running maxima of the lane's two heads over the warp's
  // earlier 32-token blocks of this split (the lazy m0/m1 may trail them)
  float tm0 = -INFINITY, tm1 = -INFINITY;
  const bool sparse_v = p.sv_log2eps < 0.f;
  float acc[KS][4];
#pragma unroll
  for (int mc = 0; mc < KS; ++mc)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[mc][e] = 0.f;
  int kx = 127;  // P' f16 scale exponent of this warp (only ever decreases)
  const int rbk = D * KB / 8, rbv = D * VB / 8;
  // (OUTL) the lane's part of the warp's value corrections (fixed point, one
  // record at a time): heads 2t, 2t + 1, coordinates (d/8) g + 2 mc (+1), as
  // its accumulator fragments
  const int GTe = (GT + 1) & ~1;
  // the pair (elements e, e + 2) of m-tile mc: head 2t + e, coordinates
  // (d/8) g + 2 mc and + 1
  auto corr_pair = [&](int e, int mc) -> int2& {
    return *reinterpret_cast<int2*>(corr + (warp * GTe + 2 * t + e) * CST + cj(VR * g + 2 * mc));
  };
  const bool own_corr = OUTL && p.vout && 2 * t < GT;
  if (own_corr) {
#pragma unroll
    for (int mc = 0; mc < KS; ++mc)
#pragma unroll
      for (int e = 0; e < 2; ++e) corr_pair(e, mc) = make_int2(0, 0);
  }
  // (OUTL) a record's value corrections are folded into the accumulators
  // during the next record (before its softmax may rescale them), when the
  // value MMAs that last wrote them have long completed: folding right after
  // those MMAs stalls the warp on their results
  bool fold_pending = false;
  float fold_iS = 0.f;
  auto fold = [&]() {
    __syncwarp();
    if (own_corr) {
#pragma unroll
      for (int mc = 0; mc < KS; ++mc)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          int2& v = corr_pair(e, mc);
          const int2 w = v;
          v = make_int2(0, 0);
          acc[mc][e] = fmaf((float)w.x, fold_iS, acc[mc][e]);
          acc[mc][e + 2] = fmaf((float)w.y, fold_iS, acc[mc][e + 2]);
        }
    }
    __syncwarp();
    fold_pending = false;
  };
  __syncthreads();  // pair tables and query fragments complete for every group

  for (int i = 0; i < ng; ++i) {
    cp_async_wait<0>();
    if constexpr (OUTL) group_sync(grp);  // record i is in; record i-1 is done with
    else __syncthreads();
    issue_main(i + 1);
    const unsigned char* st = stage(i);
    const unsigned char* kcodes = st + wg * 32 * rbk;
    const float* knorm = reinterpret_cast<const float*>(st + p.k_off_norm) + wg * 32;
    const unsigned char* vbase = p.shared_kv ? st : st + p.k_main;
    const unsigned char* vcodes = vbase + wg * 32 * rbv;
    const float* vnorm = reinterpret_cast<const float*>(vbase + p.v_off_norm) + wg * 32;

    // ---- scores: tile mt holds tokens 16 mt + g (elements 0, 1) and + 8 (2, 3)
    float sc[2][4];
    {
      uint32_t w[4][KNW];  // runs of tokens g, g + 8, 16 + g, 24 + g
#pragma unroll
      for (int r = 0; r < 4; ++r) load_run<KNB, KAL>(kcodes + (8 * r + g) * rbk, KNB * t, w[r]);
      // hi.hi, hi.lo and lo.hi in separate accumulators: independent MMA chains
      float cc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      float cl[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      float ch[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      // the k loop specialised on packing (a uniform branch, not predicated MMAs)
      auto score_mmas = [&](auto pkc) {
        constexpr bool P = decltype(pkc)::value;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const uint4 f = qfrag[kk * 32 + lane];
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            uint32_t ah[4], al[4];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const int off = (4 * kk + 2 * hf) * KB;
              const uint2 e0 = kpair_at(pair_off(w[2 * mt], off, 2 * KB, loff));
              const uint2 e1 = kpair_at(pair_off(w[2 * mt + 1], off, 2 * KB, loff));
              ah[2 * hf] = e0.x;
              al[2 * hf] = e0.y;
              ah[2 * hf + 1] = e1.x;
              al[2 * hf + 1] = e1.y;
            }
            mma_f16(cc[mt], ah, f.x, f.y);
            if constexpr (!P) mma_f16(cl[mt], ah, f.z, f.w);
            mma_f16(ch[mt], al, f.x, f.y);
          }
        }
      };
      if (pk) score_mmas(std::true_type{});
      else score_mmas(std::false_type{});
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) cc[mt][e] += cl[mt][e] + ch[mt][e];
      if (pk) {  // q~ hi columns (t < 2) plus lo columns (t >= 2)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) cc[mt][e] += __shfl_xor_sync(0xffffffffu, cc[mt][e], 2);
      }
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        sc[mt][0] = cc[mt][0] * fq0;
        sc[mt][1] = cc[mt][1] * fq1;
        sc[mt][2] = cc[mt][2] * fq0;
        sc[mt][3] = cc[mt][3] * fq1;
      }
    }
    // ---- key side lists: sc (centroid scores, before the norm) += sum over
    // the token's entries of (value - c[code_j]) q~_h[j].  Lane l takes the
    // entries of the warp's token l, one per round (as many rounds as the
    // warp's longest list); the sums then move to the lanes whose score
    // fragments hold the token.
    if constexpr (OUTL) {
      if (p.kout) {
        const int oc = slot_entries(st + p.k_off_count, wg, lane);
        const int off = oc >> 8, cnt = max(0, min(oc & 255, p.kcap - off));  // (a list longer than its capacity reads no further)
        const uint32_t* ent_s = reinterpret_cast<const uint32_t*>(st + p.k_off_ent);
        const int nse = (p.k_main - p.k_off_ent) >> 2;  // entries staged
        const bool staged = __all_sync(0xffffffffu, off + cnt <= nse);
        const uint32_t* ent_g = reinterpret_cast<const uint32_t*>(krec_at(rec_of(i)) + p.k_off_ent);
        const unsigned char* krow = kcodes + lane * rbk;
        const int rounds = (int)__reduce_max_sync(0xffffffffu, (unsigned)cnt);
        float dk[kMmaHeads];
#pragma unroll
        for (int h = 0; h < kMmaHeads; ++h) dk[h] = 0.f;
        // four entries per trip, their loads independent of one another
        for (int k0 = 0; k0 < rounds; k0 += 4) {
          uint32_t e[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int idx = k0 + u < cnt ? off + k0 + u : 0;
            if (staged || idx < nse) e[u] = ent_s[idx];
            else e[u] = __ldg(ent_g + idx);
          }
          float delta[4];
          int j[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            j[u] = (int)(e[u] & (uint32_t)(D - 1));
            delta[u] = k0 + u < cnt ? __uint_as_float(e[u] & 0xFFFF0000u) - kcf[row_code<KB>(krow, j[u])] : 0.f;
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float4 qa = qi4[2 * j[u]];
            dk[0] = fmaf(delta[u], qa.x, dk[0]);
            dk[1] = fmaf(delta[u], qa.y, dk[1]);
            dk[2] = fmaf(delta[u], qa.z, dk[2]);
            dk[3] = fmaf(delta[u], qa.w, dk[3]);
            if (GT > 4) {
              const float4 qb = qi4[2 * j[u] + 1];
              dk[4] = fmaf(delta[u], qb.x, dk[4]);
              dk[5] = fmaf(delta[u], qb.y, dk[5]);
              dk[6] = fmaf(delta[u], qb.z, dk[6]);
              dk[7] = fmaf(delta[u], qb.w, dk[7]);
            }
          }
        }
        // token g + 8 q sits in sc[q >> 1][2 (q & 1) + {0, 1}] (heads 2 th, 2 th + 1)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float d0 = 0.f, d1 = 0.f;
#pragma unroll
          for (int h = 0; h < kMmaHeads; h += 2) {
            if (h < GT) {
              const float a = __shfl_sync(0xffffffffu, dk[h], g + 8 * q);
              const float c2 = __shfl_sync(0xffffffffu, dk[h + 1], g + 8 * q);
              if (h == 2 * th) {
                d0 = a;
                d1 = c2;
              }
            }
          }
          sc[q >> 1][2 * (q & 1)] += d0;
          sc[q >> 1][2 * (q & 1) + 1] += d1;
        }
      }
    }
    if (OUTL && fold_pending) fold();
    // logits (log2 domain)
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const float fa = knorm[16 * mt + g] * p.sscale, fb = knorm[16 * mt + g + 8] * p.sscale;
      sc[mt][0] = hv0 ? sc[mt][0] * fa : -INFINITY;
      sc[mt][1] = hv1 ? sc[mt][1] * fa : -INFINITY;
      sc[mt][2] = hv0 ? sc[mt][2] * fb : -INFINITY;
      sc[mt][3] = hv1 ? sc[mt][3] * fb : -INFINITY;
    }
    if (p.scap > 0.f) {
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[mt][e] = soft_cap(sc[mt][e], p.scap, p.iscap);
    }
    // ---- sparse-V (turboquant_plus commit log, "sparse-V dequant"): the
    // values of the warp's 32 tokens of this record are skipped when, for
    // every head of the CTA, each of their logits lies below the exact
    // maximum of the warp's earlier blocks plus log2(eps); their weights
    // still enter the denominators
    bool skip_v = false;
    if (sparse_v) {
      float x0 = fmaxf(fmaxf(sc[0][0], sc[0][2]), fmaxf(sc[1][0], sc[1][2]));
      float x1 = fmaxf(fmaxf(sc[0][1], sc[0][3]), fmaxf(sc[1][1], sc[1][3]));
#pragma unroll
      for (int m = 4; m < 32; m <<= 1) {
        x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, m));
        x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, m));
      }
      const bool low = (!hv0 || x0 < tm0 + p.sv_log2eps) && (!hv1 || x1 < tm1 + p.sv_log2eps);
      skip_v = __all_sync(0xffffffffu, low);
      tm0 = fmaxf(tm0, x0);
      tm1 = fmaxf(tm1, x1);
    }
    // ---- online softmax (the max moves only when a logit passes it by 2^8)
    {
      bool need = false;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
        need |= (sc[mt][0] > m0 + 8.f) | (sc[mt][2] > m0 + 8.f) | (sc[mt][1] > m1 + 8.f) | (sc[mt][3] > m1 + 8.f);
      if (__any_sync(0xffffffffu, need)) {
        float x0 = fmaxf(fmaxf(sc[0][0], sc[0][2]), fmaxf(sc[1][0], sc[1][2]));
        float x1 = fmaxf(fmaxf(sc[0][1], sc[0][3]), fmaxf(sc[1][1], sc[1][3]));
#pragma unroll
        for (int m = 4; m < 32; m <<= 1) {
          x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, m));
          x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, m));
        }
        const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
        const float a0 = n0 == -INFINITY ? 1.f : exp2f(m0 - n0);
        const float a1 = n1 == -INFINITY ? 1.f : exp2f(m1 - n1);
        m0 = n0;
        m1 = n1;
        l0 *= a0;
        l1 *= a1;
#pragma unroll
        for (int mc = 0; mc < KS; ++mc) {
          acc[mc][0] *= a0;
          acc[mc][1] *= a1;
          acc[mc][2] *= a0;
          acc[mc][3] *= a1;
        }
      }
    }
    // p, l, p' = p * n_v (unscaled), in place of the logits
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const float va = vnorm[16 * mt + g], vb = vnorm[16 * mt + g + 8];
      const float p0 = hv0 ? exp2f(sc[mt][0] - m0) : 0.f, p1 = hv1 ? exp2f(sc[mt][1] - m1) : 0.f;
      const float p2 = hv0 ? exp2f(sc[mt][2] - m0) : 0.f, p3 = hv1 ? exp2f(sc[mt][3] - m1) : 0.f;
      l0 += p0 + p2;
      l1 += p1 + p3;
      sc[mt][0] = p0 * va;
      sc[mt][1] = p1 * va;
      sc[mt][2] = p2 * vb;
      sc[mt][3] = p3 * vb;
    }
    // f16 range of P': p <= 2^8, so p' 2^kx <= 2^15 with kx = 6 - floor(log2 max n_v)
    {
      const float vmax = warp_max(vnorm[lane]);
      if (vmax > 0.f) {
        const int kn = 6 - exp_of(vmax);
        if (kn < kx) {
          const float r = pow2i(kn - kx);
#pragma unroll
          for (int mc = 0; mc < KS; ++mc)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[mc][e] *= r;
          kx = kn;
        }
      }
    }
    const float psc = pow2i(kx);
    if (skip_v) continue;
    // ---- values: k-step mt = the 16 tokens of score tile mt
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      uint32_t thw, tlw, bhw, blw;  // (p' hi / lo) of tokens g (top) and g + 8 (bottom)
      split_f16x2(sc[mt][0] * psc, sc[mt][1] * psc, thw, tlw);
      split_f16x2(sc[mt][2] * psc, sc[mt][3] * psc, bhw, blw);
      // column g of P'^T: head g, or packed head g & 3, hi for g < 4 and lo beyond
      const int hb = pk ? (g & 3) : g;
      const int sa = 4 * (2 * t) + (hb >> 1), sb = sa + 4;
      const uint32_t sel = (hb & 1) ? 0x7632u : 0x5410u;
      uint32_t pb0h = __byte_perm(__shfl_sync(0xffffffffu, thw, sa), __shfl_sync(0xffffffffu, thw, sb), sel);
      const uint32_t pb0l = __byte_perm(__shfl_sync(0xffffffffu, tlw, sa), __shfl_sync(0xffffffffu, tlw, sb), sel);
      uint32_t pb1h = __byte_perm(__shfl_sync(0xffffffffu, bhw, sa), __shfl_sync(0xffffffffu, bhw, sb), sel);
      const uint32_t pb1l = __byte_perm(__shfl_sync(0xffffffffu, blw, sa), __shfl_sync(0xffffffffu, blw, sb), sel);
      if (pk && g >= 4) {
        pb0h = pb0l;
        pb1h = pb1l;
      }
      // value runs of tokens 2t, 2t+1 (k columns 2t, 2t+1) and 2t+8, 2t+9
      uint32_t r0[VNW], r1[VNW], r2[VNW], r3[VNW];
      const unsigned char* vt = vcodes + 16 * mt * rbv;
      load_run<VNB, VAL>(vt + (2 * t) * rbv, VNB * g, r0);
      load_run<VNB, VAL>(vt + (2 * t + 1) * rbv, VNB * g, r1);
      load_run<VNB, VAL>(vt + (2 * t + 8) * rbv, VNB * g, r2);
      load_run<VNB, VAL>(vt + (2 * t + 9) * rbv, VNB * g, r3);
      uint32_t ze01[ZW], zo01[ZW], ze23[ZW], zo23[ZW];
      v_pair_words<VB, VNW>(r0, r1, ze01, zo01);
      v_pair_words<VB, VNW>(r2, r3, ze23, zo23);
      auto value_mmas = [&](auto pkc) {
        constexpr bool P = decltype(pkc)::value;
#pragma unroll
        for (int mc = 0; mc < KS; ++mc) {
          const int off = mc * 2 * FW;
          const uint2 e0 = vpair_at(pair_off(ze01, off, 2 * FW, loff));
          const uint2 e1 = vpair_at(pair_off(zo01, off, 2 * FW, loff));
          const uint2 e2 = vpair_at(pair_off(ze23, off, 2 * FW, loff));
          const uint2 e3 = vpair_at(pair_off(zo23, off, 2 * FW, loff));
          const uint32_t ah[4] = {e0.x, e1.x, e2.x, e3.x};
          const uint32_t al[4] = {e0.y, e1.y, e2.y, e3.y};
          mma_f16(acc[mc], ah, pb0h, pb1h);
          if constexpr (!P) mma_f16(acc[mc], ah, pb0l, pb1l);
          mma_f16(acc[mc], al, pb0h, pb1h);
        }
      };
      if (pk) value_mmas(std::true_type{});
      else value_mmas(std::false_type{});
    }
    // ---- value side lists: corr[h][j] += (value - c[code_j]) 2^16 P'(token, h)
    // in fixed point S = 2^(23 - floor(log2 max 2^16 P')) (shared integer
    // atomics retire about four times faster than f32 ones): a term is below
    // 2^25 in magnitude (|value - c| < 2) and a (head, coordinate) takes at
    // most one term per token, so a record's sums stay below 2^30.  Lane l
    // takes the entries of the warp's token l, one per round, with the
    // token's P' gathered from the score fragments; the owners fold the sums
    // into their accumulators during the next record.
    if constexpr (OUTL) {
      if (p.vout) {
        const int oc = slot_entries(vbase + p.v_off_count, wg, lane);
        const int off = oc >> 8, cnt = max(0, min(oc & 255, p.vcap - off));
        const uint32_t* ent_s = reinterpret_cast<const uint32_t*>(vbase + p.v_off_ent);
        const int nse = (p.v_main - p.v_off_ent) >> 2;
        const bool staged = __all_sync(0xffffffffu, off + cnt <= nse);
        const uint32_t* ent_g = reinterpret_cast<const uint32_t*>(vrec_at(rec_of(i)) + p.v_off_ent);
        const unsigned char* vrow = vcodes + lane * rbv;
        float pmx = fmaxf(fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[0][2], sc[0][3])),
                          fmaxf(fmaxf(sc[1][0], sc[1][1]), fmaxf(sc[1][2], sc[1][3])));
        pmx = warp_max(pmx * (65536.f * psc));
        const int ef = min(254, max(1, 277 - (int)((__float_as_uint(pmx) >> 23) & 0xFFu)));
        const float S = __uint_as_float((uint32_t)ef << 23), iS = __uint_as_float((uint32_t)(254 - ef) << 23);
        const float fsc = 65536.f * psc * S;
        // token l = 16 mt + 8 eh + r8 sits in lane 4 r8 + h / 2, sc[mt][2 eh + (h & 1)]
        float pv[kMmaHeads];
        {
          const int mt = lane >> 4, eh = (lane >> 3) & 1, src0 = 4 * (lane & 7);
#pragma unroll
          for (int h = 0; h < kMmaHeads; h += 2) {
            pv[h] = 0.f;
            pv[h + 1] = 0.f;
            if (h < GT) {
              float v[2][4];
#pragma unroll
              for (int m2 = 0; m2 < 2; ++m2)
#pragma unroll
                for (int e = 0; e < 4; ++e) v[m2][e] = __shfl_sync(0xffffffffu, sc[m2][e], src0 + (h >> 1));
              pv[h] = (mt ? (eh ? v[1][2] : v[1][0]) : (eh ? v[0][2] : v[0][0])) * fsc;
              pv[h + 1] = (mt ? (eh ? v[1][3] : v[1][1]) : (eh ? v[0][3] : v[0][1])) * fsc;
            }
          }
        }
        int* cw = corr + warp * GTe * CST;
        const int rounds = (int)__reduce_max_sync(0xffffffffu, (unsigned)cnt);
        for (int k0 = 0; k0 < rounds; k0 += 4) {
          uint32_t e[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int idx = k0 + u < cnt ? off + k0 + u : 0;
            if (staged || idx < nse) e[u] = ent_s[idx];
            else e[u] = __ldg(ent_g + idx);
          }
          float f[4];
          int j[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            j[u] = (int)(e[u] & (uint32_t)(D - 1));
            f[u] = __uint_as_float(e[u] & 0xFFFF0000u) - vcf[row_code<VB>(vrow, j[u])];
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (k0 + u < cnt) {
#pragma unroll
              for (int h = 0; h < kMmaHeads; ++h)
                if (h < GT) atomicAdd(cw + h * CST + cj(j[u]), __float2int_rn(f[u] * pv[h]));
            }
          }
        }
        fold_pending = true;
        fold_iS = iS;
      }
    }
  }
  if (OUTL && fold_pending) fold();

  if (pk) {  // P' hi columns (t < 2) plus lo columns (t >= 2)
#pragma unroll
    for (int mc = 0; mc < KS; ++mc)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mc][e] += __shfl_xor_sync(0xffffffffu, acc[mc][e], 2);
  }
  mma_split_merge<D>(p, mainb, wml, acc, pow2i(-16 - kx), m0, m1, l0, l1, GT, qh0, split);
}

template <int D, int KB, int VB, bool OUTL>
cudaError_t attn_mma_launch_o(const AttnParams& p, dim3 grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(attn_mma_kernel<D, KB, VB, OUTL>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, p.sm_total);
  if (e != cudaSuccess) return e;
  attn_mma_kernel<D, KB, VB, OUTL><<<grid, kThreads * std::max(1, p.groups), p.sm_total, s>>>(p);
  return cudaGetLastError();
}
template <int D, int KB, int VB>
cudaError_t attn_mma_launch_t(const AttnParams& p, dim3 grid, cudaStream_t s) {
  return (p.kout || p.vout) ? attn_mma_launch_o<D, KB, VB, true>(p, grid, s)
                            : attn_mma_launch_o<D, KB, VB, false>(p, grid, s);
}

}  // namespace tq
