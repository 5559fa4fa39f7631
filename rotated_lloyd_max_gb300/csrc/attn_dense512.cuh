// Decode attention over dense bf16 tokens at head dim 512 on the tensor cores:
// the dense splits (a tail ring, bf16 layers) of calls whose compressed splits
// run the head-dim-512 kernels, for groups of a multiple of 16 query heads.
//
// One CTA (4 warps) per (layer, batch, kv head, group of 16 query heads, dense
// split).  The heads are the MMA's M dimension, so a CTA reads each token once
// for its 16 heads.  Tokens go through shared memory in chunks of 32 (K and V
// rows, bf16; rows past the split's end are zeros):
//   scores   S[h][t] = q[h] . k[t]       mma.sync m16n8k16 bf16, A = q (16 x 512,
//            staged once), B = K rows; warp w takes tokens 8w .. 8w + 7 of the
//            chunk, over the 32 k-steps in two independent chains;
//   softmax  per head over the chunk (the warps' maxima meet in shared memory),
//            running maximum and sum in the log2 domain as in the other kernels;
//   values   O[h][j] += P[h][t] V[t][j]  A = P split into three bf16 parts
//            (its f32 value to 24 bits), B = V rows read transposed (ldmatrix
//            .trans); warp w owns coordinates 128w .. 128w + 127.
// bf16 q, K and V are exact MMA operands, their products exact and the sums
// f32.  The split's partial (m, l, acc) goes to the workspace like every
// other kernel's, for the merge.
#pragma once

#include <cuda_bf16.h>

#include "attn.cuh"

namespace tq {

constexpr int kD5Heads = 16;           // query heads per CTA (the MMA's M)
constexpr int kD5Chunk = 32;           // tokens staged per step
constexpr int kD5Row = 512 + 8;        // bf16 per shared row: 1,040 bytes, so the 8 rows an
                                       // ldmatrix reads start in 8 different 16-byte bank groups
constexpr int kD5PRow = kD5Chunk + 8;  // bf16 per row of P

struct D5Smem {
  __nv_bfloat16 q[kD5Heads][kD5Row];
  __nv_bfloat16 k[kD5Chunk][kD5Row];
  __nv_bfloat16 v[kD5Chunk][kD5Row];
  __nv_bfloat16 pp[3][kD5Heads][kD5PRow];  // P in three bf16 parts
  float wred[4][kD5Heads];                 // per-warp maxima, sums, final maxima
};
constexpr int attn_dense512_smem() { return (int)sizeof(D5Smem); }

__device__ __forceinline__ void d5_ldsm(uint32_t (&r)[4], const void* p) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
__device__ __forceinline__ void d5_ldsm_t(uint32_t (&r)[4], const void* p) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
__device__ __forceinline__ void d5_mma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// (x0, x1) -> three bf16 pairs whose sum is (x0, x1) to 24 significant bits.
__device__ __forceinline__ void d5_split3(float x0, float x1, uint32_t (&w)[3]) {
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    w[k] = *reinterpret_cast<const uint32_t*>(&h);
    const float2 f = __bfloat1622float2(h);
    x0 -= f.x;
    x1 -= f.y;
  }
}

__global__ void __launch_bounds__(kThreads, 2) attn_dense512_kernel(const __grid_constant__ AttnParams p) {
  constexpr int D = 512;
  extern __shared__ __align__(128) unsigned char smraw[];
  D5Smem& sm = *reinterpret_cast<D5Smem*>(smraw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t = lane & 3;
  const int l = blockIdx.z;
  int rem = blockIdx.y;
  const int hg = rem % p.n_hg;
  rem /= p.n_hg;
  const int kvh = rem % p.Hkv, b = rem / p.Hkv;
  const int split = blockIdx.x + p.split_base;
  const int h0 = kvh * p.G + hg * kD5Heads;
  const int lb = l * p.B + b;
  const int64_t qh0 = (int64_t)lb * p.Hq + h0;
  const int len = min(p.tail_len ? p.tail_len[lb] : 0, p.tail_cap);
  const int t_begin = (split - p.Sc) * p.tps;
  const int t_end = min(t_begin + p.tps, len);
  if (t_begin >= t_end) {
    if (tid < kD5Heads) {
      float* ml = p.ws_ml + ((qh0 + tid) * p.S + split) * 2;
      ml[0] = -INFINITY;
      ml[1] = 0.f;
    }
    return;
  }
  const int n = t_end - t_begin, cap = p.tail_cap;
  const int tstart = p.tail_start ? ((p.tail_start[lb] % cap) + cap) % cap : 0;
  const uint16_t* kt0 = p.ktail + l * p.tail_ls + (int64_t)(b * p.Hkv + kvh) * cap * D;
  const uint16_t* vt0 = p.vtail + l * p.tail_ls + (int64_t)(b * p.Hkv + kvh) * cap * D;
  // q rows of the 16 heads (64 16-byte pieces each), in the first chunk's group
  const uint16_t* qp = p.q + l * p.q_ls + b * p.q_bs + (int64_t)h0 * D;
  for (int i = tid; i < kD5Heads * 64; i += kThreads)
    cp_async16(&sm.q[i >> 6][8 * (i & 63)], qp + (int64_t)(i >> 6) * D + 8 * (i & 63));

  // ldmatrix row addresses of a 16 x 16 A tile: lane L gives row (L & 7) +
  // 8 ((L >> 3) & 1), column 8 (L >> 4) of the tile
  const int ar = (lane & 7) + ((lane >> 3) & 1) * 8, ac = (lane >> 4) * 8;
  float acc[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY;  // running maxima of heads g, g + 8
  float l0 = 0.f, l1 = 0.f;              // this lane's part of their sums
  const int nch = (n + kD5Chunk - 1) / kD5Chunk;
  for (int ch = 0; ch < nch; ++ch) {
    const int c0 = ch * kD5Chunk, cn = min(kD5Chunk, n - c0);
    for (int i = tid; i < kD5Chunk * 64; i += kThreads) {
      const int r = i >> 6, c = 8 * (i & 63);
      if (r < cn) {
        int s = tstart + t_begin + c0 + r;  // < 2 cap
        if (s >= cap) s -= cap;
        cp_async16(&sm.k[r][c], kt0 + (int64_t)s * D + c);
        cp_async16(&sm.v[r][c], vt0 + (int64_t)s * D + c);
      } else {
        *reinterpret_cast<uint4*>(&sm.k[r][c]) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(&sm.v[r][c]) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();

    // ---- scores of heads g, g + 8 and tokens 8w + 2t, + 1 of the chunk
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int kk = 0; kk < 32; kk += 2) {
      uint32_t a0[4], a1[4], bk[4];
      d5_ldsm(a0, &sm.q[ar][16 * kk + ac]);
      d5_ldsm(a1, &sm.q[ar][16 * kk + 16 + ac]);
      // K rows of the warp's tokens: matrices (k-step kk, low/high 8 coordinates), (kk + 1, ...)
      d5_ldsm(bk, &sm.k[8 * warp + (lane & 7)][16 * kk + 8 * (lane >> 3)]);
      d5_mma(sa, a0, bk[0], bk[1]);
      d5_mma(sb, a1, bk[2], bk[3]);
    }
    const int tk = 8 * warp + 2 * t;
    float s[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      s[e] = (sa[e] + sb[e]) * p.sscale;
      if (p.scap > 0.f) s[e] = soft_cap(s[e], p.scap, p.iscap);
    }
    if (tk >= cn) s[0] = s[2] = -INFINITY;
    if (tk + 1 >= cn) s[1] = s[3] = -INFINITY;
    // ---- online softmax over the chunk
    float x0 = fmaxf(s[0], s[1]), x1 = fmaxf(s[2], s[3]);
    x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 1));
    x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 1));
    x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 2));
    x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 2));
    if (t == 0) {
      sm.wred[warp][g] = x0;
      sm.wred[warp][g + 8] = x1;
    }
    __syncthreads();
    float cm0 = sm.wred[0][g], cm1 = sm.wred[0][g + 8];
#pragma unroll
    for (int w = 1; w < 4; ++w) {
      cm0 = fmaxf(cm0, sm.wred[w][g]);
      cm1 = fmaxf(cm1, sm.wred[w][g + 8]);
    }
    const float n0 = fmaxf(m0, cm0), n1 = fmaxf(m1, cm1);
    const float al0 = n0 == -INFINITY ? 1.f : exp2f(m0 - n0), al1 = n1 == -INFINITY ? 1.f : exp2f(m1 - n1);
    m0 = n0;
    m1 = n1;
    l0 *= al0;
    l1 *= al1;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      acc[i][0] *= al0;
      acc[i][1] *= al0;
      acc[i][2] *= al1;
      acc[i][3] *= al1;
    }
    const float p0 = s[0] == -INFINITY ? 0.f : exp2f(s[0] - m0), p1 = s[1] == -INFINITY ? 0.f : exp2f(s[1] - m0);
    const float p2 = s[2] == -INFINITY ? 0.f : exp2f(s[2] - m1), p3 = s[3] == -INFINITY ? 0.f : exp2f(s[3] - m1);
    l0 += p0 + p1;
    l1 += p2 + p3;
    uint32_t w01[3], w23[3];
    d5_split3(p0, p1, w01);
    d5_split3(p2, p3, w23);
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      *reinterpret_cast<uint32_t*>(&sm.pp[k][g][tk]) = w01[k];
      *reinterpret_cast<uint32_t*>(&sm.pp[k][g + 8][tk]) = w23[k];
    }
    __syncthreads();

    // ---- values: coordinates 128w .. 128w + 127 (16 n-tiles), tokens of the chunk
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      uint32_t ap[3][4];
#pragma unroll
      for (int k = 0; k < 3; ++k) d5_ldsm(ap[k], &sm.pp[k][ar][16 * ks + ac]);
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        uint32_t bv[4];  // V rows (tokens 16 ks ..) read transposed: n-tiles 2 np and 2 np + 1
        d5_ldsm_t(bv, &sm.v[16 * ks + ar][128 * warp + 16 * np + ac]);
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          d5_mma(acc[2 * np], ap[k], bv[0], bv[1]);
          d5_mma(acc[2 * np + 1], ap[k], bv[2], bv[3]);
        }
      }
    }
    __syncthreads();  // the chunk's K, V and P are consumed
  }

  // ---- the split's partial: acc rows (heads) relative to m, (m, l) per head
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int j = 128 * warp + 8 * i + 2 * t;
    *reinterpret_cast<float2*>(p.ws_acc + ((qh0 + g) * p.S + split) * D + j) = make_float2(acc[i][0], acc[i][1]);
    *reinterpret_cast<float2*>(p.ws_acc + ((qh0 + g + 8) * p.S + split) * D + j) = make_float2(acc[i][2], acc[i][3]);
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  if (t == 0) {
    sm.wred[warp][g] = l0;
    sm.wred[warp][g + 8] = l1;
  }
  __syncthreads();
  if (tid < kD5Heads) {
    const float L = sm.wred[0][tid] + sm.wred[1][tid] + sm.wred[2][tid] + sm.wred[3][tid];
    float* ml = p.ws_ml + ((qh0 + tid) * p.S + split) * 2;
    ml[1] = L;
  }
  if (warp == 0 && t == 0) {  // every lane holds the same maxima of its heads
    float* ml0 = p.ws_ml + ((qh0 + g) * p.S + split) * 2;
    float* ml1 = p.ws_ml + ((qh0 + g + 8) * p.S + split) * 2;
    ml0[0] = m0;
    ml1[0] = m1;
  }
}

inline cudaError_t attn_dense512_launch(const AttnParams& p, dim3 grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(attn_dense512_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       attn_dense512_smem());
  if (e != cudaSuccess) return e;
  attn_dense512_kernel<<<grid, kThreads, attn_dense512_smem(), s>>>(p);
  return cudaGetLastError();
}

}  // namespace tq
