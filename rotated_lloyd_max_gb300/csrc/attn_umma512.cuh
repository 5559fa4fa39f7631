// Decode attention at head dim 512 on the fifth-generation tensor cores (tcgen05.mma,
// accumulators in tensor memory), for compressed records of codecs without
// outlier side lists and groups of up to 64 query heads per kv head (MQA).
//
// Arithmetic (same contract as the mma.sync kernels): centroids x 2^16 and
// q~ x 2^s (per head) are split into f16 hi + lo; every product is the sum
// of the hi.hi, hi.lo and lo.hi MMAs with f32 accumulation; P' = p * n_V *
// 2^kx is split likewise.  One CTA is one split of one (layer, batch, kv head,
// group of <= 64 heads) and keeps all its heads, so each record is dequantised
// once per pass for the whole group:
//
//  * scores, one 128-token record at a time: S^T[token][n] = K~ . B_q with
//    B_q = [q~_hi (64 rows) | q~_lo (64 rows)] (N = 128, K-major, resident in
//    shared memory) plus K~_lo . q~_hi (N = 64) into the same accumulator, so
//    head h's logit is column h + column 64 + h of the token's TMEM lane;
//    two score buffers let a record's scores run while the previous record's
//    softmax is computed;
//  * softmax: a thread owns one token (its TMEM lane) and all 64 heads, in two
//    halves of 32; the running max per head moves only when a logit passes it
//    by 2^8 (or the record's largest V norm needs a smaller P' scale), which is
//    the one step that reduces across tokens and rescales the accumulator;
//  * values: O^T[coordinate][head] += V~^T . P' for four 128-coordinate
//    blocks (A = the dequantised record, MN-major; B = P', MN-major, N = 64);
//    O^T stays in tensor memory for the whole split.
//
// Warp roles (672 threads): warps 0-3 softmax and epilogue (warp w reads TMEM
// lanes 32 w .. 32 w + 31); warps 4-19 dequantise records into a two-stage
// ring of 32 KB operand tiles (16 stages per record: 8 score chunks of 64
// coordinates, hi and lo; 8 value blocks of 128 coordinates, hi or lo),
// 4-bit codes through byte-plane tables held in registers (byte permutes, no
// shared-memory lookups); warp 20 allocates tensor memory and its lane 0 only
// issues MMAs, each stage's once all sixteen warps have written it.  Stages,
// scores, P' and outputs are handed over through mbarriers; every wait is
// bounded and a CTA whose wait expires sets the launch's status word and
// finishes without further waiting.
#pragma once

#include "attn_mma.cuh"
#include "umma.cuh"

namespace tq {

constexpr int kU512Threads = 672;
constexpr int kUSoftWarps = 4;
constexpr int kUDeqWarps = 16;
constexpr int kUIssueWarp = kUSoftWarps + kUDeqWarps;
// shared memory (bytes from a 1024-aligned base)
constexpr int kUQ = 0;          // q~ operand: [8 chunks of 64 coordinates][128 rows][128 B]
constexpr int kUP = 131072;     // P' operand: hi [128 tokens][64 heads f16] | lo
constexpr int kURing = 163840;  // 2 stages x 32 KB
constexpr int kUMisc = 229376;
constexpr int kUSmem = kUMisc + 2048 + 1024;  // + bookkeeping + alignment slack

struct U512Misc {
  uint64_t full[2], empty[2], s_full[2], p_full, o_done, fin;
  uint32_t tbase;
  int abort_;
  uint32_t ctab_k[16], ctab_v[16];  // centroid x 2^16 as f16 {hi, lo} per code
  uint32_t plane_k[4][4], plane_v[4][4];  // the same as byte planes: hi.b0, hi.b1, lo.b0, lo.b1 of codes 4w..4w+3
  float qsc[64];                    // per head: softmax scale * log2(e) * 2^(-16 - s)
  float mst[64];                    // running max per head (log2 units)
  float red[4][64];                 // cross-quarter reductions; red[0] then holds the output rescale per head
  float vmx[4];
};
static_assert(sizeof(U512Misc) <= 2048, "bookkeeping block");

__device__ __forceinline__ bool bar_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbarrier.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, "
      "q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void bar_sync(int id, int nthreads) {
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// 16-entry byte plane lookup of four 4-bit codes (nibbles of sel): entries
// 0-7 and 8-15 by index sel & 7, then per byte the half chosen by bit 3
__device__ __forceinline__ uint32_t plane_lookup(const uint32_t (&P)[4], uint32_t sel7, uint32_t pick) {
  return __byte_perm(__byte_perm(P[0], P[1], sel7), __byte_perm(P[2], P[3], sel7), pick);
}
// 8 four-bit codes -> f16x2 hi / lo words from byte planes in registers
__device__ __forceinline__ void deq8_planes(uint32_t w, const uint32_t (&pl)[4][4], uint4& hi, uint4& lo) {
  uint32_t out_h[4], out_l[4];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const uint32_t sel = k ? (w >> 16) : w;
    const uint32_t sel7 = sel & 0x7777u;
    const uint32_t pick = 0x3210u + ((sel >> 3) & 0x1111u) * 4u;  // byte i from the low (i) or high (i + 4) lookup
    const uint32_t h0 = plane_lookup(pl[0], sel7, pick), h1 = plane_lookup(pl[1], sel7, pick);
    const uint32_t l0 = plane_lookup(pl[2], sel7, pick), l1 = plane_lookup(pl[3], sel7, pick);
    out_h[2 * k] = __byte_perm(h0, h1, 0x5140);
    out_h[2 * k + 1] = __byte_perm(h0, h1, 0x7362);
    out_l[2 * k] = __byte_perm(l0, l1, 0x5140);
    out_l[2 * k + 1] = __byte_perm(l0, l1, 0x7362);
  }
  hi = make_uint4(out_h[0], out_h[1], out_h[2], out_h[3]);
  lo = make_uint4(out_l[0], out_l[1], out_l[2], out_l[3]);
}

// dequantise 8 codes into f16x2 hi / lo words (coordinate 2i in the low half)
template <int B>
__device__ __forceinline__ void deq8(uint32_t w, const uint32_t* tab, uint4& hi, uint4& lo) {
  uint32_t e[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) e[i] = tab[(w >> (B * i)) & ((1u << B) - 1u)];
  hi = make_uint4(__byte_perm(e[0], e[1], 0x5410), __byte_perm(e[2], e[3], 0x5410), __byte_perm(e[4], e[5], 0x5410),
                  __byte_perm(e[6], e[7], 0x5410));
  lo = make_uint4(__byte_perm(e[0], e[1], 0x7632), __byte_perm(e[2], e[3], 0x7632), __byte_perm(e[4], e[5], 0x7632),
                  __byte_perm(e[6], e[7], 0x7632));
}

// 32 values per lane -> lane i holds the reduction over the warp of value i
template <bool MAX>
__device__ __forceinline__ float transpose_reduce(float (&v)[32], int lane) {
#pragma unroll
  for (int half = 16; half >= 1; half >>= 1) {
    const bool up = (lane & half) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float keep = up ? v[half + i] : v[i];
      const float give = up ? v[i] : v[half + i];
      const float got = __shfl_xor_sync(0xffffffffu, give, half);
      v[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  return v[0];
}

// Phase ph of a split of n records: S(0), then per record r S(r + 1) (when
// r + 1 < n) and V(r).  kind 0 = scores, 1 = values.
__device__ __forceinline__ void umma_phase(int ph, int n, int& kind, int& rec) {
  if (ph == 0) {
    kind = 0;
    rec = 0;
    return;
  }
  const int q = ph - 1, r = q >> 1;
  if ((q & 1) == 0 && r + 1 < n) {
    kind = 0;
    rec = r + 1;
  } else {
    kind = 1;
    rec = r;
  }
}

// loads issued where they stand (the compiler does not sink them to their use)
__device__ __forceinline__ uint32_t ldg_keep(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}
__device__ __forceinline__ uint32_t ldg_keep16(const void* p) {
  uint16_t r;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(p));
  return r;
}
__device__ __forceinline__ uint2 ldg_keep2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}
// words holding the 16-code unit u (coordinates 16 u .. 16 u + 15) of a packed row
template <int B>
__device__ __forceinline__ void load_unit(uint32_t (&w)[2], const uint8_t* row, int u) {
  if constexpr (B == 4) {
    const uint2 v = ldg_keep2(row + 8 * u);
    w[0] = v.x;
    w[1] = v.y;
  } else if constexpr (B == 2) {
    w[0] = ldg_keep(row + 4 * u);
  } else if constexpr (B == 1) {
    w[0] = ldg_keep16(row + 2 * u);
  } else {  // 6 bytes at 6u: the two words from 4-aligned (6u & ~3), still inside the row
    const uint32_t* a = reinterpret_cast<const uint32_t*>(row + ((6 * u) & ~3));
    w[0] = ldg_keep(a);
    w[1] = ldg_keep(a + 1);
  }
}
// codes 8 c .. 8 c + 7 (c = 0, 1) of the unit; sh = the unit's bit offset in w
// (nonzero only for 3-bit codes)
template <int B>
__device__ __forceinline__ uint32_t codes8(const uint32_t (&w)[2], int c, int sh) {
  if constexpr (B == 4) {
    return w[c];
  } else if constexpr (B == 3) {
    const int o = sh + 24 * c;
    return o < 32 ? __funnelshift_r(w[0], w[1], o) : (w[1] >> (o - 32));
  } else {
    return w[0] >> (8 * B * c);
  }
}

__device__ __forceinline__ void set_status(const AttnParams& p, int code) {
  if (p.status) atomicOr(p.status, code);
}

template <int KB, int VB>
__global__ void __launch_bounds__(kU512Threads, 1) attn_umma512_kernel(const __grid_constant__ AttnParams p) {
  constexpr int D = 512;
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
  U512Misc& ms = *reinterpret_cast<U512Misc*>(sm + kUMisc);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int l = blockIdx.z;
  int rem = blockIdx.y;
  const int hg = rem % p.n_hg;
  rem /= p.n_hg;
  const int kvh = rem % p.Hkv, b = rem / p.Hkv;
  const int split = blockIdx.x;
  const int GT = p.G / p.n_hg;  // <= 64
  const int h0 = kvh * p.G + hg * GT;
  const int lb = l * p.B + b;
  const int64_t qh0 = (int64_t)lb * p.Hq + h0;
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
  // record c of this unit (contiguous, or through the block table)
  const uint8_t* kl0 = p.krec + l * p.krec_ls;
  const uint8_t* vl0 = p.shared_kv ? kl0 : p.vrec + l * p.vrec_ls;
  auto krec_at = [&](int64_t c) {
    return kl0 + rec_offset(p.table, p.table_stride, p.rec_cap, p.Hkv, b, kvh, (int)c, p.krec_bytes);
  };
  auto vrec_at = [&](int64_t c) {
    return vl0 + rec_offset(p.table, p.table_stride, p.rec_cap, p.Hkv, b, kvh, (int)c, p.vrec_bytes);
  };

  // ---------------------------------------------------------------- set-up
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms.full[i], kUDeqWarps);
      mbar_init(&ms.empty[i], 1);
      mbar_init(&ms.s_full[i], 1);
    }
    mbar_init(&ms.p_full, kUSoftWarps);
    mbar_init(&ms.o_done, 1);
    mbar_init(&ms.fin, 1);
    ms.abort_ = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kUIssueWarp) tmem_alloc(&ms.tbase, 512);
  if (tid < 32) {
    const int e = tid & 15, bits = tid < 16 ? KB : VB;
    const float v = e < (1 << bits) ? (tid < 16 ? p.kc[e] : p.vc[e]) * 65536.f : 0.f;
    const __half h = __float2half_rn(v);
    const __half r = __float2half_rn(v - __half2float(h));
    (tid < 16 ? ms.ctab_k : ms.ctab_v)[e] = (uint32_t)__half_as_ushort(h) | ((uint32_t)__half_as_ushort(r) << 16);
  }
  if (tid >= 32 && tid < 64) {  // byte planes: table (tid - 32) / 16, plane ((tid - 32) / 4) % 4, word (tid - 32) % 4
    const int i = tid - 32, tb = i >> 4, pln = (i >> 2) & 3, wd = i & 3, bits = tb ? VB : KB;
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = 4 * wd + j;
      const float v = e < (1 << bits) ? (tb ? p.vc[e] : p.kc[e]) * 65536.f : 0.f;
      const __half h = __float2half_rn(v);
      const __half r = __float2half_rn(v - __half2float(h));
      const uint32_t hv = (pln < 2) ? __half_as_ushort(h) : __half_as_ushort(r);
      word |= ((hv >> (8 * (pln & 1))) & 0xFFu) << (8 * j);
    }
    (tb ? ms.plane_v : ms.plane_k)[pln][wd] = word;
  }
  if (tid < 64) ms.mst[tid] = -INFINITY;
  // q~ rows (warps 0-15, four heads each): lane holds coordinates 16 lane .. + 15
  if (warp < 16) {
    for (int hh = warp; hh < 64; hh += 16) {
      float x[16];
      if (hh < GT) {
        const uint16_t* qp = p.q + l * p.q_ls + b * p.q_bs + (int64_t)(h0 + hh) * D + lane * 16;
#pragma unroll
        for (int r = 0; r < 16; r += 2) {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(qp + r);
          x[r] = bf16_lo(w);
          x[r + 1] = bf16_hi(w);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          const int j = lane * 16 + r;
          if ((p.ksign[j >> 5] >> (j & 31)) & 1u) x[r] = -x[r];
        }
        fwht_regs<16>(x);
        fwht_lanes<16>(x, lane, 32);
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] *= inv_sqrt_dim<D>();
      } else {
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = 0.f;
      }
      float mx = 0.f;
#pragma unroll
      for (int r = 0; r < 16; ++r) mx = fmaxf(mx, fabsf(x[r]));
      mx = warp_max(mx);
      const int s = mx > 0.f ? 13 - exp_of(mx) : 0;
      const float sc = pow2i(s);
      if (lane == 0) ms.qsc[hh] = hh < GT ? p.sscale * pow2i(-16 - s) : 0.f;
      uint32_t hw[8], lw[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) split_f16x2(x[2 * e] * sc, x[2 * e + 1] * sc, hw[e], lw[e]);
      unsigned char* qc = sm + kUQ + (lane >> 2) * 16384;
      const int c16 = 2 * (lane & 3);
      *reinterpret_cast<uint4*>(qc + sw128_off(hh, c16)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4*>(qc + sw128_off(hh, c16 + 1)) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
      *reinterpret_cast<uint4*>(qc + sw128_off(64 + hh, c16)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      *reinterpret_cast<uint4*>(qc + sw128_off(64 + hh, c16 + 1)) = make_uint4(lw[4], lw[5], lw[6], lw[7]);
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tS = ms.tbase;        // scores: two buffers of 128 columns
  const uint32_t tO = ms.tbase + 256;  // O^T: 4 blocks x 64 columns
  volatile int* abort_f = &ms.abort_;

  if (warp == kUIssueWarp) {
    // ------------------------------------------------------------ MMA issue
    // Descriptors are built once; a byte offset o moves one by o / 16.
    if (lane == 0) {
      const uint32_t ra = smem_u32(sm + kURing);
      const uint64_t dQ = sdesc_sw128(smem_u32(sm + kUQ), 16, 1024);
      const uint64_t dP = sdesc_sw128(smem_u32(sm + kUP), 1024, 1024);
      const uint64_t dK0 = sdesc_sw128(ra, 16, 1024), dK1 = sdesc_sw128(ra + 32768, 16, 1024);
      const uint64_t dV0 = sdesc_sw128(ra, 16384, 1024), dV1 = sdesc_sw128(ra + 32768, 16384, 1024);
      constexpr uint32_t IS128 = idesc_f16(128, 128, false, false);
      constexpr uint32_t IS64 = idesc_f16(128, 64, false, false);
      constexpr uint32_t IV = idesc_f16(128, 64, true, true);
      uint32_t g = 0;
      for (int ph = 0; ph < 2 * n; ++ph) {
        int kind, rec;
        umma_phase(ph, n, kind, rec);
        if (kind == 0) {
          const uint32_t dS = tS + 128 * (rec & 1);
#pragma unroll 1
          for (int kc = 0; kc < 8; ++kc, ++g) {
            mbar_wait(&ms.full[g & 1], (g >> 1) & 1, abort_f);
            tc_fence_after();
            const uint64_t a = (g & 1) ? dK1 : dK0;
            const uint64_t bq = dQ + (uint64_t)(kc * 1024);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              umma_f16(dS, a + 2 * ks, bq + 2 * ks, IS128, (kc | ks) != 0);
              umma_f16(dS, a + 1024 + 2 * ks, bq + 2 * ks, IS64, 1);
            }
            umma_commit(&ms.empty[g & 1]);
          }
          umma_commit(&ms.s_full[rec & 1]);
        } else {
          mbar_wait(&ms.p_full, rec & 1, abort_f);  // P' of this record is in shared memory
          tc_fence_after();
#pragma unroll 1
          for (int st = 0; st < 8; ++st, ++g) {
            const int j = st >> 1, part = st & 1;
            mbar_wait(&ms.full[g & 1], (g >> 1) & 1, abort_f);
            tc_fence_after();
            const uint64_t a = (g & 1) ? dV1 : dV0;
            const uint32_t dO = tO + 64 * j;
            if (part == 0) {
#pragma unroll
              for (int ks = 0; ks < 8; ++ks) {
                umma_f16(dO, a + 128 * ks, dP + 128 * ks, IV, !(rec == 0 && ks == 0));
                umma_f16(dO, a + 128 * ks, dP + 1024 + 128 * ks, IV, 1);
              }
            } else {
#pragma unroll
              for (int ks = 0; ks < 8; ++ks) umma_f16(dO, a + 128 * ks, dP + 128 * ks, IV, 1);
            }
            umma_commit(&ms.empty[g & 1]);
          }
          umma_commit(&ms.o_done);
        }
      }
      umma_commit(&ms.fin);
    }
    __syncwarp();
  } else if (warp >= kUSoftWarps) {
    // ------------------------------------------------------------ dequantisation
    // Thread d owns token d / 4 and its 16-coordinate units u = 4 i + d % 4
    // (i = 0..7): unit i feeds score chunk i (coordinates 64 i + 16 (d % 4) ..)
    // and half i % 2 of value block i / 2, so the words loaded for a record
    // serve both of its passes.  Phases run in the order S(0), S(1), V(0),
    // S(2), V(1), ..., S(n-1), V(n-2), V(n-1) (scores one record ahead, into
    // alternating score buffers); each phase's words are loaded one phase ahead.
    const int d = tid - 32 * kUSoftWarps, tkn = d >> 2, sub = d & 3;
    const int shk = KB == 3 ? 16 * (sub & 1) : 0, shv = VB == 3 ? 16 * (sub & 1) : 0;
    uint32_t cur[8][2], nxt[8][2];
    auto load_phase = [&](uint32_t (&w)[8][2], int ph) {
      int kind, rec;
      umma_phase(ph, n, kind, rec);
      if (kind == 0) {
        const uint8_t* row = krec_at(c_begin + rec) + tkn * (D * KB / 8);
#pragma unroll
        for (int i = 0; i < 8; ++i) load_unit<KB>(w[i], row, 4 * i + sub);
      } else {
        const uint8_t* row = vrec_at(c_begin + rec) + tkn * (D * VB / 8);
#pragma unroll
        for (int i = 0; i < 8; ++i) load_unit<VB>(w[i], row, 4 * i + sub);
      }
    };
    uint32_t g = 0;  // stages handed over so far
    auto acquire = [&]() -> unsigned char* {
      const uint32_t slot = g & 1;
      mbar_wait(&ms.empty[slot], ((g >> 1) & 1) ^ 1, abort_f);
      return sm + kURing + slot * 32768;
    };
    auto release = [&]() {
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms.full[g & 1]);
      ++g;
    };
    load_phase(cur, 0);
    for (int ph = 0; ph < 2 * n; ++ph) {
      int kind, rec;
      umma_phase(ph, n, kind, rec);
      if (ph + 1 < 2 * n) load_phase(nxt, ph + 1);
      uint32_t pl[4][4];  // byte planes of this phase's codec (4-bit codes)
      if constexpr (KB == 4 || VB == 4) {
        const uint32_t(&src)[4][4] = kind == 0 ? ms.plane_k : ms.plane_v;
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int c = 0; c < 4; ++c) pl[a][c] = src[a][c];
      }
      if (kind == 0) {
        // score chunk i: row tkn, 16-byte chunks 2 sub, 2 sub + 1 of its hi and lo tiles
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          unsigned char* st = acquire();
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint4 hi, lo;
            if constexpr (KB == 4) {
              deq8_planes(codes8<KB>(cur[i], c, shk), pl, hi, lo);
            } else {
              deq8<KB>(codes8<KB>(cur[i], c, shk), ms.ctab_k, hi, lo);
            }
            const uint32_t o = sw128_off(tkn, 2 * sub + c);
            *reinterpret_cast<uint4*>(st + o) = hi;
            *reinterpret_cast<uint4*>(st + 16384 + o) = lo;
          }
          release();
        }
      } else {
        // value block j: unit 2 j + e -> half e, chunks 2 sub, 2 sub + 1
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            unsigned char* st = acquire();
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
              for (int c = 0; c < 2; ++c) {
                uint4 hi, lo;
                if constexpr (VB == 4) {
                  deq8_planes(codes8<VB>(cur[2 * j + e], c, shv), pl, hi, lo);
                } else {
                  deq8<VB>(codes8<VB>(cur[2 * j + e], c, shv), ms.ctab_v, hi, lo);
                }
                *reinterpret_cast<uint4*>(st + e * 16384 + sw128_off(tkn, 2 * sub + c)) = part ? lo : hi;
              }
            release();
          }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        cur[i][0] = nxt[i][0];
        cur[i][1] = nxt[i][1];
      }
    }
  } else {
    // ------------------------------------------------------------ softmax, epilogue
    const int q = warp;  // TMEM lane quarter
    const int tok = 32 * q + lane;
    const uint32_t lrow = (uint32_t)(32 * q) << 16;
    float lacc[2] = {0.f, 0.f};  // softmax denominators of heads lane and 32 + lane over this warp's tokens
    int kx = 127;                // P' scale exponent (only decreases)
    auto norm_at = [&](bool key, int rec) {
      const uint8_t* r = key ? krec_at(c_begin + rec) + p.k_off_norm : vrec_at(c_begin + rec) + p.v_off_norm;
      return __ldg(reinterpret_cast<const float*>(r) + tok);
    };
    // logits of heads 32 hh .. 32 hh + 31 of this token (-inf past the group)
    auto logits = [&](uint32_t tSr, int hh, float nk, float (&t)[32]) {
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        uint32_t a[16], c[16];
        tmem_ld16(tSr + lrow + 32 * hh + 16 * x, a);
        tmem_ld16(tSr + lrow + 64 + 32 * hh + 16 * x, c);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int h = 32 * hh + 16 * x + i;
          t[16 * x + i] = h < GT ? (__uint_as_float(a[i]) + __uint_as_float(c[i])) * nk * ms.qsc[h] : -INFINITY;
        }
      }
      if (p.scap > 0.f) {
#pragma unroll
        for (int i = 0; i < 32; ++i) t[i] = soft_cap(t[i], p.scap, p.iscap);
      }
    };
    float nk = norm_at(true, 0);
    float nv = norm_at(false, 0);
    for (int r = 0; r < n; ++r) {
      float nk1 = 0.f, nv1 = 0.f;
      if (r + 1 < n) {
        nk1 = norm_at(true, r + 1);
        nv1 = norm_at(false, r + 1);
      }
      mbar_wait(&ms.s_full[r & 1], (r >> 1) & 1, abort_f);
      tc_fence_after();
      const uint32_t tSr = tS + 128 * (r & 1);
      bool need = nv > 0.f && 6 - exp_of(nv) < kx;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        float t[32];
        logits(tSr, hh, nk, t);
#pragma unroll
        for (int i = 0; i < 32; ++i) need |= t[i] > ms.mst[32 * hh + i] + 8.f;
      }
      bool owaited = false;
      if (bar_or(1, 32 * kUSoftWarps, need)) {
        // new running max per head (moves only past the 2^8 margin), rescale
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          float t[32];
          logits(tSr, hh, nk, t);
          ms.red[q][32 * hh + lane] = transpose_reduce<true>(t, lane);
        }
        const float vm = warp_max(nv);
        if (lane == 0) ms.vmx[q] = vm;
        bar_sync(1, 32 * kUSoftWarps);
        if (q == 0) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int h = 32 * hh + lane;
            const float mx = fmaxf(fmaxf(ms.red[0][h], ms.red[1][h]), fmaxf(ms.red[2][h], ms.red[3][h]));
            const float mo = ms.mst[h];
            const float mn = mx > mo + 8.f ? mx : mo;
            ms.red[0][h] = mo == -INFINITY ? 0.f : exp2f(mo - mn);
            ms.mst[h] = mn;
          }
        }
        const float vmax = fmaxf(fmaxf(ms.vmx[0], ms.vmx[1]), fmaxf(ms.vmx[2], ms.vmx[3]));
        int kn = kx;
        if (vmax > 0.f) kn = min(kx, 6 - exp_of(vmax));
        const float gamma = pow2i(kn - kx);
        bar_sync(1, 32 * kUSoftWarps);
        lacc[0] *= ms.red[0][lane];
        lacc[1] *= ms.red[0][32 + lane];
        if (r > 0) {
          mbar_wait(&ms.o_done, (r - 1) & 1, abort_f);
          tc_fence_after();
          owaited = true;
#pragma unroll 1
          for (int j = 0; j < 8; ++j) {  // block j / 2, heads 32 (j % 2) ..
            const uint32_t col = 64 * (j >> 1) + 32 * (j & 1);
            uint32_t o[32];
            tmem_ld32(tO + lrow + col, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              o[i] = __float_as_uint(__uint_as_float(o[i]) * (ms.red[0][32 * (j & 1) + i] * gamma));
            tmem_st32(tO + lrow + col, o);
          }
          tmem_st_wait();
        }
        kx = kn;
      }
      if (r > 0 && !owaited) {
        mbar_wait(&ms.o_done, (r - 1) & 1, abort_f);
        tc_fence_after();
      }
      // P' (hi, lo): row `tok` of the MN-major operand, heads in 16-byte chunks
      const float vs = nv * pow2i(kx);
      unsigned char* pb = sm + kUP;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        float t[32];
        logits(tSr, hh, nk, t);
#pragma unroll
        for (int i = 0; i < 32; ++i) t[i] = t[i] == -INFINITY ? 0.f : exp2f(t[i] - ms.mst[32 * hh + i]);
        uint32_t ph[16], pl[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) split_f16x2(t[2 * i] * vs, t[2 * i + 1] * vs, ph[i], pl[i]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t o = sw128_off(tok, 4 * hh + k);
          *reinterpret_cast<uint4*>(pb + o) = make_uint4(ph[4 * k], ph[4 * k + 1], ph[4 * k + 2], ph[4 * k + 3]);
          *reinterpret_cast<uint4*>(pb + 16384 + o) = make_uint4(pl[4 * k], pl[4 * k + 1], pl[4 * k + 2], pl[4 * k + 3]);
        }
        lacc[hh] += transpose_reduce<false>(t, lane);
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms.p_full);
      nk = nk1;
      nv = nv1;
    }
    mbar_wait(&ms.o_done, (n - 1) & 1, abort_f);
    tc_fence_after();
    // the split's partial: softmax denominators and O^T (rotated basis)
    ms.red[q][lane] = lacc[0];
    ms.red[q][32 + lane] = lacc[1];
    bar_sync(1, 32 * kUSoftWarps);
    const float un = pow2i(-16 - kx);
#pragma unroll 1
    for (int j = 0; j < 8; ++j) {
      const int hb = 32 * (j & 1);
      uint32_t o[32];
      tmem_ld32(tO + lrow + 64 * (j >> 1) + hb, o);
      tmem_ld_wait();
      float* dst = p.ws_acc + ((qh0 + hb) * p.S + split) * D + 128 * (j >> 1) + tok;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (hb + i < GT) dst[(int64_t)i * p.S * D] = __uint_as_float(o[i]) * un;
    }
    if (q == 0) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int h = 32 * hh + lane;
        if (h < GT) {
          float* ml = p.ws_ml + ((qh0 + h) * p.S + split) * 2;
          ml[0] = ms.mst[h];
          ml[1] = ms.red[0][h] + ms.red[1][h] + ms.red[2][h] + ms.red[3][h];
        }
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == kUIssueWarp) {
    // every MMA has completed (drain bounded independently of the abort flag)
    volatile int drain = 0;
    mbar_wait(&ms.fin, 0, &drain);
    tc_fence_after();
    tmem_dealloc(ms.tbase, 512);
    if (lane == 0 && (*abort_f || drain)) set_status(p, 1);
  }
}

template <int KB, int VB>
cudaError_t attn_umma512_launch_t(const AttnParams& p, dim3 grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(attn_umma512_kernel<KB, VB>, cudaFuncAttributeMaxDynamicSharedMemorySize, kUSmem);
  if (e != cudaSuccess) return e;
  attn_umma512_kernel<KB, VB><<<grid, kU512Threads, kUSmem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace tq
