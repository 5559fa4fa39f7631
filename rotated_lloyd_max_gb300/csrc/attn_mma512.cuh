// Decode attention on the tensor cores at head dim 512 (many query heads per kv head,
// e.g. MQA with 64 query heads): decode attention over the compressed records
// of codecs without outlier side lists.
//
// Same arithmetic as the head-dim 64/128 kernel (f16 hi/lo operand splits,
// three mma.sync per product, f32 accumulation; pair-table dequantisation;
// centroids x 2^16, q~ x 2^s per head, P' x 2^k), organised for d = 512,
// where one warp cannot hold a whole output row of 8 heads:
//  * a CTA is 8 warps and one group of 8 query heads; per record (128 tokens)
//    warp w scores tokens 16w .. 16w+15 against all 512 coordinates (score
//    fragment column 2t+e <-> coordinate 128 t + 4 kk + e, +2 for column
//    2t+8+e, kk = 0..31; query fragments read from shared memory);
//  * the logits go to shared memory; warp 0 turns them into the record's
//    running max, rescale factors and softmax denominator for the CTA;
//  * warp w then accumulates output coordinates 64w .. 64w+63 over all 128
//    tokens (value fragment row g <-> coordinate 64 w + 8 g + 2 mc, row g+8
//    <-> +1; P' fragments built from the shared logits), so every warp shares
//    one softmax state and writes its own slice of the split's partial.
#pragma once

#include "attn_mma.cuh"

namespace tq {

constexpr int kT512 = 256;  // threads of the d-512 kernel (8 warps)

__device__ __forceinline__ void cta256_copy_async(void* smem, const void* gmem, int bytes) {
  char* s = (char*)smem;
  const char* gp = (const char*)gmem;
  for (int off = threadIdx.x * 16; off < bytes; off += kT512 * 16) cp_async16(s + off, gp + off);
}

template <int KB, int VB, int NT>
__global__ void __launch_bounds__(kT512, 1) attn_mma512_kernel(const __grid_constant__ AttnParams p) {
  constexpr int HN = 8 * NT;  // query heads per CTA (NT n-tiles of 8)
  constexpr int D = 512, KS = 32, KR = 128;
  constexpr int KNB = KR * KB;                 // bits of a lane's score run (multiple of 32)
  constexpr int VNB = 8 * VB;                  // bits of a lane group's value run (8 codes)
  constexpr int VNW = (VNB + 31) / 32;
  constexpr bool VAL = (VNB % 32) == 0;
  constexpr int FW = VIdx<VB>::FW;
  constexpr int ZW = (VB == 3) ? 2 * VNW : VNW;
  constexpr int EK = 1 << (2 * KB), EV = VIdx<VB>::ENTRIES;
  constexpr int KP_OFF = 0, VP_OFF = EK * 128;
  extern __shared__ __align__(128) unsigned char sm[];
  uint4* qfrag = reinterpret_cast<uint4*>(sm + p.sm_logit);   // [32 k-steps][NT][32 lanes]
  uint2* cent = reinterpret_cast<uint2*>(sm + p.sm_slot);     // [32] centroid halves x 2^16
  float* lg_s = reinterpret_cast<float*>(sm + p.sm_red);      // [128 tokens][HN heads] logits
  float* st_s = reinterpret_cast<float*>(sm + p.sm_corr);     // m[16] | scale[16] | l[16] | kx
  unsigned char* mainb = sm + p.sm_main;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int l = blockIdx.z;
  int rem = blockIdx.y;
  const int hg = rem % p.n_hg;
  rem /= p.n_hg;
  const int kvh = rem % p.Hkv, b = rem / p.Hkv;
  const int split = blockIdx.x;
  const int GT = p.G / p.n_hg;
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
  auto stage = [&](int i) { return mainb + (i & 1) * p.sm_stage; };
  auto issue_main = [&](int i) {
    if (i < n) {
      const int64_t c = c_begin + i;
      cta256_copy_async(stage(i), krec_at(c), p.k_main);
      if (!p.shared_kv) cta256_copy_async(stage(i) + p.k_main, vrec_at(c), p.v_main);
    }
    cp_async_commit();
  };
  issue_main(0);

  // ---- q~ of the CTA's heads into the second staging buffer (free until
  // record 1 is issued), rows >= GT zero
  // [HN heads][4 lane runs of 128, padded to 129][+1]: coordinate c of head h at
  // h*516 + (c/128)*129 + c%128, so the 32 lanes' runs start in 32 different banks
  float* qf = reinterpret_cast<float*>(stage(1));
  auto qidx = [](int h, int c) { return h * 516 + (c >> 7) * 129 + (c & 127); };
  {
    constexpr int R = D / 32;
    for (int hh = warp; hh < HN; hh += 8) {
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
    }
  }
  if (tid < 32) {
    const float v = (tid < 16 ? p.kc[tid] : p.vc[tid - 16]) * 65536.f;
    const __half h = __float2half_rn(v);
    const __half r = __float2half_rn(v - __half2float(h));
    cent[tid] = make_uint2(__half_as_ushort(h), __half_as_ushort(r));
  }
  if (tid < 16) {
    st_s[tid] = -INFINITY;  // m
    st_s[32 + tid] = 0.f;   // l
  }
  __syncthreads();
  for (int i = tid; i < EK * 16; i += kT512) {
    const int e = i >> 4;
    const uint2 a = cent[e & ((1 << KB) - 1)], c = cent[e >> KB];
    *reinterpret_cast<uint2*>(sm + KP_OFF + i * 8) = make_uint2(__byte_perm(a.x, c.x, 0x5410), __byte_perm(a.y, c.y, 0x5410));
  }
  for (int i = tid; i < EV * 16; i += kT512) {
    const int e = i >> 4;
    const int c0 = e & ((1 << FW) - 1), c1 = e >> FW;
    uint2 v = make_uint2(0u, 0u);
    if (c0 < (1 << VB) && c1 < (1 << VB)) {
      const uint2 a = cent[16 + c0], c = cent[16 + c1];
      v = make_uint2(__byte_perm(a.x, c.x, 0x5410), __byte_perm(a.y, c.y, 0x5410));
    }
    *reinterpret_cast<uint2*>(sm + VP_OFF + i * 8) = v;
  }
  // query fragments (head 8 nt + g, lane t's coordinates), scaled per head
  float fq[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const float* qrow = qf + qidx(8 * nt + g, KR * t);
    float mx = 0.f;
#pragma unroll 8
    for (int j = 0; j < KR; ++j) mx = fmaxf(mx, fabsf(qrow[j]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const int s = mx > 0.f ? 13 - exp_of(mx) : 0;
    const float sc = pow2i(s);
    for (int kk = warp; kk < KS; kk += 8) {
      uint4 f;
      split_f16x2(qrow[4 * kk] * sc, qrow[4 * kk + 1] * sc, f.x, f.z);
      split_f16x2(qrow[4 * kk + 2] * sc, qrow[4 * kk + 3] * sc, f.y, f.w);
      qfrag[(kk * NT + nt) * 32 + lane] = f;
    }
    const int s0 = __shfl_sync(0xffffffffu, s, 4 * (2 * t));
    const int s1 = __shfl_sync(0xffffffffu, s, 4 * (2 * t + 1));
    fq[nt][0] = pow2i(-s0 - 16);
    fq[nt][1] = pow2i(-s1 - 16);
  }
  // head of element e of n-tile nt in the score / value fragments: 8 nt + 2t + (e & 1)
  const uint32_t loff = (lane & 15) * 8;
  auto kpair_at = [&](uint32_t o) { return *reinterpret_cast<const uint2*>(sm + KP_OFF + o); };
  auto vpair_at = [&](uint32_t o) { return *reinterpret_cast<const uint2*>(sm + VP_OFF + o); };
  float acc[4][NT][4];
#pragma unroll
  for (int mc = 0; mc < 4; ++mc)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mc][nt][e] = 0.f;
  int kx = 127;  // P' f16 scale exponent (CTA-wide, only decreases)
  const int rbk = D * KB / 8, rbv = D * VB / 8;

  for (int i = 0; i < n; ++i) {
    cp_async_wait<0>();
    __syncthreads();  // record i is in (q~ consumed), the previous record is done with
    issue_main(i + 1);
    const unsigned char* st = stage(i);
    const float* knorm = reinterpret_cast<const float*>(st + p.k_off_norm);
    const unsigned char* vbase = p.shared_kv ? st : st + p.k_main;
    const unsigned char* vcodes = vbase;
    const float* vnorm = reinterpret_cast<const float*>(vbase + p.v_off_norm);

    // ---- scores of tokens 16 warp + g (elements 0, 1) and + 8 (2, 3)
    {
      const unsigned char* r0 = st + (16 * warp + g) * rbk;
      const unsigned char* r1 = r0 + 8 * rbk;
      // hi.hi, hi.lo and lo.hi in separate accumulators: independent MMA chains
      float cc[NT][4], cl[NT][4], ch[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) cc[nt][e] = cl[nt][e] = ch[nt][e] = 0.f;
#pragma unroll 2
      for (int q8 = 0; q8 < 4; ++q8) {  // 8 k-steps = 32 coordinates of the lane's run
        constexpr int PB = 32 * KB;
        uint32_t w0[PB / 32], w1[PB / 32];
        load_run<PB, true>(r0, KNB * t + PB * q8, w0);
        load_run<PB, true>(r1, KNB * t + PB * q8, w1);
#pragma unroll
        for (int k8 = 0; k8 < 8; ++k8) {
          const int kk = 8 * q8 + k8;
          uint32_t ah[4], al[4];
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int off = (4 * k8 + 2 * hf) * KB;
            const uint2 e0 = kpair_at(pair_off(w0, off, 2 * KB, loff));
            const uint2 e1 = kpair_at(pair_off(w1, off, 2 * KB, loff));
            ah[2 * hf] = e0.x;
            al[2 * hf] = e0.y;
            ah[2 * hf + 1] = e1.x;
            al[2 * hf + 1] = e1.y;
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint4 f = qfrag[(kk * NT + nt) * 32 + lane];
            mma_f16(cc[nt], ah, f.x, f.y);
            mma_f16(cl[nt], ah, f.z, f.w);
            mma_f16(ch[nt], al, f.x, f.y);
          }
        }
      }
      const int ta = 16 * warp + g, tb = ta + 8;
      const float fa = knorm[ta] * p.sscale, fb = knorm[tb] * p.sscale;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int h = 8 * nt + 2 * t;
        const bool v0 = h < GT, v1 = h + 1 < GT;
        float x[4] = {v0 ? (cc[nt][0] + cl[nt][0] + ch[nt][0]) * fq[nt][0] * fa : -INFINITY,
                      v1 ? (cc[nt][1] + cl[nt][1] + ch[nt][1]) * fq[nt][1] * fa : -INFINITY,
                      v0 ? (cc[nt][2] + cl[nt][2] + ch[nt][2]) * fq[nt][0] * fb : -INFINITY,
                      v1 ? (cc[nt][3] + cl[nt][3] + ch[nt][3]) * fq[nt][1] * fb : -INFINITY};
        if (p.scap > 0.f) {
#pragma unroll
          for (int e = 0; e < 4; ++e) x[e] = soft_cap(x[e], p.scap, p.iscap);
        }
        lg_s[ta * HN + h] = x[0];
        lg_s[ta * HN + h + 1] = x[1];
        lg_s[tb * HN + h] = x[2];
        lg_s[tb * HN + h + 1] = x[3];
      }
    }
    __syncthreads();
    // ---- warp w: heads w (and w + 8): max over the record (lane: tokens
    // lane + 32j), lazy rescale (only when a logit passes the max by 2^8),
    // softmax denominator; and the P' scale exponent from the norms
    {
      const float vmax = warp_max(fmaxf(fmaxf(vnorm[lane], vnorm[32 + lane]), fmaxf(vnorm[64 + lane], vnorm[96 + lane])));
      int kn = kx;
      if (vmax > 0.f) kn = min(kx, 6 - exp_of(vmax));
      const float gamma = pow2i(kn - kx);
#pragma unroll
      for (int hw = warp; hw < HN; hw += 8) {
        float lv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) lv[j] = lg_s[(lane + 32 * j) * HN + hw];
        const float mx = warp_max(fmaxf(fmaxf(lv[0], lv[1]), fmaxf(lv[2], lv[3])));
        const float mo = st_s[hw];
        const float mn = mx > mo + 8.f ? mx : mo;
        const float alpha = (mn == mo || mo == -INFINITY) ? (mo == -INFINITY ? 0.f : 1.f) : exp2f(mo - mn);
        float ls = 0.f;
        if (mn != -INFINITY) {
#pragma unroll
          for (int j = 0; j < 4; ++j) ls += exp2f(lv[j] - mn);
        }
        ls = warp_sum(ls);
        __syncwarp();
        if (lane == 0) {
          st_s[hw] = mn;
          st_s[16 + hw] = (mo == -INFINITY ? 1.f : alpha) * gamma;  // acc rescale (acc is 0 before the first record)
          st_s[32 + hw] = st_s[32 + hw] * alpha + ls;
        }
      }
      if (tid == 0) st_s[48] = __int_as_float(kn);
    }
    __syncthreads();
    kx = __float_as_int(st_s[48]);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float s0 = st_s[16 + 8 * nt + 2 * t], s1 = st_s[16 + 8 * nt + 2 * t + 1];
#pragma unroll
      for (int mc = 0; mc < 4; ++mc) {
        acc[mc][nt][0] *= s0;
        acc[mc][nt][1] *= s1;
        acc[mc][nt][2] *= s0;
        acc[mc][nt][3] *= s1;
      }
    }
    // ---- values: output coordinates 64 warp + 8 g + 2 mc (+1), all 128 tokens
    {
      const float psc = pow2i(kx);
#pragma unroll 2
      for (int ks = 0; ks < 8; ++ks) {
        const int tk = 16 * ks + 2 * t;
        uint32_t pbh[NT][2], pbl[NT][2];  // P'^T fragments of heads 8 nt + g
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int hg2 = 8 * nt + g;
          const float mg = st_s[hg2];
          float pp[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int tok = tk + (r & 1) + 8 * (r >> 1);
            const float lgv = lg_s[tok * HN + hg2];
            pp[r] = (hg2 < GT && lgv != -INFINITY) ? exp2f(lgv - mg) * vnorm[tok] * psc : 0.f;
          }
          split_f16x2(pp[0], pp[1], pbh[nt][0], pbl[nt][0]);
          split_f16x2(pp[2], pp[3], pbh[nt][1], pbl[nt][1]);
        }
        uint32_t r0[VNW], r1[VNW], r2[VNW], r3[VNW];
        const int voff = (64 * warp + 8 * g) * VB;
        load_run<VNB, VAL>(vcodes + tk * rbv, voff, r0);
        load_run<VNB, VAL>(vcodes + (tk + 1) * rbv, voff, r1);
        load_run<VNB, VAL>(vcodes + (tk + 8) * rbv, voff, r2);
        load_run<VNB, VAL>(vcodes + (tk + 9) * rbv, voff, r3);
        uint32_t ze01[ZW], zo01[ZW], ze23[ZW], zo23[ZW];
        v_pair_words<VB, VNW>(r0, r1, ze01, zo01);
        v_pair_words<VB, VNW>(r2, r3, ze23, zo23);
#pragma unroll
        for (int mc = 0; mc < 4; ++mc) {
          const int off = mc * 2 * FW;
          const uint2 e0 = vpair_at(pair_off(ze01, off, 2 * FW, loff));
          const uint2 e1 = vpair_at(pair_off(zo01, off, 2 * FW, loff));
          const uint2 e2 = vpair_at(pair_off(ze23, off, 2 * FW, loff));
          const uint2 e3 = vpair_at(pair_off(zo23, off, 2 * FW, loff));
          const uint32_t ah[4] = {e0.x, e1.x, e2.x, e3.x};
          const uint32_t al[4] = {e0.y, e1.y, e2.y, e3.y};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma_f16(acc[mc][nt], ah, pbh[nt][0], pbh[nt][1]);
            mma_f16(acc[mc][nt], ah, pbl[nt][0], pbl[nt][1]);
            mma_f16(acc[mc][nt], al, pbh[nt][0], pbh[nt][1]);
          }
        }
      }
    }
  }
  cp_async_wait<0>();
  // ---- the split's partial: this warp's coordinate slice, the CTA's (m, l)
  const float un = pow2i(-16 - kx);
#pragma unroll
  for (int mc = 0; mc < 4; ++mc)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = 64 * warp + 8 * g + 2 * mc + (e >> 1), h = 8 * nt + 2 * t + (e & 1);
        if (h < GT) p.ws_acc[((qh0 + h) * p.S + split) * D + j] = acc[mc][nt][e] * un;
      }
  if (tid < GT) {
    float* ml = p.ws_ml + ((qh0 + tid) * p.S + split) * 2;
    ml[0] = st_s[tid];
    ml[1] = st_s[32 + tid];
  }
}

template <int KB, int VB, int NT>
cudaError_t attn_mma512_launch_nt(const AttnParams& p, dim3 grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(attn_mma512_kernel<KB, VB, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       p.sm_total);
  if (e != cudaSuccess) return e;
  attn_mma512_kernel<KB, VB, NT><<<grid, kT512, p.sm_total, s>>>(p);
  return cudaGetLastError();
}
// 16 heads per CTA (two n-tiles) when the group holds more than 8
template <int KB, int VB>
cudaError_t attn_mma512_launch_t(const AttnParams& p, dim3 grid, cudaStream_t s) {
  return (p.G / p.n_hg > 8) ? attn_mma512_launch_nt<KB, VB, 2>(p, grid, s) : attn_mma512_launch_nt<KB, VB, 1>(p, grid, s);
}

}  // namespace tq
