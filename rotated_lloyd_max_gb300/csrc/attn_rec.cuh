// Decode attention over the compressed records (head dims 64 and 128),
// warp-local variant.
//
// Dense splits of the same call (tail tokens, bf16 layers) run the general
// dense path (attn_dense_split) inside this launch.
// Same arithmetic as attn.cuh (q~ = H(s_k . q)/sqrt(d) once per CTA; a record
// token scores as n_i * q~ . c[codes] from a shared-memory LUT; values
// accumulate p_i n_i yhat_i in the rotated basis), organised so that a record
// costs one CTA barrier:
//  * the CTA stages records global -> shared with cp.async in a 3-deep ring;
//    warps 0 and 1 turn a record's per-slot outlier counts into prefix sums and
//    fetch just the used entries, one record ahead;
//  * each warp owns 32 of the record's 128 tokens end to end: scores (a lane
//    holds 4 tokens x one 32-coordinate slice, so a q~ load serves 4 tokens,
//    then a transposed shuffle reduction leaves each lane with one token's
//    logits), an online softmax whose running max only moves when a logit
//    exceeds it by 2^8 (warp vote), and the value accumulation (a lane holds 4
//    coordinates x GT heads in registers);
//  * outlier entries are applied as deltas (stored value - centroid): on the
//    logits by the token's own lane, on the values through per-warp shared
//    integer atomics in a fixed-point buffer (scaled per record by the warp's
//    largest weight; integer adds retire about four times faster than f32
//    ones), folded into the lanes' accumulators after each record;
//  * at the end the 4 warps' (m, l, acc) are merged in shared memory into the
//    split's partial.
#pragma once

#include "attn.cuh"

namespace tq {

template <int D, int GT>
struct RCfg {
  static constexpr int SL = D / 32;          // lanes per token in the score phase
  static constexpr int TPL = SL;             // tokens per lane in the score phase
  static constexpr int QR = 32 / SL;         // token rows per warp in the score phase
  static constexpr int GTP = (GT == 6) ? 8 : GT;
  static constexpr int GH = (GT + 1) / 2;
  static constexpr int QPAD = GTP < 4 ? GTP : 4;
  static constexpr int QS = 32 * GTP + QPAD;  // floats per slice of q~
  static constexpr int LPT = D / 4;           // value phase: lanes per token
  static constexpr int TLW = 32 / LPT;        // value phase: token lanes per warp
};

// Transposed reduction of a[TPL][GH] over the SL lanes of a token group:
// afterwards lane s of the group holds the full sums of its token s.
template <int SL, int GH>
__device__ __forceinline__ void reduce_transpose(float2 (&a)[SL][GH], int s, float2 (&out)[GH]) {
  if constexpr (SL == 4) {
    const bool h1 = (s >> 1) & 1, h0 = s & 1;
    float2 b[2][GH];
#pragma unroll
    for (int kk = 0; kk < 2; ++kk)
#pragma unroll
      for (int k = 0; k < GH; ++k) {
        const float2 send = h1 ? a[kk][k] : a[2 + kk][k];
        const float2 keep = h1 ? a[2 + kk][k] : a[kk][k];
        float2 r;
        r.x = __shfl_xor_sync(0xffffffffu, send.x, 2);
        r.y = __shfl_xor_sync(0xffffffffu, send.y, 2);
        b[kk][k] = add2(keep, r);
      }
#pragma unroll
    for (int k = 0; k < GH; ++k) {
      const float2 send = h0 ? b[0][k] : b[1][k];
      const float2 keep = h0 ? b[1][k] : b[0][k];
      float2 r;
      r.x = __shfl_xor_sync(0xffffffffu, send.x, 1);
      r.y = __shfl_xor_sync(0xffffffffu, send.y, 1);
      out[k] = add2(keep, r);
    }
  } else {  // SL == 2
    const bool h0 = s & 1;
#pragma unroll
    for (int k = 0; k < GH; ++k) {
      const float2 send = h0 ? a[0][k] : a[1][k];
      const float2 keep = h0 ? a[1][k] : a[0][k];
      float2 r;
      r.x = __shfl_xor_sync(0xffffffffu, send.x, 1);
      r.y = __shfl_xor_sync(0xffffffffu, send.y, 1);
      out[k] = add2(keep, r);
    }
  }
}

// Score partials of TPL tokens x one 32-coordinate slice.
template <int B, int GT, int GTP, int TPL>
__device__ __forceinline__ void score_tokens(const unsigned char* kcodes, int rb, const int (&tok)[TPL],
                                             int slice, const float* qs, const float* lut,
                                             float2 (&a)[TPL][(GT + 1) / 2]) {
  uint32_t w[TPL][B];
#pragma unroll
  for (int i = 0; i < TPL; ++i) load_words<B>(kcodes + tok[i] * rb + slice * 4 * B, w[i]);
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    float2 q[(GT + 1) / 2];
    load_heads<GT>(qs + r * GTP, q);
#pragma unroll
    for (int i = 0; i < TPL; ++i) {
      const float cv = lut[code_of<B>(w[i], r)];
#pragma unroll
      for (int k = 0; k < (GT + 1) / 2; ++k) a[i][k] = fma2(make_float2(cv, cv), q[k], a[i][k]);
    }
  }
}

// Value accumulation of the warp's tokens tl, tl + TLW, ... < 32 for the
// lane's 4 coordinates 4g..4g+3.
template <int B, int GT, int GTP, int TLW>
__device__ __forceinline__ void pv_tokens(const unsigned char* vrows, int rb, const float* pw,
                                          const float* lut, int g, int tl,
                                          float2 (&acc)[4][(GT + 1) / 2]) {
  const int bit0 = 4 * g * B, wi = bit0 >> 5, sh = bit0 & 31;
#pragma unroll 4
  for (int t = tl; t < 32; t += TLW) {
    const uint32_t* row = reinterpret_cast<const uint32_t*>(vrows + t * rb);
    uint32_t v;
    if constexpr (B == 3) {
      v = __funnelshift_r(row[wi], row[wi + 1], sh);
    } else {
      v = row[wi] >> sh;
    }
    float2 pp[(GT + 1) / 2];
    load_heads<GT>(pw + t * GTP, pp);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float val = lut[(v >> (c * B)) & ((1u << B) - 1u)];
#pragma unroll
      for (int k = 0; k < (GT + 1) / 2; ++k) acc[c][k] = fma2(make_float2(val, val), pp[k], acc[c][k]);
    }
  }
}

__device__ __forceinline__ uint32_t code_in_row(const unsigned char* row, int idx, int b) {
  const uint32_t* r = reinterpret_cast<const uint32_t*>(row);
  const int bit = idx * b;
  return __funnelshift_r(r[bit >> 5], r[(bit >> 5) + 1], bit & 31) & ((1u << b) - 1u);
}

template <int D, int GT>
__global__ void __launch_bounds__(kThreads, (GT == 2 || GT == 4) ? 5 : (GT >= 8 ? 3 : 4)) attn_rec_kernel(const __grid_constant__ AttnParams p) {
  using C = RCfg<D, GT>;
  constexpr int GTP = C::GTP, GH = C::GH, SL = C::SL, TPL = C::TPL, QR = C::QR, LPT = C::LPT, TLW = C::TLW;
  extern __shared__ __align__(128) unsigned char sm[];
  float* qv = reinterpret_cast<float*>(sm + p.sm_q);
  float* lutk = reinterpret_cast<float*>(sm + p.sm_lut);
  float* lutv = lutk + 16;
  float* pbuf = reinterpret_cast<float*>(sm + p.sm_logit);  // [4][32][GTP]
  int* corr = reinterpret_cast<int*>(sm + p.sm_corr);       // [4][GTP][D] fixed point (head-major: atomics on random coordinates spread over the banks)
  unsigned char* mainb = sm + p.sm_main;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int l = blockIdx.z;
  int rem = blockIdx.y;
  const int hg = rem % p.n_hg;
  rem /= p.n_hg;
  const int kvh = rem % p.Hkv, b = rem / p.Hkv;
  const int split = blockIdx.x + p.split_base;
  const int h0 = kvh * p.G + hg * GT;
  const int lb = l * p.B + b;
  const int64_t qh0 = (int64_t)lb * p.Hq + h0;
  // a split is a run of whole records, or of dense tokens (a tail ring or a
  // bf16 layer) handled by the warp-local dense path of the same launch
  const bool dense = split >= p.Sc;
  int t_begin, t_end;
  if (dense) {
    const int len = min(p.tail_len ? p.tail_len[lb] : 0, p.tail_cap);
    t_begin = (split - p.Sc) * p.tps;
    t_end = min(t_begin + p.tps, len);
  } else {
    const int nch = min(p.n_chunks ? p.n_chunks[lb] : 0, p.rec_limit);
    t_begin = split * p.cps;
    t_end = min(t_begin + p.cps, nch);
  }
  if (t_begin >= t_end) {
    if (tid < GT) {
      float* ml = p.ws_ml + ((qh0 + tid) * p.S + split) * 2;
      ml[0] = -INFINITY;
      ml[1] = 0.f;
    }
    return;
  }
  const int n = t_end - t_begin;
  // record c of this unit (contiguous, or through the block table)
  const uint8_t* kl0 = p.krec + l * p.krec_ls;
  const uint8_t* vl0 = p.shared_kv ? kl0 : p.vrec + l * p.vrec_ls;
  auto krec_at = [&](int64_t c) {
    return kl0 + rec_offset(p.table, p.table_stride, p.rec_cap, p.Hkv, b, kvh, (int)c, p.krec_bytes);
  };
  auto vrec_at = [&](int64_t c) {
    return vl0 + rec_offset(p.table, p.table_stride, p.rec_cap, p.Hkv, b, kvh, (int)c, p.vrec_bytes);
  };
  const int kcap = p.kcap, vcap = p.shared_kv ? p.kcap : p.vcap;
  const bool kout = p.kout && !dense, vout = p.vout && !dense;
  auto stage = [&](int i) { return mainb + (i & 1) * p.sm_stage; };
  auto issue_main = [&](int i) {
    if (i < n) {
      const int64_t c = t_begin + i;
      cta_copy_async(stage(i), krec_at(c), p.k_main);
      if (!p.shared_kv) cta_copy_async(stage(i) + p.k_main, vrec_at(c), p.v_main);
    }
    cp_async_commit();
  };
  // the first record goes out before the query work so its latency overlaps it
  if (!dense) issue_main(0);

  // ---- query: load, rotate, store as [slice][32][GTP]
  for (int hh = warp; hh < GT; hh += 4) {
    constexpr int R = D / 32;
    const uint16_t* qp = p.q + l * p.q_ls + b * p.q_bs + (int64_t)(h0 + hh) * D + lane * R;
    float x[R];
#pragma unroll
    for (int r = 0; r < R; r += 2) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(qp + r);
      x[r] = bf16_lo(w);
      x[r + 1] = bf16_hi(w);
    }
    float f = 1.f;
    if (!dense) {  // records are scored against q~ = H(s_k . q)/sqrt(d)
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int j = lane * R + r;
        if ((p.ksign[j >> 5] >> (j & 31)) & 1u) x[r] = -x[r];
      }
      fwht_regs<R>(x);
      fwht_lanes<R>(x, lane, 32);
      f = inv_sqrt_dim<D>();
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int j = lane * R + r;
      qv[(j >> 5) * C::QS + (j & 31) * GTP + hh] = x[r] * f;
    }
  }
  if (GTP != GT)
    for (int i = tid; i < D; i += kThreads)
#pragma unroll
      for (int hh = GT; hh < GTP; ++hh) qv[(i >> 5) * C::QS + (i & 31) * GTP + hh] = 0.f;
  if (tid < 16) {
    lutk[tid] = p.kc[tid];
    lutv[tid] = p.vc[tid];
  }
  if (vout)
    for (int i = tid; i < 4 * D * GTP; i += kThreads) corr[i] = 0;

  // per-warp state
  float m_w[GT], l_ln[GT];
#pragma unroll
  for (int h = 0; h < GT; ++h) {
    m_w[h] = -INFINITY;
    l_ln[h] = 0.f;
  }
  float2 acc[4][GH];
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int k = 0; k < GH; ++k) acc[c][k] = make_float2(0.f, 0.f);
  const int q = lane / SL, s = lane % SL;          // score phase
  const int tl = lane / LPT, g = lane % LPT;       // value phase
  const int tloc = q + QR * s;                     // the token whose logits this lane ends with
  float* pw = pbuf + warp * 32 * GTP;
  int* cw = corr + warp * D * GTP;
  const int rbk = D * p.kb / 8, rbv = D * p.vb / 8;

  // Entry range of the lane's token in one stream's side list: a per-warp
  // prefix sum of the record's per-slot counts (lane j <-> slot warp*32 + j).
  auto token_entries = [&](const unsigned char* cnts, int cap, int& e_begin, int& e_cnt) {
    int base = 0;
    for (int u = 0; u < warp; ++u) base += cnts[u * 32 + lane];
#pragma unroll
    for (int m = 16; m; m >>= 1) base += __shfl_xor_sync(0xffffffffu, base, m);
    const int c = cnts[warp * 32 + lane];
    int inc = c;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, inc, m);
      if (lane >= m) inc += o;
    }
    e_begin = __shfl_sync(0xffffffffu, base + inc - c, tloc);
    e_cnt = __shfl_sync(0xffffffffu, c, tloc);
    e_cnt = max(0, min(e_cnt, cap - e_begin));
  };

  if (dense) {
    // ---- dense tokens, warp-local: a warp takes TW tokens per step (lane =
    // token x 32-coordinate slice for the scores, 4 coordinates for the
    // values), loaded straight from global memory with the next step's keys
    // in flight
    constexpr int TW = 32 / SL;
    const int tstart = p.tail_start ? ((p.tail_start[lb] % p.tail_cap) + p.tail_cap) % p.tail_cap : 0;
    const uint16_t* kt0 = p.ktail + l * p.tail_ls + (int64_t)(b * p.Hkv + kvh) * p.tail_cap * D;
    const uint16_t* vt0 = p.vtail + l * p.tail_ls + (int64_t)(b * p.Hkv + kvh) * p.tail_cap * D;
    const int steps = (n + 4 * TW - 1) / (4 * TW);
    auto kload = [&](int kk, uint4 (&kw)[4]) {
      const int t = t_begin + (kk * 4 + warp) * TW + q;
      if (kk < steps && t < t_end) {
        const int64_t slot = (tstart + t) % p.tail_cap;
        const uint4* src = reinterpret_cast<const uint4*>(kt0 + slot * D + s * 32);
#pragma unroll
        for (int k = 0; k < 4; ++k) kw[k] = __ldg(src + k);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) kw[k] = make_uint4(0u, 0u, 0u, 0u);
      }
    };
    uint4 kn[4];
    kload(0, kn);
    for (int kk = 0; kk < steps; ++kk) {
      uint4 kc[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) kc[k] = kn[k];
      const int tb = t_begin + (kk * 4 + warp) * TW;
      uint2 vc[TW / TLW];
#pragma unroll
      for (int j = 0; j < TW / TLW; ++j) {
        const int t = tb + tl + j * TLW;
        if (t < t_end) {
          const int64_t slot = (tstart + t) % p.tail_cap;
          vc[j] = __ldg(reinterpret_cast<const uint2*>(vt0 + slot * D + 4 * g));
        } else {
          vc[j] = make_uint2(0u, 0u);
        }
      }
      kload(kk + 1, kn);
      const bool valid = tb + q < t_end;
      // scores
      float2 a[GH];
#pragma unroll
      for (int k = 0; k < GH; ++k) a[k] = make_float2(0.f, 0.f);
      const float* qs = qv + s * C::QS;
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        const uint32_t ww[4] = {kc[k4].x, kc[k4].y, kc[k4].z, kc[k4].w};
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float kv = (u & 1) ? bf16_hi(ww[u >> 1]) : bf16_lo(ww[u >> 1]);
          float2 qq[GH];
          load_heads<GT>(qs + (k4 * 8 + u) * GTP, qq);
#pragma unroll
          for (int k = 0; k < GH; ++k) a[k] = fma2(make_float2(kv, kv), qq[k], a[k]);
        }
      }
#pragma unroll
      for (int m = 1; m < SL; m <<= 1)
#pragma unroll
        for (int k = 0; k < GH; ++k) {
          a[k].x += __shfl_xor_sync(0xffffffffu, a[k].x, m);
          a[k].y += __shfl_xor_sync(0xffffffffu, a[k].y, m);
        }
      float lg[GT];
#pragma unroll
      for (int h = 0; h < GT; ++h) lg[h] = valid ? ((h & 1) ? a[h >> 1].y : a[h >> 1].x) * p.sscale : -INFINITY;
      if (p.scap > 0.f) {
#pragma unroll
        for (int h = 0; h < GT; ++h) lg[h] = soft_cap(lg[h], p.scap, p.iscap);
      }
      // online softmax (the SL lanes of a token hold the same logits)
      bool need = false;
#pragma unroll
      for (int h = 0; h < GT; ++h) need |= lg[h] > m_w[h] + 8.f;
      if (__any_sync(0xffffffffu, need)) {
        float al[GT];
#pragma unroll
        for (int h = 0; h < GT; ++h) {
          const float mn = fmaxf(m_w[h], warp_max(lg[h]));
          al[h] = exp2f(m_w[h] - mn);
          m_w[h] = mn;
          l_ln[h] *= al[h];
        }
#pragma unroll
        for (int k = 0; k < GH; ++k) {
          const float2 a2 = make_float2(al[2 * k], (2 * k + 1 < GT) ? al[2 * k + 1] : 0.f);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) acc[cc][k] = mul2(acc[cc][k], a2);
        }
      }
#pragma unroll
      for (int h = 0; h < GT; ++h) {
        const float pe = valid ? exp2f(lg[h] - m_w[h]) : 0.f;
        if (s == 0) {
          l_ln[h] += pe;
          pw[q * GTP + h] = pe;
        }
      }
      __syncwarp();
      // values
#pragma unroll
      for (int j = 0; j < TW / TLW; ++j) {
        const int tt = tl + j * TLW;
        const float vv[4] = {bf16_lo(vc[j].x), bf16_hi(vc[j].x), bf16_lo(vc[j].y), bf16_hi(vc[j].y)};
        float2 pp[GH];
        load_heads<GT>(pw + tt * GTP, pp);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
          for (int k = 0; k < GH; ++k) acc[cc][k] = fma2(make_float2(vv[cc], vv[cc]), pp[k], acc[cc][k]);
      }
      __syncwarp();
    }
  } else {
    for (int i = 0; i < n; ++i) {
      cp_async_wait<0>();
      __syncthreads();  // record i is in; record i-1 is done with
      issue_main(i + 1);

      const unsigned char* st = stage(i);
      const unsigned char* kcodes = st + warp * 32 * rbk;  // the warp's 32 rows
      const float* knorm = reinterpret_cast<const float*>(st + p.k_off_norm) + warp * 32;
      const unsigned char* vbase = p.shared_kv ? st : st + p.k_main;
      const unsigned char* vcodes = vbase + warp * 32 * rbv;
      const float* vnorm = reinterpret_cast<const float*>(vbase + p.v_off_norm) + warp * 32;
      const int64_t c = t_begin + i;

      // outlier entries of the lane's own token; the first 8 of each stream are
      // fetched now so that their latency overlaps the scores
      int ke0 = 0, kec = 0, ve0 = 0, vec = 0;
      uint32_t kent[8], vent[8];
      const uint32_t* kge = reinterpret_cast<const uint32_t*>(krec_at(c) + p.k_off_ent);
      const uint32_t* vge = reinterpret_cast<const uint32_t*>(vrec_at(c) + p.v_off_ent);
      if (kout) {
        token_entries(st + p.k_off_count, kcap, ke0, kec);
  #pragma unroll
        for (int k = 0; k < 8; ++k) kent[k] = k < kec ? __ldg(kge + ke0 + k) : 0u;
      }
      if (vout) {
        token_entries(vbase + p.v_off_count, vcap, ve0, vec);
  #pragma unroll
        for (int k = 0; k < 8; ++k) vent[k] = k < vec ? __ldg(vge + ve0 + k) : 0u;
      }

      // ---- scores
      float lg[GT];
      {
        float2 a[TPL][GH];
  #pragma unroll
        for (int i2 = 0; i2 < TPL; ++i2)
  #pragma unroll
          for (int k = 0; k < GH; ++k) a[i2][k] = make_float2(0.f, 0.f);
        int tok[TPL];
  #pragma unroll
        for (int i2 = 0; i2 < TPL; ++i2) tok[i2] = q + QR * i2;
        const float* qs = qv + s * C::QS;
        switch (p.kb) {
          case 1: score_tokens<1, GT, GTP, TPL>(kcodes, rbk, tok, s, qs, lutk, a); break;
          case 2: score_tokens<2, GT, GTP, TPL>(kcodes, rbk, tok, s, qs, lutk, a); break;
          case 3: score_tokens<3, GT, GTP, TPL>(kcodes, rbk, tok, s, qs, lutk, a); break;
          default: score_tokens<4, GT, GTP, TPL>(kcodes, rbk, tok, s, qs, lutk, a); break;
        }
        float2 r[GH];
        reduce_transpose<SL, GH>(a, s, r);
  #pragma unroll
        for (int h = 0; h < GT; ++h) lg[h] = (h & 1) ? r[h >> 1].y : r[h >> 1].x;
      }
      if (kout) {
        // the stored value replaces the centroid: logit += (val - c[code]) q~_idx
        const unsigned char* krow = kcodes + tloc * rbk;
        auto kfix = [&](uint32_t v) {
          const int idx = (int)(v & 0xFFFFu) & (D - 1);
          const float delta = bf16_to_f32((uint16_t)(v >> 16)) - lutk[code_in_row(krow, idx, p.kb)];
          float2 qq[GH];
          load_heads<GT>(qv + (idx >> 5) * C::QS + (idx & 31) * GTP, qq);
  #pragma unroll
          for (int h = 0; h < GT; ++h) lg[h] = fmaf(delta, (h & 1) ? qq[h >> 1].y : qq[h >> 1].x, lg[h]);
        };
  #pragma unroll
        for (int k = 0; k < 8; ++k)
          if (k < kec) kfix(kent[k]);
        for (int k = 8; k < kec; ++k) kfix(__ldg(kge + ke0 + k));
      }
      {
        const float f = knorm[tloc] * p.sscale;
  #pragma unroll
        for (int h = 0; h < GT; ++h) lg[h] *= f;
        if (p.scap > 0.f) {
  #pragma unroll
          for (int h = 0; h < GT; ++h) lg[h] = soft_cap(lg[h], p.scap, p.iscap);
        }
      }

      // ---- online softmax (warp-local, the max moves only when a logit passes it by 2^8)
      float pv[GT];
      {
        bool need = false;
  #pragma unroll
        for (int h = 0; h < GT; ++h) need |= lg[h] > m_w[h] + 8.f;
        if (__any_sync(0xffffffffu, need)) {
          float al[GT];
  #pragma unroll
          for (int h = 0; h < GT; ++h) {
            const float mn = fmaxf(m_w[h], warp_max(lg[h]));
            al[h] = exp2f(m_w[h] - mn);
            m_w[h] = mn;
            l_ln[h] *= al[h];
          }
  #pragma unroll
          for (int k = 0; k < GH; ++k) {
            const float2 a2 = make_float2(al[2 * k], (2 * k + 1 < GT) ? al[2 * k + 1] : 0.f);
  #pragma unroll
            for (int cc = 0; cc < 4; ++cc) acc[cc][k] = mul2(acc[cc][k], a2);
          }
        }
        const float vn = vnorm[tloc];
  #pragma unroll
        for (int h = 0; h < GT; ++h) {
          const float pe = exp2f(lg[h] - m_w[h]);
          l_ln[h] += pe;
          pv[h] = pe * vn;
          pw[tloc * GTP + h] = pv[h];
        }
        __syncwarp();
      }

      // ---- values
      if (vout) {
        // the stored value replaces the centroid: acc_idx += p' (val - c[code]),
        // in fixed point S = 2^(23 - floor(log2 max p')): a term is below 2^25
        // in magnitude (|val - c| < 2) and a (head, coordinate) takes at most
        // one term per token, 32 per record, so a record's sums stay below 2^30
        float pmx = 0.f;
  #pragma unroll
        for (int h = 0; h < GT; ++h) pmx = fmaxf(pmx, pv[h]);
        pmx = warp_max(pmx);
        const int ef = min(254, max(1, 277 - (int)((__float_as_uint(pmx) >> 23) & 0xFFu)));
        const float S = __uint_as_float((uint32_t)ef << 23), iS = __uint_as_float((uint32_t)(254 - ef) << 23);
        const unsigned char* vrow = vcodes + tloc * rbv;
        auto vfix = [&](uint32_t v) {
          const int idx = (int)(v & 0xFFFFu) & (D - 1);
          const float delta = (bf16_to_f32((uint16_t)(v >> 16)) - lutv[code_in_row(vrow, idx, p.vb)]) * S;
  #pragma unroll
          for (int h = 0; h < GT; ++h) atomicAdd(&cw[h * D + idx], __float2int_rn(pv[h] * delta));
        };
  #pragma unroll
        for (int k = 0; k < 8; ++k)
          if (k < vec) vfix(vent[k]);
        for (int k = 8; k < vec; ++k) vfix(__ldg(vge + ve0 + k));
        __syncwarp();
        // fold the record's sums into the accumulators of the coordinates'
        // owners (4 g .. 4 g + 3, every head) and clear them
        if (tl == 0) {
  #pragma unroll
          for (int h = 0; h < GT; ++h) {
            int4* cp = reinterpret_cast<int4*>(cw + h * D + 4 * g);
            const int4 w = *cp;
            *cp = make_int4(0, 0, 0, 0);
            const float f[4] = {(float)w.x * iS, (float)w.y * iS, (float)w.z * iS, (float)w.w * iS};
  #pragma unroll
            for (int c = 0; c < 4; ++c) {
              if (h & 1) acc[c][h >> 1].y += f[c];
              else acc[c][h >> 1].x += f[c];
            }
          }
        }
        __syncwarp();
      }
      switch (p.vb) {
        case 1: pv_tokens<1, GT, GTP, TLW>(vcodes, rbv, pw, lutv, g, tl, acc); break;
        case 2: pv_tokens<2, GT, GTP, TLW>(vcodes, rbv, pw, lutv, g, tl, acc); break;
        case 3: pv_tokens<3, GT, GTP, TLW>(vcodes, rbv, pw, lutv, g, tl, acc); break;
        default: pv_tokens<4, GT, GTP, TLW>(vcodes, rbv, pw, lutv, g, tl, acc); break;
      }
    }
  }

  // ---- merge the warps' (m, l, acc) into the split's partial
#pragma unroll
  for (int h = 0; h < GT; ++h) l_ln[h] = warp_sum(l_ln[h]);
  if constexpr (TLW == 2) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int k = 0; k < GH; ++k) {
        acc[c][k].x += __shfl_xor_sync(0xffffffffu, acc[c][k].x, 16);
        acc[c][k].y += __shfl_xor_sync(0xffffffffu, acc[c][k].y, 16);
      }
  }
  __syncwarp();
  cp_async_wait<0>();
  __syncthreads();  // all records consumed: the staging ring becomes the merge buffer
  float* red = reinterpret_cast<float*>(mainb);          // [4][D][GTP]
  float* wml = reinterpret_cast<float*>(sm + p.sm_red);  // [4][2][GTP]
  if (tl == 0) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int h = 0; h < GT; ++h) {
        const float v = (h & 1) ? acc[c][h >> 1].y : acc[c][h >> 1].x;
        red[(warp * D + 4 * g + c) * GTP + h] = v;
      }
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < GT; ++h) {
      wml[(warp * 2) * GTP + h] = m_w[h];
      wml[(warp * 2 + 1) * GTP + h] = l_ln[h];
    }
  }
  __syncthreads();
  for (int idx = tid; idx < GT * D; idx += kThreads) {
    const int h = idx / D, j = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, wml[(w * 2) * GTP + h]);
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) v = fmaf(exp2f(wml[(w * 2) * GTP + h] - M), red[(w * D + j) * GTP + h], v);
    p.ws_acc[((qh0 + h) * p.S + split) * D + j] = v;
    if (j == 0) {
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) L = fmaf(exp2f(wml[(w * 2) * GTP + h] - M), wml[(w * 2 + 1) * GTP + h], L);
      float* ml = p.ws_ml + ((qh0 + h) * p.S + split) * 2;
      ml[0] = M;
      ml[1] = L;
    }
  }
}

template <int D, int GT>
cudaError_t attn_rec_launch_t(const AttnParams& p, dim3 grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(attn_rec_kernel<D, GT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       p.sm_total);
  if (e != cudaSuccess) return e;
  attn_rec_kernel<D, GT><<<grid, kThreads, p.sm_total, s>>>(p);
  return cudaGetLastError();
}

}  // namespace tq
