// Fused split-K decode attention over rotated Lloyd-Max records and a
// dense bf16 tail (or a whole bf16 layer).
//
// The query is rotated once per CTA, q~ = H(s_k . q)/sqrt(d); since H is
// orthonormal and symmetric, q . khat_i = n_i * q~ . yhat_i, so a compressed
// key scores straight from its codes through a shared-memory centroid table,
// and compressed values accumulate sum_i p_i n_i yhat_i in the rotated basis
// (one inverse transform at the merge).  Dense tokens are scored and
// accumulated in the original basis.  Online softmax in the log2 domain.
// (Problem statement of the pages: fused decode attention with q rotated once,
// a shared-memory LUT, online softmax, values accumulated in the rotated basis
// and one inverse RHT of the output; arc PR #98 "What landed": the dense tail
// is attended alongside the packed region.)
//
// CTA = 4 warps = one (layer, batch, kv head, group of GT query heads, split).
// A split is a run of whole records (128 tokens each) or a run of dense tail
// tokens.  Tiles are staged global -> shared with cp.async in a 3-deep ring;
// with outliers, a record's side list is fetched one tile behind its header
// once the per-slot counts are known, so only the used entries are read.
// Scores: thread = (token, 32-coordinate slice); the slice's codes are b words,
// partial dot products are reduced across the slices of a token by shuffles.
// Values: thread = (4 consecutive coordinates, token lane); accumulators for
// GT heads stay in registers as packed f32 pairs.
#pragma once

#include "tq_common.cuh"
#include "tq_params.h"

namespace tq {

template <int D, int GT>
struct ACfg {
  static constexpr int SL = D / 32;          // 32-coordinate slices per token
  static constexpr int TT = kThreads / SL;   // tokens per score pass = dense tile tokens
  static constexpr int CG = D / 4;           // 4-coordinate groups
  static constexpr int TL = kThreads / CG;   // token lanes of the value phase
  static constexpr int GTP = (GT == 6) ? 8 : GT;
  static constexpr int QPAD = GTP < 4 ? GTP : 4;
  static constexpr int QS = 32 * GTP + QPAD;  // floats per slice of the q array
  static constexpr int GH = (GT + 1) / 2;     // packed accumulator pairs
};

// ---- loads of GT consecutive floats (heads) as pairs
template <int GT>
__device__ __forceinline__ void load_heads(const float* p, float2 (&o)[(GT + 1) / 2]) {
  if constexpr (GT == 1) {
    o[0] = make_float2(p[0], 0.f);
  } else if constexpr (GT == 2) {
    o[0] = *reinterpret_cast<const float2*>(p);
  } else if constexpr (GT == 4) {
    float4 a = *reinterpret_cast<const float4*>(p);
    o[0] = make_float2(a.x, a.y); o[1] = make_float2(a.z, a.w);
  } else if constexpr (GT == 6) {
    float4 a = *reinterpret_cast<const float4*>(p);
    float2 b = *reinterpret_cast<const float2*>(p + 4);
    o[0] = make_float2(a.x, a.y); o[1] = make_float2(a.z, a.w); o[2] = b;
  } else {
    float4 a = *reinterpret_cast<const float4*>(p);
    float4 b = *reinterpret_cast<const float4*>(p + 4);
    o[0] = make_float2(a.x, a.y); o[1] = make_float2(a.z, a.w);
    o[2] = make_float2(b.x, b.y); o[3] = make_float2(b.z, b.w);
  }
}

template <int D>
__device__ __forceinline__ constexpr float inv_sqrt_dim() {
  return D == 64 ? 0.125f : D == 128 ? 0.08838834764831845f : D == 256 ? 0.0625f : 0.04419417382415922f;
}

template <int B>
__device__ __forceinline__ uint32_t code_of(const uint32_t (&w)[B], int r) {  // compile-time r
  const int bit = r * B;
  uint32_t v = w[bit >> 5] >> (bit & 31);
  if ((bit & 31) + B > 32) v |= w[(bit >> 5) + 1] << (32 - (bit & 31));
  return v & ((1u << B) - 1u);
}

template <int B>
__device__ __forceinline__ void load_words(const unsigned char* p, uint32_t (&w)[B]) {
  if constexpr (B == 4) {
    uint4 a = *reinterpret_cast<const uint4*>(p);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  } else if constexpr (B == 2) {
    uint2 a = *reinterpret_cast<const uint2*>(p);
    w[0] = a.x; w[1] = a.y;
  } else {
#pragma unroll
    for (int q = 0; q < B; ++q) w[q] = reinterpret_cast<const uint32_t*>(p)[q];
  }
}

// Score contribution of one token's 32-coordinate slice of codes.
template <int B, int GT, int GTP>
__device__ __forceinline__ void score_slice(const unsigned char* row_slice, const float* qs,
                                            const float* lut, float2 (&acc)[(GT + 1) / 2],
                                            bool with_out, const uint32_t* ent, int e0, int e1,
                                            int slice) {
  uint32_t w[B];
  load_words<B>(row_slice, w);
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    const float cv = lut[code_of<B>(w, r)];
    float2 q[(GT + 1) / 2];
    load_heads<GT>(qs + r * GTP, q);
#pragma unroll
    for (int k = 0; k < (GT + 1) / 2; ++k) acc[k] = fma2(make_float2(cv, cv), q[k], acc[k]);
  }
  if (with_out) {
    // outlier coordinates: the stored value replaces the centroid
    for (int e = e0; e < e1; ++e) {
      const uint32_t v = ent[e];
      const int idx = (int)(v & 0xFFFFu);
      if ((idx >> 5) != slice) continue;
      const int r = idx & 31;
      const float delta = bf16_to_f32((uint16_t)(v >> 16)) - lut[code_at<B>(w, r)];
      float2 q[(GT + 1) / 2];
      load_heads<GT>(qs + r * GTP, q);
#pragma unroll
      for (int k = 0; k < (GT + 1) / 2; ++k) acc[k] = fma2(make_float2(delta, delta), q[k], acc[k]);
    }
  }
}

// Value accumulation of tokens t = tl, tl + TL, ... < ntok for coordinates 4g..4g+3.
template <int B, int GT, int GTP, int TL>
__device__ __forceinline__ void pv_codes(const unsigned char* vcodes, int rb, const float* pb,
                                         const float* lut, int g, int tl, int ntok,
                                         float2 (&acc)[4][(GT + 1) / 2]) {
  const int bit0 = 4 * g * B, wi = bit0 >> 5, sh = bit0 & 31;
  for (int t = tl; t < ntok; t += TL) {
    const uint32_t* row = reinterpret_cast<const uint32_t*>(vcodes + t * rb);
    uint32_t v;
    if constexpr (B == 3) {
      const uint64_t x = (uint64_t)row[wi] | ((uint64_t)row[wi + 1] << 32);
      v = (uint32_t)(x >> sh);
    } else {
      v = row[wi] >> sh;
    }
    float2 p[(GT + 1) / 2];
    load_heads<GT>(pb + t * GTP, p);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float val = lut[(v >> (c * B)) & ((1u << B) - 1u)];
#pragma unroll
      for (int k = 0; k < (GT + 1) / 2; ++k) acc[c][k] = fma2(make_float2(val, val), p[k], acc[c][k]);
    }
  }
}

// One dense split: bf16 tokens (a tail ring or a whole bf16 layer) attended
// in the original basis, 4096/D tokens per tile staged by cp.async in a
// 2-deep ring, online softmax across the CTA.  Writes the split's partial.
template <int D, int GT>
__device__ __forceinline__ void attn_dense_split(const AttnParams& p, unsigned char* sm, int l, int b,
                                                 int kvh, int h0, int split, int64_t qh0, int t_begin,
                                                 int t_end) {
  using C = ACfg<D, GT>;
  constexpr int GTP = C::GTP, GH = C::GH, SL = C::SL, TT = C::TT, CG = C::CG, TL = C::TL;
  float* qv = reinterpret_cast<float*>(sm + p.sm_q);
  float* redm = reinterpret_cast<float*>(sm + p.sm_red);
  float* reds = redm + 4 * GTP;
  float* logit = reinterpret_cast<float*>(sm + p.sm_logit);
  unsigned char* mainb = sm + p.sm_main;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int lb = l * p.B + b;
  const int tstart = p.tail_start ? ((p.tail_start[lb] % p.tail_cap) + p.tail_cap) % p.tail_cap : 0;
  const uint16_t* kt0 = p.ktail + l * p.tail_ls + (int64_t)(b * p.Hkv + kvh) * p.tail_cap * D;
  const uint16_t* vt0 = p.vtail + l * p.tail_ls + (int64_t)(b * p.Hkv + kvh) * p.tail_cap * D;
  const int n_tiles = (t_end - t_begin + TT - 1) / TT;
  constexpr int TB = TT * D * 2;  // bytes of one stream's tile
  auto stage = [&](int i) { return mainb + (i & 1) * p.sm_stage; };
  auto issue = [&](int i) {
    if (i < n_tiles) {
      const int tok0 = t_begin + i * TT;
      const int cnt = min(TT, t_end - tok0);
      unsigned char* s = stage(i);
      for (int pc = tid; pc < TT * (D / 8); pc += kThreads) {
        const int tok = pc / (D / 8), part = pc % (D / 8);
        if (tok < cnt) {
          const int64_t slot = (tstart + tok0 + tok) % p.tail_cap;
          cp_async16(s + (tok * D + part * 8) * 2, kt0 + slot * D + part * 8);
          cp_async16(s + TB + (tok * D + part * 8) * 2, vt0 + slot * D + part * 8);
        }
      }
    }
    cp_async_commit();
  };
  issue(0);
  // query (original basis) as [slice][32][GTP]
  for (int hh = warp; hh < GT; hh += 4) {
    constexpr int R = D / 32;
    const uint16_t* qp = p.q + l * p.q_ls + b * p.q_bs + (int64_t)(h0 + hh) * D + lane * R;
#pragma unroll
    for (int r = 0; r < R; r += 2) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(qp + r);
      const int j = lane * R + r;
      qv[(j >> 5) * C::QS + (j & 31) * GTP + hh] = bf16_lo(w);
      qv[((j + 1) >> 5) * C::QS + ((j + 1) & 31) * GTP + hh] = bf16_hi(w);
    }
  }
  if (GTP != GT)
    for (int i = tid; i < D; i += kThreads)
#pragma unroll
      for (int hh = GT; hh < GTP; ++hh) qv[(i >> 5) * C::QS + (i & 31) * GTP + hh] = 0.f;

  float m_run[GT], l_run[GT], alpha[GT];
#pragma unroll
  for (int h = 0; h < GT; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.f;
  }
  float2 acc[4][GH];
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int k = 0; k < GH; ++k) acc[c][k] = make_float2(0.f, 0.f);
  const int g = tid % CG, tl = tid / CG;
  const int stok = tid / SL, slice = tid % SL;
  for (int i = 0; i < n_tiles; ++i) {
    cp_async_wait<0>();
    __syncthreads();  // tile i is in; tile i-1 is done with
    issue(i + 1);
    const int ntok = min(TT, t_end - (t_begin + i * TT));
    const unsigned char* s = stage(i);
    {
      float2 a[GH];
#pragma unroll
      for (int k = 0; k < GH; ++k) a[k] = make_float2(0.f, 0.f);
      if (stok < ntok) {
        const uint4* kr = reinterpret_cast<const uint4*>(s + (stok * D + slice * 32) * 2);
        const float* qs = qv + slice * C::QS;
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const uint4 w = kr[k4];
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float kv = (u & 1) ? bf16_hi(ww[u >> 1]) : bf16_lo(ww[u >> 1]);
            float2 q[GH];
            load_heads<GT>(qs + (k4 * 8 + u) * GTP, q);
#pragma unroll
            for (int k = 0; k < GH; ++k) a[k] = fma2(make_float2(kv, kv), q[k], a[k]);
          }
        }
      }
#pragma unroll
      for (int m = 1; m < SL; m <<= 1)
#pragma unroll
        for (int k = 0; k < GH; ++k) {
          a[k].x += __shfl_xor_sync(0xffffffffu, a[k].x, m);
          a[k].y += __shfl_xor_sync(0xffffffffu, a[k].y, m);
        }
      if (slice == 0 && stok < ntok) {
#pragma unroll
        for (int h = 0; h < GT; ++h) {
          float t = (h & 1 ? a[h >> 1].y : a[h >> 1].x) * p.sscale;
          if (p.scap > 0.f) t = soft_cap(t, p.scap, p.iscap);
          logit[stok * GTP + h] = t;
        }
      }
    }
    __syncthreads();
    // online softmax over the tile (CTA-wide)
    {
      float v[GT];
#pragma unroll
      for (int h = 0; h < GT; ++h) {
        v[h] = tid < ntok ? logit[tid * GTP + h] : -INFINITY;
        const float mx = warp_max(v[h]);
        if (lane == 0) redm[warp * GTP + h] = mx;
      }
      __syncthreads();
#pragma unroll
      for (int h = 0; h < GT; ++h) {
        const float mx = fmaxf(fmaxf(redm[h], redm[GTP + h]), fmaxf(redm[2 * GTP + h], redm[3 * GTP + h]));
        const float mnew = fmaxf(m_run[h], mx);
        alpha[h] = exp2f(m_run[h] - mnew);
        m_run[h] = mnew;
        const float pe = tid < ntok ? exp2f(v[h] - mnew) : 0.f;
        if (tid < ntok) logit[tid * GTP + h] = pe;
        const float sum = warp_sum(pe);
        if (lane == 0) reds[warp * GTP + h] = sum;
      }
      __syncthreads();
#pragma unroll
      for (int h = 0; h < GT; ++h)
        l_run[h] = l_run[h] * alpha[h] + ((reds[h] + reds[GTP + h]) + (reds[2 * GTP + h] + reds[3 * GTP + h]));
    }
#pragma unroll
    for (int k = 0; k < GH; ++k) {
      const float2 a2 = make_float2(alpha[2 * k], (2 * k + 1 < GT) ? alpha[2 * k + 1] : 0.f);
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[c][k] = mul2(acc[c][k], a2);
    }
    for (int t = tl; t < ntok; t += TL) {
      const uint2 w = *reinterpret_cast<const uint2*>(s + TB + (t * D + 4 * g) * 2);
      const float vv[4] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y)};
      float2 pp[GH];
      load_heads<GT>(logit + t * GTP, pp);
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int k = 0; k < GH; ++k) acc[c][k] = fma2(make_float2(vv[c], vv[c]), pp[k], acc[c][k]);
    }
  }
  cp_async_wait<0>();
  __syncthreads();
  float* part = reinterpret_cast<float*>(mainb);  // [TL][D][GTP]
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int h = 0; h < GT; ++h) part[(tl * D + 4 * g + c) * GTP + h] = (h & 1) ? acc[c][h >> 1].y : acc[c][h >> 1].x;
  __syncthreads();
  for (int i = tid; i < GT * D; i += kThreads) {
    const int h = i / D, j = i % D;
    float sum = 0.f;
#pragma unroll
    for (int t = 0; t < TL; ++t) sum += part[(t * D + j) * GTP + h];
    p.ws_acc[((qh0 + h) * p.S + split) * D + j] = sum;
  }
#pragma unroll
  for (int h = 0; h < GT; ++h)
    if (tid == h) {
      float* ml = p.ws_ml + ((qh0 + h) * p.S + split) * 2;
      ml[0] = m_run[h];
      ml[1] = l_run[h];
    }
}

template <int D, int GT>
__global__ void __launch_bounds__(kThreads) attn_kernel(const __grid_constant__ AttnParams p) {
  using C = ACfg<D, GT>;
  constexpr int GTP = C::GTP, GH = C::GH, SL = C::SL, TT = C::TT, CG = C::CG, TL = C::TL;
  extern __shared__ __align__(128) unsigned char sm[];
  float* qv = reinterpret_cast<float*>(sm + p.sm_q);
  float* lutk = reinterpret_cast<float*>(sm + p.sm_lut);
  float* lutv = lutk + 16;
  float* redm = reinterpret_cast<float*>(sm + p.sm_red);
  float* reds = redm + 4 * GTP;
  float* logit = reinterpret_cast<float*>(sm + p.sm_logit);
  float* corr = reinterpret_cast<float*>(sm + p.sm_corr);
  int* pre = reinterpret_cast<int*>(sm + p.sm_pre);          // [2][2][129]
  uint8_t* slotof = sm + p.sm_slot;                         // [2][vcap]
  unsigned char* mainb = sm + p.sm_main;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int l = blockIdx.z;
  int rem = blockIdx.y;
  const int hg = rem % p.n_hg;
  rem /= p.n_hg;
  const int kvh = rem % p.Hkv, b = rem / p.Hkv;
  const int split = blockIdx.x + p.split_base;
  const int h0 = kvh * p.G + hg * GT;
  const bool comp = split < p.Sc;
  const int lb = l * p.B + b;
  const int64_t qh0 = (int64_t)lb * p.Hq + h0;

  int t_begin, t_end;
  // device counters are clamped to the buffers they index, so a corrupt
  // counter can never move a copy outside the caller's arrays
  if (comp) {
    const int nch = min(p.n_chunks ? p.n_chunks[lb] : 0, p.rec_limit);
    t_begin = split * p.cps;
    t_end = min(t_begin + p.cps, nch);
  } else {
    const int tl = min(p.tail_len ? p.tail_len[lb] : 0, p.tail_cap);
    t_begin = (split - p.Sc) * p.tps;
    t_end = min(t_begin + p.tps, tl);
  }
  if (t_begin >= t_end) {
    if (tid < GT) {
      float* ml = p.ws_ml + ((qh0 + tid) * p.S + split) * 2;
      ml[0] = -INFINITY;
      ml[1] = 0.f;
    }
    return;
  }
  if (!comp) {
    attn_dense_split<D, GT>(p, sm, l, b, kvh, h0, split, qh0, t_begin, t_end);
    return;
  }

  const int n_tiles_c = t_end - t_begin;
  // ---- compressed splits: record staging (3-deep cp.async ring)
  // record c of this unit (contiguous, or through the block table)
  const uint8_t* kl0 = p.krec + l * p.krec_ls;
  const uint8_t* vl0 = p.shared_kv ? kl0 : p.vrec + l * p.vrec_ls;
  auto krec_at = [&](int64_t c) {
    return kl0 + rec_offset(p.table, p.table_stride, p.rec_cap, p.Hkv, b, kvh, (int)c, p.krec_bytes);
  };
  auto vrec_at = [&](int64_t c) {
    return vl0 + rec_offset(p.table, p.table_stride, p.rec_cap, p.Hkv, b, kvh, (int)c, p.vrec_bytes);
  };
  const bool anyout = p.kout || p.vout;
  const int vcap = p.shared_kv ? p.kcap : p.vcap;
  auto stage = [&](int i) { return mainb + (i % 3) * p.sm_stage; };
  auto entb = [&](int i) { return reinterpret_cast<uint32_t*>(sm + p.sm_ent + (i & 1) * p.sm_ent_stage); };
  auto issue_main = [&](int i) {
    if (i < n_tiles_c) {
      const int64_t c = t_begin + i;
      cta_copy_async(stage(i), krec_at(c), p.k_main);
      if (!p.shared_kv) cta_copy_async(stage(i) + p.k_main, vrec_at(c), p.v_main);
    }
    cp_async_commit();
  };
  auto prefix = [&](int i) {
    if (i >= n_tiles_c || !anyout || warp >= 2) return;
    const bool isk = warp == 0;
    if (isk ? !p.kout : (!p.vout || p.shared_kv)) return;
    const unsigned char* cnts = isk ? stage(i) + p.k_off_count : stage(i) + p.k_main + p.v_off_count;
    int* pr = pre + ((i & 1) * 2 + (isk ? 0 : 1)) * 129;
    const uint32_t c4 = reinterpret_cast<const uint32_t*>(cnts)[lane];  // slots 4*lane .. 4*lane+3
    const int n0 = c4 & 0xff, n1 = (c4 >> 8) & 0xff, n2 = (c4 >> 16) & 0xff, n3 = c4 >> 24;
    const int tot = n0 + n1 + n2 + n3;
    int inc = tot;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, inc, m);
      if (lane >= m) inc += o;
    }
    const int ex = inc - tot;
    pr[4 * lane] = ex;
    pr[4 * lane + 1] = ex + n0;
    pr[4 * lane + 2] = ex + n0 + n1;
    pr[4 * lane + 3] = ex + n0 + n1 + n2;
    if (lane == 31) pr[128] = inc;
    const bool vmap = !isk || p.shared_kv;  // value corrections need entry -> slot
    if (vmap && p.vout) {
      uint8_t* so = slotof + (i & 1) * vcap;
      int e = ex;
      const int ns[4] = {n0, n1, n2, n3};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        for (int k = 0; k < ns[q]; ++k, ++e)
          if (e < vcap) so[e] = (uint8_t)(4 * lane + q);
    }
  };
  auto issue_ent = [&](int i) {
    if (i < n_tiles_c && anyout) {
      const int64_t c = t_begin + i;
      uint32_t* eb = entb(i);
      if (p.kout) {
        const int E = min(pre[((i & 1) * 2) * 129 + 128], p.kcap);
        cta_copy_async(eb, krec_at(c) + p.k_off_ent, (E * 4 + 15) & ~15);
      }
      if (p.vout && !p.shared_kv) {
        const int E = min(pre[((i & 1) * 2 + 1) * 129 + 128], p.vcap);
        cta_copy_async(eb + p.kcap * p.kout, vrec_at(c) + p.v_off_ent, (E * 4 + 15) & ~15);
      }
    }
    cp_async_commit();
  };

  // the first copies go out before the query work so their latency overlaps it
  issue_main(0);
  issue_main(1);

  // ---- query: load, rotate (compressed split), store as [slice][32][GTP]
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
    if (comp) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int j = lane * R + r;
        if ((p.ksign[j >> 5] >> (j & 31)) & 1u) x[r] = -x[r];
      }
      fwht_regs<R>(x);
      fwht_lanes<R>(x, lane, 32);
      const float f = inv_sqrt_dim<D>();
#pragma unroll
      for (int r = 0; r < R; ++r) x[r] *= f;
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int j = lane * R + r;
      qv[(j >> 5) * C::QS + (j & 31) * GTP + hh] = x[r];
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
  if (p.vout)
    for (int i = tid; i < D * GTP; i += kThreads) corr[i] = 0.f;

  float m_run[GT], l_run[GT], alpha[GT];
#pragma unroll
  for (int h = 0; h < GT; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.f;
  }
  float2 acc[4][GH];
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int k = 0; k < GH; ++k) acc[c][k] = make_float2(0.f, 0.f);

  const int g = tid % CG, tl = tid / CG;  // value-phase mapping
  const int stok = tid / SL, slice = tid % SL;  // score-phase mapping

  // online softmax over `ntok` logits of the tile; p (times the value norm)
  // replaces the logit in place
  auto softmax = [&](int ntok, const float* vnorm) {
    float v[GT];
#pragma unroll
    for (int h = 0; h < GT; ++h) {
      v[h] = tid < ntok ? logit[tid * GTP + h] : -INFINITY;
      const float mx = warp_max(v[h]);
      if (lane == 0) redm[warp * GTP + h] = mx;
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < GT; ++h) {
      float mx = fmaxf(fmaxf(redm[h], redm[GTP + h]), fmaxf(redm[2 * GTP + h], redm[3 * GTP + h]));
      const float mnew = fmaxf(m_run[h], mx);
      alpha[h] = exp2f(m_run[h] - mnew);
      m_run[h] = mnew;
      const float pe = tid < ntok ? exp2f(v[h] - mnew) : 0.f;
      if (tid < ntok) logit[tid * GTP + h] = vnorm ? pe * vnorm[tid] : pe;
      const float s = warp_sum(pe);
      if (lane == 0) reds[warp * GTP + h] = s;
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < GT; ++h)
      l_run[h] = l_run[h] * alpha[h] + ((reds[h] + reds[GTP + h]) + (reds[2 * GTP + h] + reds[3 * GTP + h]));
  };
  auto rescale = [&]() {
#pragma unroll
    for (int k = 0; k < GH; ++k) {
      const float2 a = make_float2(alpha[2 * k], (2 * k + 1 < GT) ? alpha[2 * k + 1] : 0.f);
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[c][k] = mul2(acc[c][k], a);
    }
  };
  auto reduce_slices = [&](float2 (&a)[GH]) {
#pragma unroll
    for (int m = 1; m < SL; m <<= 1)
#pragma unroll
      for (int k = 0; k < GH; ++k) {
        a[k].x += __shfl_xor_sync(0xffffffffu, a[k].x, m);
        a[k].y += __shfl_xor_sync(0xffffffffu, a[k].y, m);
      }
  };

  if (comp) {
    cp_async_wait<1>();
    __syncthreads();
    prefix(0);
    __syncthreads();
    issue_ent(0);
    for (int i = 0; i < n_tiles_c; ++i) {
      issue_main(i + 2);
      cp_async_wait<2>();
      __syncthreads();
      prefix(i + 1);
      __syncthreads();
      issue_ent(i + 1);
      cp_async_wait<2>();
      __syncthreads();

      const unsigned char* st = stage(i);
      const unsigned char* kcodes = st;
      const float* knorm = reinterpret_cast<const float*>(st + p.k_off_norm);
      const unsigned char* vcodes = p.shared_kv ? st : st + p.k_main;
      const float* vnorm = reinterpret_cast<const float*>(vcodes + p.v_off_norm);
      const uint32_t* kent = entb(i);
      const uint32_t* vent = p.shared_kv ? kent : kent + p.kcap * p.kout;
      const int* preK = pre + ((i & 1) * 2) * 129;
      const int* preV = p.shared_kv ? preK : pre + ((i & 1) * 2 + 1) * 129;
      const int rbk = D * p.kb / 8, rbv = D * p.vb / 8;

      // scores
#pragma unroll 1
      for (int pass = 0; pass < kChunk / TT; ++pass) {
        const int tok = pass * TT + stok;
        float2 a[GH];
#pragma unroll
        for (int k = 0; k < GH; ++k) a[k] = make_float2(0.f, 0.f);
        const unsigned char* rs = kcodes + tok * rbk + slice * 4 * p.kb;
        const float* qs = qv + slice * C::QS;
        const int e0 = p.kout ? preK[tok] : 0, e1 = p.kout ? preK[tok + 1] : 0;
        switch (p.kb) {
          case 1: score_slice<1, GT, GTP>(rs, qs, lutk, a, p.kout, kent, e0, min(e1, p.kcap), slice); break;
          case 2: score_slice<2, GT, GTP>(rs, qs, lutk, a, p.kout, kent, e0, min(e1, p.kcap), slice); break;
          case 3: score_slice<3, GT, GTP>(rs, qs, lutk, a, p.kout, kent, e0, min(e1, p.kcap), slice); break;
          default: score_slice<4, GT, GTP>(rs, qs, lutk, a, p.kout, kent, e0, min(e1, p.kcap), slice); break;
        }
        reduce_slices(a);
        if (slice == 0) {
          const float f = knorm[tok] * p.sscale;
#pragma unroll
          for (int h = 0; h < GT; ++h) {
            float t = (h & 1 ? a[h >> 1].y : a[h >> 1].x) * f;
            if (p.scap > 0.f) t = soft_cap(t, p.scap, p.iscap);
            logit[tok * GTP + h] = t;
          }
        }
      }
      __syncthreads();
      softmax(kChunk, vnorm);
      rescale();
      switch (p.vb) {
        case 1: pv_codes<1, GT, GTP, TL>(vcodes, rbv, logit, lutv, g, tl, kChunk, acc); break;
        case 2: pv_codes<2, GT, GTP, TL>(vcodes, rbv, logit, lutv, g, tl, kChunk, acc); break;
        case 3: pv_codes<3, GT, GTP, TL>(vcodes, rbv, logit, lutv, g, tl, kChunk, acc); break;
        default: pv_codes<4, GT, GTP, TL>(vcodes, rbv, logit, lutv, g, tl, kChunk, acc); break;
      }
      if (p.vout) {
        const uint8_t* so = slotof + (i & 1) * vcap;
        const int E = min(preV[128], vcap);
        const int vb = p.vb;
        for (int e = tid; e < E; e += kThreads) {
          const uint32_t v = vent[e];
          const int idx = (int)(v & 0xFFFFu) & (D - 1);
          const int s = so[e];
          const uint32_t* row = reinterpret_cast<const uint32_t*>(vcodes + s * rbv);
          const int bit = idx * vb;
          const uint64_t x = (uint64_t)row[bit >> 5] | ((uint64_t)row[(bit >> 5) + 1] << 32);
          const uint32_t code = (uint32_t)(x >> (bit & 31)) & ((1u << vb) - 1u);
          const float delta = bf16_to_f32((uint16_t)(v >> 16)) - lutv[code];
#pragma unroll
          for (int h = 0; h < GT; ++h) atomicAdd(&corr[idx * GTP + h], logit[s * GTP + h] * delta);
        }
        __syncthreads();
        if (tl == 0) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int h = 0; h < GT; ++h) {
              float* cp = &corr[(4 * g + c) * GTP + h];
              if (h & 1) acc[c][h >> 1].y += *cp; else acc[c][h >> 1].x += *cp;
              *cp = 0.f;
            }
        }
      }
      __syncthreads();
    }
  }

  // ---- partial result of this split: reduce the token lanes, write (m, l, acc)
  cp_async_wait<0>();
  __syncthreads();
  float* part = reinterpret_cast<float*>(mainb);  // [TL][D][GTP]
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int h = 0; h < GT; ++h) part[(tl * D + 4 * g + c) * GTP + h] = (h & 1) ? acc[c][h >> 1].y : acc[c][h >> 1].x;
  __syncthreads();
  for (int i = tid; i < GT * D; i += kThreads) {
    const int h = i / D, j = i % D;
    float s = 0.f;
#pragma unroll
    for (int t = 0; t < TL; ++t) s += part[(t * D + j) * GTP + h];
    p.ws_acc[((qh0 + h) * p.S + split) * D + j] = s;
  }
#pragma unroll
  for (int h = 0; h < GT; ++h)
    if (tid == h) {
      float* ml = p.ws_ml + ((qh0 + h) * p.S + split) * 2;
      ml[0] = m_run[h];
      ml[1] = l_run[h];
    }
}

template <int D, int GT>
cudaError_t attn_launch_t(const AttnParams& p, dim3 grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(attn_kernel<D, GT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       p.sm_total);
  if (e != cudaSuccess) return e;
  attn_kernel<D, GT><<<grid, kThreads, p.sm_total, s>>>(p);
  return cudaGetLastError();
}

}  // namespace tq
