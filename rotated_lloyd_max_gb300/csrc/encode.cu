// Encode bf16 head vectors into 128-token records, and chunked
// eviction from dense ring-buffer tails into records.
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
template <int D, int B, bool OUTL>
__device__ __forceinline__ void enc_vector(const CodecDev& c, const EncLane<D, B, OUTL>& ln,
                                           const float2* cells, float* tb, const uint4 (&w)[4], bool valid,
                                           uint8_t* rec, int slot, float (&x)[32], float& inv, uint32_t& omask) {
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
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    const float aw = fabsf(x[r]);
    uint32_t code;
    if constexpr (B >= 3) {  // decision cells (shared table)
      const float z = x[r] * zscale;
      const uint32_t ci = __float_as_uint(z + 8388736.0f) & 0x1FFu;  // round(z) + 128 (2^23 + 128 magic)
      code = cell_count(cells, ci) - mask_gt(z, cell_boundary(cells, ci));
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
    if (ln.lg == 0) reinterpret_cast<float*>(rec + c.off_norm)[slot] = n;
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
template <int D, int B, bool OUTL, class RowFn>
__device__ __forceinline__ void encode_record(const CodecDev& c, const float2* cells, float* tb, RowFn row,
                                              uint8_t* rec, int s_begin, int s_end, EncSmem* sm) {
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
    enc_vector<D, B, OUTL>(c, ln, cells, tb, w, valid, rec, slot, x, inv, omask);
    if constexpr (OUTL) enc_outliers<D, B>(c, ln, x, inv, omask, valid, rec, slot, pslot, sm);
  }
}

// Record-aligned encode with outliers: one CTA per record (grid-stride).
template <int D, int B>
__global__ void __launch_bounds__(kThreads) encode_record_kernel(const __grid_constant__ EncodeParams p) {
  __shared__ EncSmem sm;
  __shared__ __align__(16) float tbuf[D == 512 ? (kThreads / 32) * 2 * kTVec : 4];
  float* tb = tbuf + (threadIdx.x >> 5) * 2 * kTVec;
  __shared__ float2 cells[B >= 3 ? kCells : 1];
  if constexpr (B >= 3) {
    build_cells<true>(p.c, cells);
    __syncthreads();
  }
  const int64_t n_tasks = p.n_groups * p.chunks_per_group;
  for (int64_t task = blockIdx.x; task < n_tasks; task += gridDim.x) {
    const int64_t g = task / p.chunks_per_group;
    const int64_t ci = p.first_chunk + task % p.chunks_per_group;
    const int64_t lo = max(p.first_vec, ci * kChunk), hi = min(p.first_vec + p.n_vec, (ci + 1) * kChunk);
    uint8_t* rec = p.dst + g * p.dst_gs + ci * (int64_t)p.c.rec_bytes;
    const uint16_t* src_g = p.src + g * p.src_gs;
    const int64_t vs = p.src_vs, v0 = ci * kChunk - p.first_vec;
    auto row = [&](int slot) { return src_g + (v0 + slot) * vs; };
    encode_record<D, B, true>(p.c, cells, tb, row, rec, (int)(lo - ci * kChunk), (int)(hi - ci * kChunk), &sm);
  }
}

// Encode without outliers: every (group, record, pass) is an independent task
// of VPC vectors; CTAs stride over tasks with the next task's loads in flight.
template <int D, int B>
__global__ void __launch_bounds__(kThreads) encode_pass_kernel(const __grid_constant__ EncodeParams p) {
  using E = Enc<D, B, false>;
  constexpr int PPR = kChunk / E::VPC;  // passes per record
  __shared__ float2 cells[B >= 3 ? kCells : 1];
  __shared__ __align__(16) float tbuf[D == 512 ? (kThreads / 32) * 2 * kTVec : 4];
  float* tb = tbuf + (threadIdx.x >> 5) * 2 * kTVec;
  if constexpr (B >= 3) {
    build_cells<true>(p.c, cells);
    __syncthreads();
  }
  const EncLane<D, B, false> ln(p.c);
  const int pslot = ln.warp * E::VPW + ln.vi;
  const int64_t per_group = p.chunks_per_group * PPR;
  const int64_t n_tasks = p.n_groups * per_group;
  const int64_t v_end = p.first_vec + p.n_vec;
  // task -> (group, token index, validity)
  auto locate = [&](int64_t task, int64_t& g, int64_t& tok) {
    g = task / per_group;
    const int64_t r = task % per_group;
    tok = (p.first_chunk + r / PPR) * kChunk + (r % PPR) * E::VPC + pslot;
    return task < n_tasks && tok >= p.first_vec && tok < v_end;
  };
  int64_t g, tok;
  bool valid = locate(blockIdx.x, g, tok);
  uint4 wn[4];
  enc_load(p.src + g * p.src_gs + (tok - p.first_vec) * p.src_vs + ln.lg * 32, valid, wn);
  for (int64_t task = blockIdx.x; task < n_tasks; task += gridDim.x) {
    uint4 w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = wn[k];
    const int64_t cg = g, ctok = tok;
    const bool cvalid = valid;
    valid = locate(task + gridDim.x, g, tok);
    enc_load(p.src + g * p.src_gs + (tok - p.first_vec) * p.src_vs + ln.lg * 32, valid, wn);
    uint8_t* rec = p.dst + cg * p.dst_gs + (ctok / kChunk) * (int64_t)p.c.rec_bytes;
    float x[32];
    float inv;
    uint32_t omask;
    enc_vector<D, B, false>(p.c, ln, cells, tb, w, cvalid, rec, (int)(ctok % kChunk), x, inv, omask);
  }
}

// Eviction: CTA (e, b*Hkv + h, l) encodes the e-th due chunk of stream (l, b, h).
template <int D, int B, bool OUTL>
__global__ void __launch_bounds__(kThreads) evict_kernel(const __grid_constant__ EvictParams p) {
  __shared__ EncSmem sm;
  const int e = blockIdx.x;
  const int h = blockIdx.y % p.Hkv, b = blockIdx.y / p.Hkv, l = blockIdx.z;
  const int lb = l * p.B + b;
  const int len = p.tail_len[lb], nch = p.n_chunks[lb];
  const int start = ((p.tail_start[lb] % p.tail_cap) + p.tail_cap) % p.tail_cap;
  const int k = len >= p.floor_ + kChunk ? min((len - p.floor_) / kChunk, p.max_evict) : 0;
  if (e >= k || nch < 0 || nch + k > p.rec_cap) return;
  __shared__ float2 cells[B >= 3 ? kCells : 1];
  __shared__ __align__(16) float tbuf[D == 512 ? (kThreads / 32) * 2 * kTVec : 4];
  float* tb = tbuf + (threadIdx.x >> 5) * 2 * kTVec;
  if constexpr (B >= 3) {
    build_cells<true>(p.c, cells);
    __syncthreads();
  }
  uint8_t* rec = p.rec + l * p.rec_ls +
                 ((int64_t)(b * p.Hkv + h) * p.rec_cap + nch + e) * (int64_t)p.c.rec_bytes;
  const uint16_t* tail = p.tail + l * p.tail_ls + (int64_t)(b * p.Hkv + h) * p.tail_cap * D;
  const int first = start + e * kChunk;
  const int cap = p.tail_cap;
  auto row = [&](int slot) { return tail + (int64_t)((first + min(slot, kChunk - 1)) % cap) * D; };
  encode_record<D, B, OUTL>(p.c, cells, tb, row, rec, 0, kChunk, &sm);
}

__global__ void evict_commit_kernel(const EvictCommitParams p) {
  for (int lb = blockIdx.x * blockDim.x + threadIdx.x; lb < p.LB; lb += gridDim.x * blockDim.x) {
    const int len = p.tail_len[lb];
    const int k = len >= p.floor_ + kChunk ? min((len - p.floor_) / kChunk, p.max_evict) : 0;
    if (k == 0 || p.n_chunks[lb] < 0 || p.n_chunks[lb] + k > p.rec_cap) continue;
    const int start = ((p.tail_start[lb] % p.tail_cap) + p.tail_cap) % p.tail_cap;
    p.n_chunks[lb] += k;
    p.tail_start[lb] = (start + k * kChunk) % p.tail_cap;
    p.tail_len[lb] = len - k * kChunk;
  }
}

template <int D, int B, bool OUTL>
static cudaError_t enc_launch(const EncodeParams& p, int grid, cudaStream_t s) {
  if constexpr (OUTL) {
    const int64_t tasks = p.n_groups * p.chunks_per_group;
    encode_record_kernel<D, B><<<(int)std::min<int64_t>(tasks, grid), kThreads, 0, s>>>(p);
  } else {
    const int64_t tasks = p.n_groups * p.chunks_per_group * (kChunk / Enc<D, B, false>::VPC);
    encode_pass_kernel<D, B><<<(int)std::min<int64_t>(tasks, grid), kThreads, 0, s>>>(p);
  }
  return cudaGetLastError();
}
template <int D, int B, bool OUTL>
static cudaError_t ev_launch(const EvictParams& p, cudaStream_t s) {
  dim3 grid(p.max_evict, p.B * p.Hkv, p.L);
  evict_kernel<D, B, OUTL><<<grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
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

cudaError_t launch_encode(const EncodeParams& p, int grid, cudaStream_t s) {
  if (p.c.d == 128) return launch_encode_mma(p, grid, s);  // Hadamard stage on the tensor cores
  TQ_DISPATCH_DBO(enc_launch, p.c.d, p.c.bits, p.c.has_outl, p, grid, s);
}

cudaError_t launch_evict(const EvictParams& p, cudaStream_t s) {
  TQ_DISPATCH_DBO(ev_launch, p.c.d, p.c.bits, p.c.has_outl, p, s);
}

cudaError_t launch_evict_commit(const EvictCommitParams& p, cudaStream_t s) {
  const int threads = 128, grid = (p.LB + threads - 1) / threads;
  evict_commit_kernel<<<grid, threads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace tq
