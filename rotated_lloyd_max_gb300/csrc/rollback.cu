// Rollback of the cache to an earlier length, mapped onto both time bases
// ("feat(v4): TurboQuant KV storage for DeepSeek-V4", "What landed": the cache
// reports its length in tokens and maps truncation onto the packed records
// and the dense tail; a deep rollback dequantises).  For a stream with n
// records, a tail of len tokens and new length T (clamped to [0, 128 n + len]):
//   T >= 128 n  the newest tail tokens go: len = T - 128 n;
//   T <  128 n  records r = T / 128 and later go; the m = T - 128 r tokens of
//               record r that stay are decoded to bf16 into ring slots 0..m-1,
//               and the stream becomes n = r, start = 0, len = m.
// rollback_kernel decodes (one CTA per (kv head, batch, layer) and stream);
// rollback_commit_kernel then moves the counters.
#include "decode_core.cuh"

#include <algorithm>

namespace tq {

struct RollbackState {
  int n, len, start, T;
};

__device__ __forceinline__ RollbackState rollback_state(const RollbackParams& p, int lb) {
  RollbackState s;
  s.n = min(max(p.n_chunks[lb], 0), p.rec_limit);
  s.len = min(max(p.tail_len[lb], 0), p.tail_cap);
  s.start = ((p.tail_start[lb] % p.tail_cap) + p.tail_cap) % p.tail_cap;
  s.T = min(max(p.new_len[lb], 0), s.n * kChunk + s.len);
  return s;
}

template <int D, int B, bool OUTL>
__global__ void __launch_bounds__(kThreads) rollback_kernel(const __grid_constant__ RollbackParams p) {
  constexpr int L = D / 32, VPW = 32 / L, VPC = 4 * VPW;
  const int h = blockIdx.x % p.Hkv, b = blockIdx.x / p.Hkv, l = blockIdx.y;
  const int lb = l * p.B + b;
  const RollbackState st = rollback_state(p, lb);
  if (st.T >= st.n * kChunk) return;  // only the tail shrinks: no decode
  const int r = st.T / kChunk, m = st.T - r * kChunk;
  if (m == 0) return;
  __shared__ float lut[16];
  __shared__ int pre[kChunk + 1];
  if (threadIdx.x < 16) lut[threadIdx.x] = p.c.centroids[threadIdx.x & ((1 << B) - 1)];
  const uint8_t* rec = p.rec + l * p.rec_ls + rec_offset(p.table, p.table_stride, p.rec_cap, p.Hkv, b, h, r,
                                                         p.c.rec_bytes);
  if (OUTL) outlier_prefix(rec, p.c, pre);
  __syncthreads();
  uint16_t* ring = p.tail + l * p.tail_ls + (int64_t)(b * p.Hkv + h) * p.tail_cap * D;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, lg = lane % L, vi = lane / L;
  for (int base = 0; base < m; base += VPC) {
    const int slot = base + warp * VPW + vi;
    const bool valid = slot < m;
    float o[32];
    __syncwarp();  // the lanes of a vector meet before the transform's shuffle stages
    decode_lane<D, B, OUTL>(p.c, rec, slot, valid, lut, pre, o);
    if (valid) {
      uint4* dst = reinterpret_cast<uint4*>(ring + (int64_t)slot * D + lg * 32);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          w[j] = (uint32_t)f32_to_bf16_rne(o[8 * k + 2 * j]) | ((uint32_t)f32_to_bf16_rne(o[8 * k + 2 * j + 1]) << 16);
        dst[k] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
}

__global__ void rollback_commit_kernel(const RollbackParams p) {
  for (int lb = blockIdx.x * blockDim.x + threadIdx.x; lb < p.L * p.B; lb += gridDim.x * blockDim.x) {
    const RollbackState st = rollback_state(p, lb);
    if (st.T >= st.n * kChunk) {
      p.tail_len[lb] = st.T - st.n * kChunk;
    } else {
      p.n_chunks[lb] = st.T / kChunk;
      p.tail_start[lb] = 0;
      p.tail_len[lb] = st.T % kChunk;
    }
  }
}

template <int D, int B, bool OUTL>
static cudaError_t rb_launch(const RollbackParams& p, cudaStream_t s) {
  rollback_kernel<D, B, OUTL><<<dim3(p.B * p.Hkv, p.L), kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

#define TQ_CASE(D_, B_)                                                        \
  case D_ * 100 + B_ * 10 + 0: return rb_launch<D_, B_, false>(p, s);          \
  case D_ * 100 + B_ * 10 + 1: return rb_launch<D_, B_, true>(p, s);

cudaError_t launch_rollback(const RollbackParams& p, cudaStream_t s) {
  switch (p.c.d * 100 + p.c.bits * 10 + (p.c.has_outl ? 1 : 0)) {
    TQ_CASE(64, 1) TQ_CASE(64, 2) TQ_CASE(64, 3) TQ_CASE(64, 4)
    TQ_CASE(128, 1) TQ_CASE(128, 2) TQ_CASE(128, 3) TQ_CASE(128, 4)
    TQ_CASE(256, 1) TQ_CASE(256, 2) TQ_CASE(256, 3) TQ_CASE(256, 4)
    TQ_CASE(512, 1) TQ_CASE(512, 2) TQ_CASE(512, 3) TQ_CASE(512, 4)
    default: return cudaErrorInvalidValue;
  }
}
#undef TQ_CASE

cudaError_t launch_rollback_commit(const RollbackParams& p, cudaStream_t s) {
  const int threads = 128, grid = std::max(1, (p.L * p.B + threads - 1) / threads);
  rollback_commit_kernel<<<grid, threads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace tq
