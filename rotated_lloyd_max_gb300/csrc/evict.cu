// Chunked eviction from dense ring-buffer tails into records ("feat(v4):
// TurboQuant KV storage for DeepSeek-V4", "Eviction is chunked, on purpose"):
// device-side decisions, the CUDA-core encoder of encode_core.cuh on the
// due chunks, and a bookkeeping kernel that advances the counters.
#include "encode_core.cuh"

namespace tq {

constexpr int kEvictParts = 4;  // CTAs per chunk without outlier lists (32 slots each)

// Eviction: CTA (e * parts + part, b*Hkv + h, l) encodes part `part` of the
// e-th due chunk of stream (l, b, h).  Without outlier lists the chunk's slots
// are independent and a chunk is split over parts = gridDim.x / max_evict
// CTAs (a single chunk per stream is otherwise a few latency-bound CTAs);
// with them one CTA keeps the chunk, whose entries it orders.
template <int D, int B, bool OUTL, bool SCALE>
__global__ void __launch_bounds__(kThreads) evict_kernel(const __grid_constant__ EvictParams p) {
  __shared__ EncSmem sm;
  const int parts = gridDim.x / p.max_evict;
  const int e = blockIdx.x / parts, part = blockIdx.x % parts;
  const int h = blockIdx.y % p.Hkv, b = blockIdx.y / p.Hkv, l = blockIdx.z;
  const int lb = l * p.B + b;
  const int len = p.tail_len[lb], nch = p.n_chunks[lb];
  const int start = ((p.tail_start[lb] % p.tail_cap) + p.tail_cap) % p.tail_cap;
  const int k = len >= p.floor_ + kChunk ? min((len - p.floor_) / kChunk, p.max_evict) : 0;
  if (e >= k || nch < 0 || nch + k > p.rec_limit) return;
  __shared__ float2 cells[B >= 3 ? kCells : 1];
  __shared__ float cent[16];
  __shared__ __align__(16) float tbuf[D == 512 ? (kThreads / 32) * 2 * kTVec : 4];
  float* tb = tbuf + (threadIdx.x >> 5) * 2 * kTVec;
  if (threadIdx.x < 16) cent[threadIdx.x] = p.c.centroids[threadIdx.x];
  if constexpr (B >= 3) build_cells<true>(p.c, cells);
  __syncthreads();
  uint8_t* rec = p.rec + l * p.rec_ls + rec_offset(p.table, p.table_stride, p.rec_cap, p.Hkv, b, h, nch + e,
                                                    p.c.rec_bytes);
  const uint16_t* tail = p.tail + l * p.tail_ls + (int64_t)(b * p.Hkv + h) * p.tail_cap * D;
  const int first = start + e * kChunk;
  const int cap = p.tail_cap;
  auto row = [&](int slot) { return tail + (int64_t)((first + min(slot, kChunk - 1)) % cap) * D; };
  const int per = kChunk / parts;
  encode_record<D, B, OUTL, SCALE>(p.c, cells, cent, tb, row, rec, part * per, part * per + per, &sm);
}

__global__ void evict_commit_kernel(const EvictCommitParams p) {
  for (int lb = blockIdx.x * blockDim.x + threadIdx.x; lb < p.LB; lb += gridDim.x * blockDim.x) {
    const int len = p.tail_len[lb];
    const int k = len >= p.floor_ + kChunk ? min((len - p.floor_) / kChunk, p.max_evict) : 0;
    if (k == 0 || p.n_chunks[lb] < 0 || p.n_chunks[lb] + k > p.rec_limit) continue;
    const int start = ((p.tail_start[lb] % p.tail_cap) + p.tail_cap) % p.tail_cap;
    p.n_chunks[lb] += k;
    p.tail_start[lb] = (start + k * kChunk) % p.tail_cap;
    p.tail_len[lb] = len - k * kChunk;
  }
}

template <int D, int B, bool OUTL>
static cudaError_t ev_launch(const EvictParams& p, cudaStream_t s) {
  dim3 grid(p.max_evict * (OUTL ? 1 : kEvictParts), p.B * p.Hkv, p.L);
  if (p.c.scale_mode != TQ_SCALE_NORM) evict_kernel<D, B, OUTL, true><<<grid, kThreads, 0, s>>>(p);
  else evict_kernel<D, B, OUTL, false><<<grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
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
