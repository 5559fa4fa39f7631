// Encode bf16 head vectors into 128-token records on the CUDA cores (head
// dims 64, 256 and 512; head dim 128 goes to the tensor-core encoder of
// encode_mma.cu).  The per-vector arithmetic is in encode_core.cuh.
#include "encode_core.cuh"

namespace tq {

// Record-aligned encode with outliers: one CTA per record (grid-stride).
template <int D, int B, bool SCALE>
__global__ void __launch_bounds__(kThreads) encode_record_kernel(const __grid_constant__ EncodeParams p) {
  __shared__ EncSmem sm;
  __shared__ __align__(16) float tbuf[D == 512 ? (kThreads / 32) * 2 * kTVec : 4];
  float* tb = tbuf + (threadIdx.x >> 5) * 2 * kTVec;
  __shared__ float2 cells[B >= 3 ? kCells : 1];
  __shared__ float cent[16];
  if (threadIdx.x < 16) cent[threadIdx.x] = p.c.centroids[threadIdx.x];
  if constexpr (B >= 3) build_cells<true>(p.c, cells);
  __syncthreads();
  const int64_t n_tasks = p.n_groups * p.chunks_per_group;
  for (int64_t task = blockIdx.x; task < n_tasks; task += gridDim.x) {
    const int64_t g = task / p.chunks_per_group;
    const int64_t ci = p.first_chunk + task % p.chunks_per_group;
    const int64_t lo = max(p.first_vec, ci * kChunk), hi = min(p.first_vec + p.n_vec, (ci + 1) * kChunk);
    uint8_t* rec = p.dst + g * p.dst_gs + ci * (int64_t)p.c.rec_bytes;
    const uint16_t* src_g = p.src + g * p.src_gs;
    const int64_t vs = p.src_vs, v0 = ci * kChunk - p.first_vec;
    auto row = [&](int slot) { return src_g + (v0 + slot) * vs; };
    encode_record<D, B, true, SCALE>(p.c, cells, cent, tb, row, rec, (int)(lo - ci * kChunk), (int)(hi - ci * kChunk),
                                     &sm);
  }
}

// Encode without outliers: every (group, record, pass) is an independent task
// of VPC vectors; CTAs stride over tasks with the next task's loads in flight.
template <int D, int B, bool SCALE>
__global__ void __launch_bounds__(kThreads) encode_pass_kernel(const __grid_constant__ EncodeParams p) {
  using E = Enc<D, B, false>;
  constexpr int PPR = kChunk / E::VPC;  // passes per record
  __shared__ float2 cells[B >= 3 ? kCells : 1];
  __shared__ float cent[16];
  __shared__ __align__(16) float tbuf[D == 512 ? (kThreads / 32) * 2 * kTVec : 4];
  float* tb = tbuf + (threadIdx.x >> 5) * 2 * kTVec;
  if (threadIdx.x < 16) cent[threadIdx.x] = p.c.centroids[threadIdx.x];
  if constexpr (B >= 3) build_cells<true>(p.c, cells);
  __syncthreads();
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
    enc_vector<D, B, false, SCALE>(p.c, ln, cells, tb, w, cvalid, rec, (int)(ctok % kChunk), x, inv, omask, cent);
  }
}

template <int D, int B, bool OUTL>
static cudaError_t enc_launch(const EncodeParams& p, int grid, cudaStream_t s) {
  const bool sc = p.c.scale_mode != TQ_SCALE_NORM;
  if constexpr (OUTL) {
    const int64_t tasks = p.n_groups * p.chunks_per_group;
    const int g = (int)std::min<int64_t>(tasks, grid);
    if (sc) encode_record_kernel<D, B, true><<<g, kThreads, 0, s>>>(p);
    else encode_record_kernel<D, B, false><<<g, kThreads, 0, s>>>(p);
  } else {
    const int64_t tasks = p.n_groups * p.chunks_per_group * (kChunk / Enc<D, B, false>::VPC);
    const int g = (int)std::min<int64_t>(tasks, grid);
    if (sc) encode_pass_kernel<D, B, true><<<g, kThreads, 0, s>>>(p);
    else encode_pass_kernel<D, B, false><<<g, kThreads, 0, s>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_encode(const EncodeParams& p, int grid, cudaStream_t s) {
  // head dims 128, 256, 512: the 16-point Hadamard stage on the tensor cores
  if (p.c.d >= 128) return launch_encode_mma(p, grid, s);
  TQ_DISPATCH_DBO(enc_launch, p.c.d, p.c.bits, p.c.has_outl, p, grid, s);
}

}  // namespace tq
