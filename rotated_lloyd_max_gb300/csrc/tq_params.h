// Kernel parameter blocks and launcher declarations shared between the C ABI
// (abi.cu) and the kernel translation units.  Host-visible plain structs.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tq {

// What a kernel needs of a codec, resolved on the host.
struct CodecDev {
  int d, bits, has_outl, cap;
  int scale_mode;  // tq_scale_mode of the stored per-vector scale
  int rec_bytes, off_norm, off_count, off_entries;
  float thr_out;     // T / sqrt(d) in f32 (+inf when T is +inf)
  float inv_sqrt_d;  // f32(1/sqrt(d))
  float inv_sqrt_d_lo;  // 1/sqrt(d) - f32(1/sqrt(d)), rounded to f32
  float sqrt_d;      // f32(sqrt(d))
  float centroids[16];
  float boundaries[15];
  uint32_t signs[16];
};

// Unsigned 32-bit division by a run-time constant as a multiply-high, an add
// and two shifts (Granlund & Montgomery, "Division by invariant integers
// using multiplication", PLDI 1994):  with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1,  n / d = (t + ((n - t) >> 1)) >> (l - 1),
// t = mulhi(m, n), for every n < 2^32.  d = 1 takes m = 0 and no shifts.
struct FastDiv {
  uint32_t d, m, s1, s2;
};
inline FastDiv make_fast_div(uint32_t d) {
  FastDiv f{d, 0u, 0u, 0u};
  if (d > 1) {
    uint32_t l = 0;
    while (l < 32 && (1ull << l) < d) ++l;
    f.m = (uint32_t)(((1ull << 32) * ((1ull << l) - d)) / d + 1);
    f.s1 = 1;
    f.s2 = l - 1;
  }
  return f;
}

struct EncodeParams {
  CodecDev c;
  const uint16_t* src;
  int64_t src_vs, src_gs;  // elements
  uint8_t* dst;
  int64_t dst_gs;  // bytes
  int64_t n_groups, n_vec, first_vec;
  int64_t first_chunk, chunks_per_group;
  FastDiv cpg;       // division by chunks_per_group
  int small_tasks;   // every task index the kernels form (with the grid's lookahead) is below 2^32
};

struct EvictParams {
  CodecDev c;               // codec of the stream this launch encodes
  uint8_t* rec;
  int64_t rec_ls;           // bytes
  int rec_cap;              // records per stream, or blocks per layer pool with a block table
  const int32_t* table;     // block table [B][table_stride] or null (contiguous records)
  int table_stride;
  int rec_limit;            // records a stream may hold: rec_cap, or table_stride when paged
  const uint16_t* tail;
  int64_t tail_ls;          // elements
  int tail_cap;
  const int32_t* n_chunks;
  const int32_t* tail_start;
  const int32_t* tail_len;
  int L, B, Hkv, floor_, max_evict;
};

struct EvictCommitParams {
  int32_t* n_chunks;
  int32_t* tail_start;
  int32_t* tail_len;
  int LB, floor_, max_evict, tail_cap, rec_limit;
};

struct RollbackParams {
  CodecDev c;               // codec of the stream this launch decodes
  const uint8_t* rec;
  int64_t rec_ls;           // bytes
  int rec_cap;              // records per stream, or blocks per layer pool with a block table
  const int32_t* table;     // block table [B][table_stride] or null
  int table_stride;
  int rec_limit;
  uint16_t* tail;           // bf16 ring [L][B][Hkv][tail_cap][D]
  int64_t tail_ls;          // elements
  int tail_cap;
  int32_t* n_chunks;
  int32_t* tail_start;
  int32_t* tail_len;
  const int32_t* new_len;   // [L][B]
  int L, B, Hkv;
};

struct DecodeParams {
  CodecDev c;
  const uint8_t* src;
  int64_t src_gs;  // bytes
  float* dst;
  int64_t dst_vs, dst_gs;  // elements
  int64_t n_groups, n_vec, first_vec;
  int64_t first_chunk, chunks_per_group;
  int log2_parts;  // 2^log2_parts CTAs per record (1, 2 or 4): few records spread their slots over more SMs
};

struct AttnParams {
  int L, B, Hq, Hkv, G, n_hg;
  float sscale;  // softmax scale * log2(e)
  float scap, iscap;  // logit soft cap * log2(e) and its reciprocal; 0, 0 = no cap
  float sv_log2eps;   // sparse-V threshold log2(eps) (< 0), or 0 = every value accumulated
  const uint16_t* q;
  int64_t q_ls, q_bs;
  const uint8_t* krec;
  const uint8_t* vrec;
  int64_t krec_ls, vrec_ls;
  int rec_cap;              // records per stream, or blocks per layer pool with a block table
  const int32_t* table;     // block table [B][table_stride] or null (contiguous records)
  int table_stride;
  int rec_limit;            // records a stream may hold: rec_cap, or table_stride when paged
  int krec_bytes, vrec_bytes;
  int kb, vb, kout, vout, kcap, vcap, shared_kv;
  int k_off_norm, v_off_norm, k_off_count, v_off_count, k_off_ent, v_off_ent;
  int k_main, v_main;  // bytes staged per record (codes, norms, counts)
  float kc[16], vc[16];
  uint32_t ksign[16];
  const uint16_t* ktail;
  const uint16_t* vtail;
  int64_t tail_ls;
  int tail_cap;
  const int32_t* n_chunks;
  const int32_t* tail_start;
  const int32_t* tail_len;
  int S, Sc, cps, tps;
  int split_base;  // index of the first split a launch covers (dense-only launches)
  int groups;      // tensor-core kernel (head dims 64/128): 4-warp groups per CTA (0 = 1)
  float* ws_acc;
  float* ws_ml;
  int* status;  // sticky launch status in the workspace (nonzero: a bounded wait expired)
  // dynamic shared memory carve-up (bytes)
  int sm_q, sm_lut, sm_red, sm_logit, sm_main, sm_stage, sm_ent, sm_ent_stage, sm_pre, sm_slot,
      sm_corr, sm_kpair, sm_vpair, sm_qi, sm_total;
};

struct MergeParams {
  const float* ws_acc;
  const float* ws_ml;
  float* out;
  int rows, S, Sc;
  const int* status;  // nonzero: the attention launch failed, outputs are NaN (may be null)
  float inv_sqrt_d;
  uint32_t vsign[16];
};

// launchers (return the launch status)
cudaError_t launch_codebook(int bits, int d, uint64_t seed, void* scratch, cudaStream_t s);
cudaError_t launch_encode(const EncodeParams& p, int grid, cudaStream_t s);
cudaError_t launch_evict(const EvictParams& p, cudaStream_t s);
cudaError_t launch_evict_commit(const EvictCommitParams& p, cudaStream_t s);
cudaError_t launch_decode(const DecodeParams& p, int grid, cudaStream_t s);
cudaError_t launch_rollback(const RollbackParams& p, cudaStream_t s);
cudaError_t launch_rollback_commit(const RollbackParams& p, cudaStream_t s);
cudaError_t launch_attn(const AttnParams& p, int D, int GT, dim3 grid, cudaStream_t s);
// dense splits of head dim 512 on the tensor cores, 16 query heads per CTA
// (p.n_hg = G / 16, p.split_base = the first dense split)
cudaError_t launch_attn_dense512(const AttnParams& p, dim3 grid, cudaStream_t s);
int attn_dense512_smem_bytes();
// warp-local kernel for the compressed splits (head dims 64 and 128)
cudaError_t launch_attn_rec(const AttnParams& p, int D, int GT, dim3 grid, cudaStream_t s);
// tensor-core kernel for the compressed splits (head dims 64 and 128)
cudaError_t launch_attn_mma(const AttnParams& p, int D, dim3 grid, cudaStream_t s);
// tensor-core kernel for the compressed splits at head dim 512 (256 threads)
cudaError_t launch_attn_mma512(const AttnParams& p, dim3 grid, cudaStream_t s);
// tcgen05 kernel for the compressed splits at head dim 512, up to 64 heads per CTA
cudaError_t launch_attn_umma512(const AttnParams& p, dim3 grid, cudaStream_t s);
int attn_umma512_smem();
cudaError_t launch_merge(const MergeParams& p, int D, cudaStream_t s);

// Dynamic shared memory of the attention kernel for head dim D and head group GT
// (everything but the record-size dependent parts is fixed by D and GT).
void attn_smem_layout(AttnParams& p, int D, int GT);
void attn_rec_smem_layout(AttnParams& p, int D, int GT);
void attn_mma_smem_layout(AttnParams& p, int D);
int attn_mma_groups(const AttnParams& base, int D);
constexpr int kMmaOutlGroups = 3;  // tensor-core kernel with side lists: 4-warp groups per CTA at most
void attn_mma512_smem_layout(AttnParams& p);

// The codebook kernel writes this block into the caller's scratch.
struct CodebookOut {
  float c[16];
  float t[16];
  uint32_t signs[16];
  double mse;
  int iters;
  int pad;
};

}  // namespace tq
