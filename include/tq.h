/*
 * tq.h -- C ABI of the GB300 (sm_103a) rotated Lloyd-Max KV-cache codec and
 * the fused decode attention that reads it.
 *
 * The codec stores each K/V head vector x (head_dim d, bf16) as
 *   n = ||x|| (f32);  y = H (s . x/n) / sqrt(d)   (s: seeded +-1 signs, H:
 *   Sylvester Walsh-Hadamard);  code_j = index of the nearest of 2^b Gaussian
 *   Lloyd-Max centroids for N(0, 1/d);  codes bit-packed; optionally the
 *   coordinates with |y_j| > T/sqrt(d) kept as (u16 index, bf16 value).
 * Sources: "v1.3 PPL on vLLM" (LLM-KV--Cache-compress PR #15), M4 Phase A/B and
 * M5 commits (rotate = H.D.x, per-row scale, Lloyd-Max argmin, outlier
 * overrides applied before the inverse WHT); larql PR #196, turbo-quant note
 * (one N(0,1) table per bit width scaled by 1/sqrt(d), append-only encode);
 * "feat(v4): TurboQuant KV storage for DeepSeek-V4" (arc PR #98), "What landed"
 * (packed records with the norm inside, 260 B/token at d = 512, b = 4),
 * "Eviction is chunked, on purpose" (EVICT_CHUNK = 128; tail bound
 * window + max(t_q-1, margin) + chunk), "Also: two silently-ignored kernel
 * parameters" (query stride honoured; no silent no-op on an unsupported head
 * dim).
 *
 * Conventions for every call:
 *  - Pointers named d_* or documented "device" are device addresses; the
 *    caller owns every buffer (inputs, outputs, workspaces).  The library
 *    allocates no memory and keeps no state between calls, with one
 *    exception: tq_decode_attn_noalloc's fixed device workspace (a static
 *    array of the library) and the per-device address of that array, which
 *    it looks up once and caches.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *    asynchronous on that stream unless stated otherwise.
 *  - Arguments are validated on the host before anything is launched; on an
 *    error nothing is launched and the status says why.  A launch failure
 *    returns TQ_ERR_CUDA.  There is no CPU fallback and no silent no-op.
 *  - bf16 data are raw 16-bit patterns; f32 little-endian.
 *
 * Record format (one record = 128 consecutive tokens of one stream):
 *   offset 0           codes: 128 rows of d*b/8 bytes; row i = token slot i;
 *                      code j occupies bits [j*b, j*b + b) of the row's
 *                      little-endian bitstream (bit k = bit k%8 of byte k/8)
 *   128*d*b/8          norms: 128 x f32
 *   when outlier_T != 0:
 *   + 512              ocount: 128 x u8, entries stored for each slot
 *   + 128              entries: outlier_cap x {u16 index, u16 bf16 value},
 *                      in (slot, index) order; a slot stores at most 255 and
 *                      a record at most outlier_cap; the rest keep their code
 *   The size is a multiple of 16 bytes (tq_record_bytes).  Slots not yet
 *   written (a partially filled last record) are unspecified.
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size or stride */
  TQ_ERR_UNSUPPORTED = 2, /* head_dim not in {64,128,256,512}, bits not in 1..4, ... */
  TQ_ERR_WORKSPACE = 3,   /* workspace or scratch smaller than required */
  TQ_ERR_CUDA = 4         /* a CUDA call or launch failed */
} tq_status;

#define TQ_CHUNK 128

/* Human-readable name of a status code (static storage). */
const char* tq_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int tq_version(void);

/*
 * Per-vector scale stored in a record's f32 "norm" field (decode multiplies
 * H(yhat) by it).  With chat the dequantised rotated unit vector (centroids,
 * outlier values at the vector's outlier coordinates) and c = s.H(chat)/sqrt(d)
 * its image in the original basis (turboquant_plus commit log: the
 * EDEN-scale commits and their Appendix A note):
 *   TQ_SCALE_NORM           ||x||                 (the plain codec)
 *   TQ_SCALE_MATCHED_NORM   ||x|| / ||chat||      the decoded vector keeps ||x||
 *   TQ_SCALE_INNER_PRODUCT  ||x||^2 / <c, x>      <xhat, x> = ||x||^2
 *   TQ_SCALE_LEAST_SQUARES  <c, x> / ||c||^2      minimises ||x - xhat||^2
 * The last two multiply to the square of the matched norm.  Codes and
 * outlier lists do not depend on the mode; a zero vector stores 0.
 */
typedef enum {
  TQ_SCALE_NORM = 0,
  TQ_SCALE_MATCHED_NORM = 1,
  TQ_SCALE_INNER_PRODUCT = 2,
  TQ_SCALE_LEAST_SQUARES = 3
} tq_scale_mode;

/*
 * Codec description, passed by pointer and read on the host at every call.
 * Filled by tq_make_codebook; plain data, copy freely.
 */
typedef struct {
  int32_t head_dim;       /* d: 64, 128, 256 or 512 */
  int32_t bits;           /* b: 1..4 */
  uint64_t sign_seed;     /* seed of the SplitMix64 sign diagonal */
  float outlier_T;        /* 0: no outlier section; > 0: keep |y_j| > T/sqrt(d) (may be +inf) */
  int32_t outlier_cap;    /* outlier entries per record (multiple of 4) */
  float centroids[16];    /* 2^b ascending f32 centroids (the Gaussian N(0, 1/d) table, or a
                             caller's table set by tq_codec_set_centroids) */
  float boundaries[15];   /* 2^b - 1 f32 midpoints of consecutive centroids */
  uint32_t sign_bits[16]; /* bit j%32 of word j/32 set <=> s_j = -1 */
  int32_t scale_mode;     /* tq_scale_mode; tq_make_codebook sets TQ_SCALE_NORM */
} tq_codec;

/* Device scratch tq_make_codebook needs (bytes). */
size_t tq_codebook_scratch_bytes(void);

/*
 * Codebook and signs: Gaussian Lloyd-Max table and sign diagonal.  Runs the 1-D Lloyd
 * iteration t_k = (c_k + c_{k+1})/2, c_k = E[X | t_{k-1} < X <= t_k] on the
 * N(0,1) density in fp64 on the device until no centroid moves by more than
 * 1e-14, scales by 1/sqrt(d), rounds to f32 and derives the f32 midpoints;
 * draws the signs s_j from SplitMix64(sign_seed) (top bit set -> -1).
 *   d_scratch: device buffer of tq_codebook_scratch_bytes(), 16-byte aligned.
 *   outlier_cap: 0 selects 4*ceil(0.08*128*d/4) (8% of a record's coordinates).
 *   out: host; filled on success.  mse_out: host, nullable: E[(X-Q(X))^2] of
 *   the unit-variance table.
 * SYNCHRONISES `stream` (the table is returned in host memory).
 */
tq_status tq_make_codebook(int bits, int head_dim, uint64_t sign_seed, float outlier_T,
                           int outlier_cap, void* d_scratch, size_t scratch_bytes, tq_codec* out,
                           double* mse_out, void* stream);

/*
 * Replace a codec's table by a caller's ascending f32 centroid table of 2^b
 * values (a calibrated table: "v1.3 PPL on vLLM" (PR #15), the calibrated
 * Lloyd-Max commit, loads a sorted 2^b f32 table in place of the Gaussian
 * one).  Host only.  Sets centroids[] and boundaries[] (f32 midpoints of
 * consecutive centroids, computed in double); every other field is kept.
 * The table must be strictly ascending and symmetric (c_k = -c_{2^b-1-k}),
 * with |c_k| < 0.999 (the tensor-core attention holds centroids x 2^16 in
 * f16), and for b >= 2 consecutive boundaries at least 1/128 apart (the
 * encoders decide codes through 1/128-wide cells holding one boundary each):
 * TQ_ERR_INVALID_ARG for an unordered or non-finite table, TQ_ERR_UNSUPPORTED
 * for one breaking the other conditions; the codec is unchanged on error.
 */
tq_status tq_codec_set_centroids(tq_codec* codec, const float* centroids, int n_centroids);

/* Bytes of one 128-token record of this codec; 0 if the codec is invalid. */
size_t tq_record_bytes(const tq_codec* codec);

/*
 * Encode.  n_groups independent streams of n_vec bf16 vectors each;
 * vector i of group g is read at src + g*src_group_stride + i*src_vec_stride
 * (elements) and written as token first_vec + i of the record array at
 * dst + g*dst_group_stride (bytes).
 *   src: device, 16-byte aligned; strides multiples of 8 elements.
 *   dst: device, 16-byte aligned; dst_group_stride multiple of 16.
 *   With outliers, first_vec must be a multiple of 128 (a record's outlier
 *   section is written whole by one call).  Encoding is append-only: records
 *   and slots outside the written range are not touched.
 */
tq_status tq_encode(const tq_codec* codec, const void* src, int64_t n_groups, int64_t n_vec,
                    int64_t src_vec_stride, int64_t src_group_stride, void* dst,
                    int64_t dst_group_stride, int64_t first_vec, void* stream);

/*
 * Decode.  Tokens [first_vec, first_vec + n_vec) of each group's record
 * array (at src + g*src_group_stride bytes) to f32 vectors
 *   xhat = n * s . H(yhat) / sqrt(d),  yhat_j = centroid[code_j], replaced by
 *   the stored value at outlier coordinates,
 * written at dst + g*dst_group_stride + i*dst_vec_stride (elements).
 *   src: device, 16-byte aligned.  dst: device, 16-byte aligned, strides
 *   multiples of 4 elements.
 */
tq_status tq_decode(const tq_codec* codec, const void* src, int64_t n_groups, int64_t n_vec,
                    int64_t src_group_stride, int64_t first_vec, float* dst,
                    int64_t dst_vec_stride, int64_t dst_group_stride, void* stream);

/*
 * Chunked eviction from dense bf16 ring-buffer tails into records, for
 * n_layers x batch x n_kv_heads streams in one launch (plus one small
 * bookkeeping launch), with every decision taken on the device (no host
 * synchronisation).  For each (layer, batch) with counters
 *   len = tail_len[l][b], start = tail_start[l][b], n = n_chunks[l][b]:
 *   floor = window + max(t_q - 1, margin);  k = len >= floor + 128 ?
 *   min((len - floor) / 128, max_evict) : 0;
 * tokens at ring slots (start + e*128 + i) % tail_cap, e < k, i < 128, are
 * encoded into record n + e of every kv head, then n += k, start advances by
 * 128k (mod tail_cap), len -= 128k.  Records that would reach rec_cap are not
 * written and the counters of that (layer, batch) are left unchanged.
 * tail_cap must be at least floor + 128 (otherwise the tail could never reach
 * the eviction bound): TQ_ERR_INVALID_ARG.
 */
typedef struct {
  int32_t n_layers, batch, n_kv_heads;
  /* records: layer l, batch b, head h, record r at
   *   k_rec + l*k_rec_layer_stride + ((b*n_kv_heads + h)*rec_cap + r)*record_bytes */
  void* k_rec;
  void* v_rec; /* may equal k_rec with v codec == k codec: keys and values share records */
  int64_t k_rec_layer_stride, v_rec_layer_stride; /* bytes, multiples of 16 */
  int32_t rec_cap;
  /* tails: bf16 [L][B][Hkv][tail_cap][d] at k_tail + l*tail_layer_stride (elements) */
  const void* k_tail;
  const void* v_tail;
  int64_t tail_layer_stride;
  int32_t tail_cap;
  int32_t* n_chunks;   /* device [L][B] */
  int32_t* tail_start; /* device [L][B] */
  int32_t* tail_len;   /* device [L][B] */
  int32_t window, margin, t_q;
  int32_t max_evict;   /* upper bound on records written per (layer, batch) per call */
  /* Paged records (optional; NULL = the contiguous layout above).  With a block
   * table the record arrays are per-layer pools of rec_cap blocks, each block
   * holding one record per kv head: record r of (l, b, h) sits at
   *   k_rec + l*k_rec_layer_stride + (block_table[b*table_stride + r]*n_kv_heads + h)*record_bytes
   * (likewise v_rec).  block_table: device int32 [batch][table_stride], shared
   * by every layer and by keys and values; a sequence holds at most
   * table_stride records.  The caller fills block_table[b][n_chunks[l][b] + e]
   * before a call can evict into it; entries outside [0, rec_cap) are clamped
   * into the pool (never an out-of-bounds access). */
  const int32_t* block_table;
  int32_t table_stride;
} tq_evict_args;

tq_status tq_evict(const tq_codec* k_codec, const tq_codec* v_codec, const tq_evict_args* args,
                   void* stream);

/*
 * Rollback: truncate every (layer, batch) stream of a cache to new_len[l][b]
 * tokens, mapping the truncation onto both time bases ("feat(v4): TurboQuant
 * KV storage for DeepSeek-V4", "What landed": length reported in tokens,
 * truncation mapped onto the packed records and the dense tail; a deep
 * rollback dequantises).  With n = n_chunks, len = tail_len and
 * T = min(max(new_len, 0), 128 n + len):
 *   T >= 128 n: tail_len = T - 128 n (the newest tail tokens go; start kept);
 *   T <  128 n: records r = T / 128 and later go; the m = T - 128 r tokens of
 *               record r that remain are decoded (as tq_decode computes them)
 *               and rounded to bf16 (nearest, ties to even) into ring slots
 *               0 .. m-1 of every kv head (K and V), then n_chunks = r,
 *               tail_start = 0, tail_len = m.
 * Records are only read; the dropped ones keep their bytes and are
 * overwritten by later evictions.  Every decision runs on the device (two
 * launches per stream kind plus one bookkeeping launch, no host sync).
 *   args: the cache as for tq_evict (window, margin, t_q and max_evict are
 *   not used); new_len: device int32 [n_layers][batch].
 */
tq_status tq_rollback(const tq_codec* k_codec, const tq_codec* v_codec, const tq_evict_args* args,
                      const int32_t* new_len, void* stream);

/*
 * Fused decode attention (query rotation, scoring of the compressed keys,
 * online softmax, values in the rotated basis, dense tail, split-K merge
 * with one inverse transform) for one group of layers sharing codecs and
 * geometry.  For layer l, batch b, query head h (kv head h / (Hq/Hkv)):
 *   out = sum_i softmax_i(cap(scale * q . k_i)) v_i  over the layer's compressed
 * tokens (records 0..n_chunks-1, scored in the rotated basis against
 * q~ = H(s_k . q)/sqrt(d) from a shared-memory centroid table, values
 * accumulated as sum p_i n_i yhat_i and brought back by one inverse
 * transform) and its dense bf16 tokens (ring slots (tail_start + t) % tail_cap,
 * t < tail_len), with split-K over context and a merge of the splits.
 * Layers without records (k_codec == NULL) are dense bf16 layers: set
 * k_rec = v_rec = NULL, n_chunks = tail_start = NULL and pass the whole cache
 * as the "tail" (tail_len = context length).
 */
typedef struct {
  int32_t n_layers, batch, n_q_heads, n_kv_heads, head_dim;
  float scale; /* softmax scale applied to q . k */
  /* q: bf16, element (l, b, h, j) at q + l*q_layer_stride + b*q_batch_stride + h*d + j */
  const void* q;
  int64_t q_layer_stride, q_batch_stride; /* elements, multiples of 8 */
  /* out: f32 [L][B][Hq][d], contiguous, 16-byte aligned */
  float* out;
  const void* k_rec; /* records as in tq_evict_args; NULL for dense layers */
  const void* v_rec;
  int64_t k_rec_layer_stride, v_rec_layer_stride;
  int32_t rec_cap;
  const void* k_tail; /* bf16 [L][B][Hkv][tail_cap][d]; NULL when there is no dense part */
  const void* v_tail;
  int64_t tail_layer_stride; /* elements */
  int32_t tail_cap;
  const int32_t* n_chunks;   /* device [L][B]; NULL = 0 */
  const int32_t* tail_start; /* device [L][B]; NULL = 0 */
  const int32_t* tail_len;   /* device [L][B]; NULL = 0 */
  int32_t max_chunks;        /* host upper bound of n_chunks (sizes the grid) */
  int32_t max_tail;          /* host upper bound of tail_len */
  int32_t splits;            /* splits per (layer, batch, kv head); 0 = automatic */
  /* 0: automatic.  Compressed tokens of codecs without outlier side lists
   * run on the tensor cores with f16 hi/lo operand splits and f32
   * accumulation: at head dim 512 with 16-64 query heads per kv head (a
   * multiple of 8) or a multiple of 64, on the fifth-generation tensor cores
   * (tcgen05, accumulators in tensor memory); at head dims 64, 128 and the
   * other head-dim-512 groups on mma.sync.  With side lists at head dims 64
   * and 128, the mma.sync kernel (corrections applied beside the MMAs) takes
   * sparse-V calls.  Everything else runs on the CUDA-core kernel (f32 FMA
   * from the centroid table).
   * 1: always the CUDA-core kernel.  2: as 0 but never tcgen05 (the
   * mma.sync kernels).  All paths meet the same tolerance. */
  int32_t cuda_core_path;
  /* Logit soft cap (arc PR #98, softcapping fix): each logit s = scale * q . k
   * becomes softcap * tanh(s / softcap) before it enters the softmax (its
   * maximum included), for compressed and dense tokens alike.  0 = no cap;
   * otherwise finite and > 0 (1.0 is an ordinary cap, not "off"). */
  float softcap;
  /* Paged records, as in tq_evict_args (NULL = contiguous): record r of
   * (l, b, h) is block block_table[b*table_stride + r] of layer l's pool of
   * rec_cap blocks of n_kv_heads records; max_chunks <= table_stride. */
  const int32_t* block_table;
  int32_t table_stride;
  /* Sparse-V (turboquant_plus commit log, "safer-asym + sparse-V dequant":
   * value dequantisation skipped where the post-softmax weight is
   * negligible).  0 = off.  With 0 < eps < 1, the tensor-core kernel for head
   * dims 64/128 skips the value work of a warp's 32 tokens of a record when,
   * for every query head of its CTA, each of their logits lies below
   * (the maximum logit of the warp's earlier records of the same split) +
   * ln(eps); their weights still count in the softmax denominator, so each
   * output coordinate moves by at most eps * (skipped tokens) * max|v|.
   * Which blocks a warp visits follows the plan (records_per_split,
   * heads_per_cta of tq_decode_attn_plan; warp w holds tokens 32w..32w+31 of
   * each record).  Dense tokens are never skipped.  Another kernel route for
   * the compressed tokens (head dims 256/512, cuda_core_path != 0) with
   * eps > 0: TQ_ERR_UNSUPPORTED. */
  float sparse_v_eps;
} tq_attn_args;

/* Kernels that run split-K decode attention (tq_attn_plan). */
typedef enum {
  TQ_ATTN_KERNEL_NONE = 0,           /* no split of this kind */
  TQ_ATTN_KERNEL_CUDA_CORE = 1,      /* f32 FMA from the centroid table, CTA-wide softmax per tile */
  TQ_ATTN_KERNEL_CUDA_CORE_WARP = 2, /* f32 FMA, warp-local softmax (head dims 64/128; outlier side lists) */
  TQ_ATTN_KERNEL_MMA = 3,            /* mma.sync f16 hi/lo splits, head dims 64/128 (side lists: sparse-V) */
  TQ_ATTN_KERNEL_MMA512 = 4,         /* mma.sync at head dim 512 (records: f16 hi/lo splits; dense: bf16, 16 heads a CTA) */
  TQ_ATTN_KERNEL_TCGEN05 = 5         /* tcgen05 with tensor-memory accumulators, head dim 512 */
} tq_attn_kernel;

/* What tq_decode_attn launches for given arguments.  Splits are per
 * (layer, batch, kv head, head group); a head group is the query heads one
 * CTA serves. */
typedef struct {
  int32_t compressed_kernel;      /* tq_attn_kernel of the splits over records */
  int32_t dense_kernel;           /* tq_attn_kernel of the splits over dense tokens */
  int32_t compressed_splits;
  int32_t dense_splits;
  int32_t records_per_split;      /* at most; 0 without compressed splits */
  int32_t dense_tokens_per_split; /* at most; 0 without dense splits */
  int32_t heads_per_cta;          /* query heads per CTA of the compressed splits */
  int32_t dense_heads_per_cta;    /* query heads per CTA of the dense splits */
  int32_t launches;               /* kernel launches of the call, the merge included */
  int32_t warps_per_cta;          /* warps per CTA of the compressed splits */
  uint64_t workspace_bytes;       /* = tq_decode_attn_workspace_size */
} tq_attn_plan;

/* Fills *plan with the kernels, split counts and launches tq_decode_attn
 * would use for these arguments.  Host only: no device work, no allocation;
 * it plans with the current device's SM count and shared memory (GB300's 152
 * SMs and 227 KB when no device is visible).  Errors as tq_decode_attn's
 * argument checks; TQ_ERR_INVALID_ARG when plan is NULL. */
tq_status tq_decode_attn_plan(const tq_attn_args* args, const tq_codec* k_codec, const tq_codec* v_codec,
                              tq_attn_plan* plan);

/* Workspace bytes tq_decode_attn needs for these arguments (0 on invalid args). */
size_t tq_decode_attn_workspace_size(const tq_attn_args* args, const tq_codec* k_codec,
                                     const tq_codec* v_codec);

/* workspace: device, 256-byte aligned, >= tq_decode_attn_workspace_size bytes.
 * Its contents need no initialisation and are garbage afterwards.  An empty
 * context (no compressed and no dense token) yields a zero output row.
 * The tcgen05 kernel bounds every internal wait (about two seconds); if one
 * expires (a fault of the device, not of the arguments) the call's outputs
 * are NaN rather than wrong numbers. */
tq_status tq_decode_attn(const tq_attn_args* args, const tq_codec* k_codec,
                         const tq_codec* v_codec, void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * Allocation-free variant of tq_decode_attn.  The pages describe no such
 * call; it exists for callers that cannot allocate device memory at the time
 * they run attention (their device memory is reserved up front by a host
 * framework or pooling allocator, a plugin enqueue step that must not
 * allocate, or a latency-critical loop that cannot take cudaMalloc's implicit
 * synchronisation).
 *   Same arguments and results as tq_decode_attn, but the split-K workspace is
 *   a fixed device array inside the library of TQ_NOALLOC_WORKSPACE_BYTES
 *   (8 MiB), present on every GPU that loads the library until the process
 *   exits.  A call needing more (tq_decode_attn_workspace_size) is rejected
 *   with TQ_ERR_WORKSPACE; lower `splits` or use tq_decode_attn.
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any
 *   stream capture.  The cached address does not survive cudaDeviceReset:
 *   after a reset of a device, do not call this entry point on it again in
 *   the same process.  Nothing in the array needs to start at zero, and each
 *   call overwrites what the previous one left.  All calls share the one
 *   array: calls whose executions overlap on the GPU (different streams,
 *   concurrent graph branches) race and corrupt each other's results.
 */
#define TQ_NOALLOC_WORKSPACE_BYTES (8u << 20)
tq_status tq_decode_attn_noalloc(const tq_attn_args* args, const tq_codec* k_codec,
                                 const tq_codec* v_codec, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* TQ_H_ */
