// The C ABI (include/tq.h): host-side validation, codec resolution, split
// planning and kernel dispatch.  Every argument is checked before anything is
// launched; there is no CPU fallback and no silent no-op (arc PR #98, "Also:
// two silently-ignored kernel parameters": an unsupported head dim must fail,
// not return early leaving the output uninitialised).
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/tq.h"
#include "tq_params.h"

using namespace tq;

namespace {

constexpr int kVersion = 10000;  // 1.0.0

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline bool dim_ok(int d) { return d == 64 || d == 128 || d == 256 || d == 512; }

int default_cap(int d) { return 4 * ((8 * TQ_CHUNK * d + 399) / 400); }

// record layout: codes, norms, [counts, entries]
int record_layout(int d, int bits, bool outl, int cap, int* off_norm, int* off_count, int* off_ent) {
  const int codes = TQ_CHUNK * d * bits / 8;
  *off_norm = codes;
  *off_count = codes + 4 * TQ_CHUNK;
  *off_ent = *off_count + TQ_CHUNK;
  return outl ? *off_ent + 4 * cap : *off_count;
}

// What the kernels need of any table: centroids below 0.999 in magnitude (the
// tensor-core attention holds centroid x 2^16 as f16 hi/lo halves) and, at
// b >= 2, consecutive boundaries at least one decision cell (1/128) apart with
// every boundary inside (-1, 1) (the encoders' cell table holds one boundary
// per cell of width 1/128 over |y| <= 1).
tq_status table_supported(const float* cent, const float* bnd, int b) {
  const int K = 1 << b;
  for (int k = 0; k < K; ++k)
    if (!(std::fabs(cent[k]) < 0.999f)) return TQ_ERR_UNSUPPORTED;
  if (b >= 2)
    for (int k = 0; k + 1 < K; ++k) {
      if (!(std::fabs(bnd[k]) < 1.0f)) return TQ_ERR_UNSUPPORTED;
      if (k + 2 < K && (double)bnd[k + 1] - (double)bnd[k] < 1.0 / 128.0) return TQ_ERR_UNSUPPORTED;
    }
  return TQ_OK;
}

tq_status resolve_codec(const tq_codec* c, CodecDev* o) {
  if (!c) return TQ_ERR_INVALID_ARG;
  const int d = c->head_dim, b = c->bits;
  if (!dim_ok(d) || b < 1 || b > 4) return TQ_ERR_UNSUPPORTED;
  if (!(c->outlier_T >= 0.f)) return TQ_ERR_INVALID_ARG;  // negative or NaN
  const bool outl = c->outlier_T != 0.f;
  if (outl && (c->outlier_cap <= 0 || c->outlier_cap % 4 != 0 || c->outlier_cap > 65536))
    return TQ_ERR_INVALID_ARG;
  const int K = 1 << b;
  for (int k = 0; k + 1 < K; ++k) {
    if (!(c->centroids[k] < c->boundaries[k] && c->boundaries[k] < c->centroids[k + 1]))
      return TQ_ERR_INVALID_ARG;  // not ascending / boundaries not between centroids
    if (c->boundaries[k] != -c->boundaries[K - 2 - k]) return TQ_ERR_UNSUPPORTED;  // asymmetric table
  }
  const tq_status tab = table_supported(c->centroids, c->boundaries, b);
  if (tab != TQ_OK) return tab;
  if (c->scale_mode < TQ_SCALE_NORM || c->scale_mode > TQ_SCALE_LEAST_SQUARES) return TQ_ERR_INVALID_ARG;
  std::memset(o, 0, sizeof(*o));
  o->d = d;
  o->bits = b;
  o->has_outl = outl ? 1 : 0;
  o->cap = outl ? c->outlier_cap : 0;
  o->scale_mode = c->scale_mode;
  o->rec_bytes = record_layout(d, b, outl, o->cap, &o->off_norm, &o->off_count, &o->off_entries);
  o->thr_out = outl ? (float)((double)c->outlier_T / std::sqrt((double)d)) : INFINITY;
  o->inv_sqrt_d = (float)(1.0 / std::sqrt((double)d));
  o->inv_sqrt_d_lo = (float)(1.0 / std::sqrt((double)d) - (double)o->inv_sqrt_d);
  o->sqrt_d = (float)std::sqrt((double)d);
  for (int k = 0; k < 16; ++k) o->centroids[k] = c->centroids[k & (K - 1)];
  for (int k = 0; k < 15; ++k) o->boundaries[k] = k + 1 < K ? c->boundaries[k] : 0.f;
  for (int w = 0; w < 16; ++w) o->signs[w] = w < d / 32 ? c->sign_bits[w] : 0u;
  return TQ_OK;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
  return n;
}

int max_dyn_smem() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 227 * 1024;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 227 * 1024;
  return n;
}

// Bytes of a record the head-dim 64/128 tensor-core kernel stages per CTA
// iteration: codes and scales, and with side lists the per-slot counts and
// the first entries of the list (a record's list is about 6 entries per slot
// at T = 2, 740 of them; entries past the staged ones are read from global memory).
constexpr int kMmaStagedEntries = 896;
int mma_stage_bytes(const CodecDev& c) {
  return c.has_outl ? c.off_entries + 4 * std::min(c.cap, kMmaStagedEntries) : c.off_count;
}

// ----------------------------------------------------------------- attention plan
struct Plan {
  int D, G, GT, n_hg, S, Sc, cps, tps;
  int64_t rows;
  size_t ws_acc_bytes, ws_bytes;
  CodecDev kc, vc;
  bool has_rec, has_tail, shared;
  bool mma;     // tensor-core kernel (head dims 64/128)
  int groups;   // its 4-warp groups per CTA
  bool mma512;  // tensor-core kernel at head dim 512 (mma.sync)
  bool umma512; // tcgen05 kernel at head dim 512 (groups of up to 64 heads per CTA)
  bool dense512; // their dense splits on the tensor cores (groups of 16 heads per CTA)
  size_t ws_status_off;
};

tq_status make_plan(const tq_attn_args* a, const tq_codec* kcod, const tq_codec* vcod, Plan* pl) {
  if (!a) return TQ_ERR_INVALID_ARG;
  std::memset(pl, 0, sizeof(*pl));
  const int D = a->head_dim;
  if (!dim_ok(D)) return TQ_ERR_UNSUPPORTED;
  if (a->n_layers <= 0 || a->n_layers > 65535 || a->batch <= 0 || a->n_q_heads <= 0 ||
      a->n_kv_heads <= 0 || a->n_q_heads % a->n_kv_heads != 0)
    return TQ_ERR_INVALID_ARG;
  if (!a->q || !a->out || !aligned(a->q, 16) || !aligned(a->out, 16)) return TQ_ERR_INVALID_ARG;
  if (a->q_layer_stride < 0 || a->q_batch_stride < 0 || a->q_layer_stride % 8 || a->q_batch_stride % 8)
    return TQ_ERR_INVALID_ARG;
  if (!(std::isfinite(a->scale))) return TQ_ERR_INVALID_ARG;
  if (!(std::isfinite(a->softcap)) || a->softcap < 0.f) return TQ_ERR_INVALID_ARG;
  if (a->max_chunks < 0 || a->max_tail < 0 || a->splits < 0) return TQ_ERR_INVALID_ARG;
  pl->D = D;
  pl->G = a->n_q_heads / a->n_kv_heads;
  const int cand[5] = {8, 6, 4, 2, 1};
  for (int c : cand)
    if (pl->G % c == 0) { pl->GT = c; break; }
  pl->n_hg = pl->G / pl->GT;
  if ((int64_t)a->batch * a->n_kv_heads * pl->n_hg > 65535) return TQ_ERR_UNSUPPORTED;

  pl->has_rec = a->k_rec != nullptr;
  if (pl->has_rec) {
    if (!kcod || !vcod || !a->v_rec) return TQ_ERR_INVALID_ARG;
    tq_status st = resolve_codec(kcod, &pl->kc);
    if (st != TQ_OK) return st;
    st = resolve_codec(vcod, &pl->vc);
    if (st != TQ_OK) return st;
    if (pl->kc.d != D || pl->vc.d != D) return TQ_ERR_INVALID_ARG;
    pl->shared = a->v_rec == a->k_rec;
    if (pl->shared && std::memcmp(kcod, vcod, sizeof(tq_codec)) != 0) return TQ_ERR_INVALID_ARG;
    if (!aligned(a->k_rec, 16) || !aligned(a->v_rec, 16) || a->k_rec_layer_stride % 16 ||
        a->v_rec_layer_stride % 16 || a->rec_cap <= 0 || !a->n_chunks)
      return TQ_ERR_INVALID_ARG;
    // the records a stream may hold: rec_cap, or the block table's row length
    if (a->block_table && (!aligned(a->block_table, 4) || a->table_stride <= 0)) return TQ_ERR_INVALID_ARG;
    if (a->max_chunks > (a->block_table ? a->table_stride : a->rec_cap)) return TQ_ERR_INVALID_ARG;
  } else {
    if (a->v_rec || a->n_chunks || a->block_table) return TQ_ERR_INVALID_ARG;
    if (vcod) {  // the merge uses the value codec's signs only for compressed splits
      tq_status st = resolve_codec(vcod, &pl->vc);
      if (st != TQ_OK) return st;
    }
  }
  pl->has_tail = a->k_tail != nullptr;
  if (pl->has_tail) {
    if (!a->v_tail || !aligned(a->k_tail, 16) || !aligned(a->v_tail, 16) || a->tail_layer_stride % 8 ||
        a->tail_cap <= 0 || a->max_tail > a->tail_cap || !a->tail_len)
      return TQ_ERR_INVALID_ARG;
  } else if (a->v_tail || a->tail_len || a->tail_start) {
    return TQ_ERR_INVALID_ARG;
  }
  // Tensor cores for head dims 64 and 128 unless the caller asks for the
  // CUDA-core kernel; the same at head dim 512 for the compressed splits of
  // codecs without side lists, with CTAs of 16 query heads where the group
  // allows (each dequantised pair then feeds two n-tiles of MMAs).  Codecs
  // with outlier side lists take the tensor-core kernel only for sparse-V:
  // its per-token corrections (shared-memory loads, lookups and atomics
  // beside the MMAs, in CTAs of three 4-warp groups) took 2.60 ms on two
  // layers of the batched cache against 2.19 ms for the CUDA-core kernel,
  // which overlaps the same work with its FMA work.
  const bool outl = pl->has_rec && (pl->kc.has_outl || pl->vc.has_outl);
  pl->mma = (D == 64 || D == 128) && !a->cuda_core_path && (!outl || a->sparse_v_eps > 0.f);
  pl->groups = 1;
  if (pl->mma && pl->has_rec) {
    tq::AttnParams t{};
    t.kb = pl->kc.bits;
    t.vb = pl->vc.bits;
    t.kout = pl->kc.has_outl;
    t.vout = pl->vc.has_outl;
    t.k_main = mma_stage_bytes(pl->kc);
    t.v_main = mma_stage_bytes(pl->vc);
    t.shared_kv = pl->shared ? 1 : 0;
    t.G = pl->G;
    t.n_hg = pl->n_hg;
    pl->groups = tq::attn_mma_groups(t, D);
    if (pl->groups == 0) pl->mma = false;
  }
  pl->mma512 = D == 512 && pl->has_rec && a->cuda_core_path != 1 && !pl->kc.has_outl && !pl->vc.has_outl;
  // tcgen05 for groups of 16-64 heads (multiples of 8, which the dense
  // splits' 8-head CTAs need) or multiples of 64: one CTA keeps 64 heads
  pl->umma512 = pl->mma512 && a->cuda_core_path == 0 && pl->G % 8 == 0 && pl->G >= 16 &&
                (pl->G <= 64 || pl->G % 64 == 0) && tq::attn_umma512_smem() <= max_dyn_smem();
  // sparse-V runs on the tensor-core kernel of head dims 64/128 only
  if (!(a->sparse_v_eps >= 0.f && a->sparse_v_eps < 1.f)) return TQ_ERR_INVALID_ARG;
  if (a->sparse_v_eps > 0.f && pl->has_rec && !pl->mma) return TQ_ERR_UNSUPPORTED;
  if (pl->umma512) {
    pl->mma512 = false;
    pl->GT = std::min(pl->G, 64);
    pl->n_hg = pl->G / pl->GT;
  } else if (pl->mma512 && pl->G % 16 == 0) {
    pl->GT = 16;
    pl->n_hg = pl->G / 16;
  }
  pl->dense512 = (pl->mma512 || pl->umma512) && pl->G % 16 == 0 && tq::attn_dense512_smem_bytes() <= max_dyn_smem();
  const int64_t comp_tiles = pl->has_rec ? a->max_chunks : 0;
  const int TT = 4096 / D;
  const int64_t max_tail = pl->has_tail ? a->max_tail : 0;
  const int64_t tail_tiles = cdiv(max_tail, TT);
  const int64_t units = (int64_t)a->n_layers * a->batch * a->n_kv_heads * pl->n_hg;
  // Splits per (layer, batch, kv head, head group): enough CTAs for several
  // waves on every SM.  Records and dense tokens get their own budgets: a
  // call may mix compressed layers with bf16 layers, whose splits then exit
  // at once on the layers that lack that kind of token.
  int64_t want = a->splits > 0 ? a->splits : std::max<int64_t>(1, cdiv(16LL * num_sms(), units));
  want = std::min<int64_t>(want, 500);  // the merge keeps <= 1024 split weights
  int64_t Sc = 0, St = 0;
  if (comp_tiles > 0) Sc = std::max<int64_t>(1, std::min(want, comp_tiles));
  if (tail_tiles > 0) St = std::max<int64_t>(1, std::min(want, tail_tiles));
  // Tensor-core kernels' CTAs take at least two records each, which amortises
  // their per-CTA set-up (pair tables, query fragments), and dense CTAs at
  // least 256 tokens (four 16-token tiles per warp), which also keeps the
  // merge's split count down (Qwen2-shaped step: 25.4 us of attention with
  // 8 dense splits of 256 tokens against 27.1 us with 16 of 128).
  if (pl->mma && a->splits <= 0) {
    if (comp_tiles >= 2) Sc = std::min<int64_t>(Sc, cdiv(comp_tiles, 2));
    if (St > 0) St = std::max<int64_t>(1, std::min<int64_t>(St, cdiv(max_tail, 256)));
  }
  // at head dim 512 a dense split's partial (512 floats per query head, written
  // and read back by the merge) outweighs a short run of tail tokens: at least
  // 128 tokens per split, as on the head-dim 64/128 tensor-core path
  if ((pl->mma512 || pl->umma512) && a->splits <= 0 && St > 0)
    St = std::max<int64_t>(1, std::min<int64_t>(St, cdiv(max_tail, 128)));
  if (pl->umma512 && a->splits <= 0 && comp_tiles > 0) {
    // one CTA per SM: the split count that minimises waves x records per
    // split (plus about two records' worth of per-CTA set-up and partials)
    const int64_t sms = num_sms();
    int64_t best = 1, best_cost = INT64_MAX;
    for (int64_t sc = 1; sc <= std::min<int64_t>(comp_tiles, 500); ++sc) {
      const int64_t cost = cdiv(units * sc, sms) * (cdiv(comp_tiles, sc) + 2);
      if (cost < best_cost) {
        best_cost = cost;
        best = sc;
      }
    }
    Sc = best;
  }
  int64_t cps = 1, tps = TT;
  if (Sc > 0) {
    cps = cdiv(comp_tiles, Sc);
    Sc = cdiv(comp_tiles, cps);
  }
  if (St > 0) {
    tps = TT * cdiv(tail_tiles, St);
    St = cdiv(max_tail, tps);
  }
  if (Sc + St == 0) St = 1;  // empty context: one empty split, zero output
  pl->Sc = (int)Sc;
  pl->S = (int)(Sc + St);
  pl->cps = (int)cps;
  pl->tps = (int)tps;
  pl->rows = (int64_t)a->n_layers * a->batch * a->n_q_heads;
  pl->ws_acc_bytes = (size_t)(((pl->rows * pl->S * D * 4) + 255) / 256 * 256);
  pl->ws_status_off = (pl->ws_acc_bytes + (size_t)pl->rows * pl->S * 2 * 4 + 15) / 16 * 16;
  pl->ws_bytes = pl->ws_status_off + 16;  // + the launch status word
  return TQ_OK;
}

// The launch sequence a plan takes: one kernel over every split at head dims
// 64/128 on the tensor cores; a head-dim-512 tensor-core kernel over the
// compressed splits plus the general kernel over the dense ones; the
// warp-local CUDA-core kernel at head dims 64/128 when there are records; the
// general CUDA-core kernel otherwise.  The merge follows each.
enum class Route { kMma, kD512, kWarp, kGeneral };

Route route_of(const Plan& pl) {
  if (pl.mma) return Route::kMma;
  if ((pl.mma512 || pl.umma512) && pl.Sc > 0) return Route::kD512;
  if ((pl.D == 64 || pl.D == 128) && pl.Sc > 0) return Route::kWarp;
  return Route::kGeneral;
}

}  // namespace

namespace tq {

void attn_smem_layout(AttnParams& p, int D, int GT) {
  const int GTP = GT == 6 ? 8 : GT;
  const int QS = 32 * GTP + (GTP < 4 ? GTP : 4);
  auto al = [](int x, int a) { return (x + a - 1) / a * a; };
  int off = 0;
  p.sm_q = off;
  off = al(off + (D / 32) * QS * 4, 16);
  p.sm_lut = off;
  off += 32 * 4;
  p.sm_red = off;
  off += 2 * 4 * GTP * 4;
  p.sm_logit = off;
  off = al(off + TQ_CHUNK * GTP * 4, 16);
  p.sm_corr = off;
  off = al(off + (p.vout ? D * GTP * 4 : 0), 16);
  const bool anyout = p.kout || p.vout;
  p.sm_pre = off;
  off = al(off + (anyout ? 2 * 2 * 129 * 4 : 0), 16);
  const int vcap = p.shared_kv ? p.kcap : p.vcap;
  p.sm_slot = off;
  off = al(off + (p.vout ? 2 * vcap : 0), 16);
  p.sm_ent_stage = (p.kout ? p.kcap * 4 : 0) + (p.vout && !p.shared_kv ? p.vcap * 4 : 0);
  p.sm_ent = off;
  off = al(off + 2 * p.sm_ent_stage, 128);
  int stage = p.krec ? p.k_main + (p.shared_kv ? 0 : p.v_main) : 0;
  if (p.ktail) stage = std::max(stage, 2 * (4096 / D) * D * 2);
  const int part = (128 / (D / 4)) * D * GTP * 4;  // token-lane partials at the end
  stage = std::max(stage, (part + 2) / 3);
  p.sm_stage = al(stage, 128);
  p.sm_main = off;
  off += 3 * p.sm_stage;
  p.sm_total = off;
}

void attn_rec_smem_layout(AttnParams& p, int D, int GT) {
  const int GTP = GT == 6 ? 8 : GT;
  const int QS = 32 * GTP + (GTP < 4 ? GTP : 4);
  auto al = [](int x, int a) { return (x + a - 1) / a * a; };
  int off = 0;
  p.sm_q = off;
  off = al(off + (D / 32) * QS * 4, 16);
  p.sm_lut = off;
  off += 32 * 4;
  p.sm_red = off;
  off += 2 * 4 * GTP * 4;
  p.sm_logit = off;
  off = al(off + 4 * 32 * GTP * 4, 16);
  p.sm_corr = off;
  off = al(off + (p.vout ? 4 * D * GTP * 4 : 0), 128);
  p.sm_pre = p.sm_slot = p.sm_ent = off;  // unused by this kernel
  p.sm_ent_stage = 0;
  int stage = p.krec ? p.k_main + (p.shared_kv ? 0 : p.v_main) : 0;
  stage = std::max(stage, (4 * D * GTP * 4 + 1) / 2);  // the warps' partials at the end
  p.sm_stage = al(stage, 128);
  p.sm_main = off;
  off += 2 * p.sm_stage;
  p.sm_total = off;
}

void attn_mma_smem_layout(AttnParams& p, int D) {
  auto al = [](int x, int a) { return (x + a - 1) / a * a; };
  const int NG = std::max(1, p.groups), NW = 4 * NG;  // 4-warp groups, warps
  int off = 0;
  p.sm_kpair = off;  // the kernel addresses both pair tables at these fixed offsets
  off += (1 << (2 * p.kb)) * 128;
  p.sm_vpair = off;
  off += (p.vb == 3 ? 120 : (1 << (2 * p.vb))) * 128;
  p.sm_q = off;      // q~ [8 heads][4 lane runs padded], see the kernel
  off += 8 * 4 * (std::max(D / 4, 32) + 1) * 4;
  p.sm_slot = off;   // centroid halves
  off += 32 * 8;
  p.sm_red = off;    // the warps' (m, l) at the end
  off += NW * 2 * 8 * 4;
  p.sm_logit = off;  // query fragments [d/16][32 lanes][16 B]
  off = al(off + (D / 16) * 32 * 16, 128);
  // side lists: f32 centroids (K, V), q~ by coordinate [D][8 heads] and the
  // warps' value corrections [warps][heads rounded up to even][D + D/8 + pad]
  p.sm_lut = off;
  off += (p.kout || p.vout) ? 32 * 4 : 0;
  p.sm_qi = off;
  off += p.kout ? D * 8 * 4 : 0;
  p.sm_corr = off;
  const int GT = p.n_hg > 0 ? p.G / p.n_hg : 8;
  off = al(off + (p.vout ? NW * ((GT + 1) & ~1) * (D == 128 ? 168 : 72) * 4 : 0), 128);
  p.sm_pre = p.sm_ent = off;  // unused by this kernel
  p.sm_ent_stage = 0;
  int stage = p.k_main + (p.shared_kv ? 0 : p.v_main) + 16;  // + the word a run load may read past a row
  stage = std::max(stage, (4 * 8 * (D + D / 8) * 4 + 1) / 2);  // the warps' partials at the end
  p.sm_stage = al(stage, 128);
  p.sm_main = off;
  off += 2 * NG * p.sm_stage;  // a two-deep ring per group
  p.sm_total = off;
}

// 4-warp groups per CTA of the tensor-core kernel: one for codecs without
// side lists (up to four such CTAs per SM); with side lists as many as one
// CTA per SM holds (at most 3), so that the SM keeps 12 warps and one copy
// of the pair tables (4-bit keys: 32 KB) rather than two 4-warp CTAs with a
// copy each.  0 if not even one group fits.
int attn_mma_groups(const AttnParams& base, int D) {
  AttnParams t = base;
  for (int ng = (base.kout || base.vout) ? kMmaOutlGroups : 1; ng >= 1; --ng) {
    t.groups = ng;
    attn_mma_smem_layout(t, D);
    if (t.sm_total <= max_dyn_smem()) return ng;
  }
  return 0;
}

void attn_mma512_smem_layout(AttnParams& p) {
  const int NT = (p.G / p.n_hg > 8) ? 2 : 1;  // n-tiles of 8 query heads per CTA
  auto al = [](int x, int a) { return (x + a - 1) / a * a; };
  int off = 0;
  p.sm_kpair = off;  // fixed offsets, as in the d 64/128 kernel
  off += (1 << (2 * p.kb)) * 128;
  p.sm_vpair = off;
  off += (p.vb == 3 ? 120 : (1 << (2 * p.vb))) * 128;
  p.sm_logit = off;  // query fragments [32 k-steps][NT][32 lanes][16 B]
  off += 32 * NT * 32 * 16;
  p.sm_slot = off;   // centroid halves
  off += 32 * 8;
  p.sm_red = off;    // logits [128][8 NT]
  off += 128 * 8 * NT * 4;
  p.sm_corr = off;   // softmax state m[16] | scale[16] | l[16] | kx
  off = al(off + 64 * 4, 128);
  p.sm_q = p.sm_lut = p.sm_pre = p.sm_ent = off;  // unused by this kernel
  p.sm_ent_stage = 0;
  int stage = p.k_main + (p.shared_kv ? 0 : p.v_main) + 16;  // + the word a run load may read past a row
  stage = std::max(stage, 8 * NT * 516 * 4);                  // q~ is built in the second buffer
  p.sm_stage = al(stage, 128);
  p.sm_main = off;
  off += 2 * p.sm_stage;
  p.sm_total = off;
}

}  // namespace tq

extern "C" {

const char* tq_status_string(int status) {
  switch (status) {
    case TQ_OK: return "TQ_OK";
    case TQ_ERR_INVALID_ARG: return "TQ_ERR_INVALID_ARG: null, misaligned or out-of-range argument";
    case TQ_ERR_UNSUPPORTED: return "TQ_ERR_UNSUPPORTED: head_dim/bits/table/geometry not supported";
    case TQ_ERR_WORKSPACE: return "TQ_ERR_WORKSPACE: workspace or scratch too small";
    case TQ_ERR_CUDA: return "TQ_ERR_CUDA: a CUDA call or kernel launch failed";
    default: return "unknown tq_status";
  }
}

int tq_version(void) { return kVersion; }

size_t tq_codebook_scratch_bytes(void) { return sizeof(CodebookOut); }

tq_status tq_make_codebook(int bits, int head_dim, uint64_t sign_seed, float outlier_T, int outlier_cap,
                           void* d_scratch, size_t scratch_bytes, tq_codec* out, double* mse_out,
                           void* stream) {
  if (bits < 1 || bits > 4 || !dim_ok(head_dim)) return TQ_ERR_UNSUPPORTED;
  if (!out || !d_scratch || !aligned(d_scratch, 16)) return TQ_ERR_INVALID_ARG;
  if (!(outlier_T >= 0.f) || outlier_cap < 0 || outlier_cap % 4 != 0 || outlier_cap > 65536)
    return TQ_ERR_INVALID_ARG;
  if (scratch_bytes < sizeof(CodebookOut)) return TQ_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  if (launch_codebook(bits, head_dim, sign_seed, d_scratch, s) != cudaSuccess) return TQ_ERR_CUDA;
  CodebookOut h;
  if (cudaMemcpyAsync(&h, d_scratch, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return TQ_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return TQ_ERR_CUDA;
  std::memset(out, 0, sizeof(*out));
  out->head_dim = head_dim;
  out->bits = bits;
  out->sign_seed = sign_seed;
  out->outlier_T = outlier_T;
  out->outlier_cap = outlier_cap ? outlier_cap : default_cap(head_dim);
  const int K = 1 << bits;
  for (int k = 0; k < K; ++k) out->centroids[k] = h.c[k];
  for (int k = 0; k + 1 < K; ++k) out->boundaries[k] = h.t[k];
  for (int w = 0; w < head_dim / 32; ++w) out->sign_bits[w] = h.signs[w];
  if (mse_out) *mse_out = h.mse;
  return TQ_OK;
}

tq_status tq_codec_set_centroids(tq_codec* codec, const float* centroids, int n_centroids) {
  if (!codec || !centroids) return TQ_ERR_INVALID_ARG;
  const int b = codec->bits;
  if (b < 1 || b > 4) return TQ_ERR_UNSUPPORTED;
  const int K = 1 << b;
  if (n_centroids != K) return TQ_ERR_INVALID_ARG;
  float c[16], t[15];
  for (int k = 0; k < K; ++k) {
    if (!std::isfinite(centroids[k])) return TQ_ERR_INVALID_ARG;
    if (k && !(centroids[k - 1] < centroids[k])) return TQ_ERR_INVALID_ARG;
    c[k] = centroids[k];
  }
  for (int k = 0; k < K; ++k)
    if (c[k] != -c[K - 1 - k]) return TQ_ERR_UNSUPPORTED;
  for (int k = 0; k + 1 < K; ++k) t[k] = (float)(0.5 * ((double)c[k] + (double)c[k + 1]));
  for (int k = 0; k + 1 < K; ++k)  // the midpoint must fall strictly between its centroids
    if (!(c[k] < t[k] && t[k] < c[k + 1])) return TQ_ERR_UNSUPPORTED;
  const tq_status st = table_supported(c, t, b);
  if (st != TQ_OK) return st;
  for (int k = 0; k < 16; ++k) codec->centroids[k] = k < K ? c[k] : 0.f;
  for (int k = 0; k < 15; ++k) codec->boundaries[k] = k + 1 < K ? t[k] : 0.f;
  return TQ_OK;
}

size_t tq_record_bytes(const tq_codec* codec) {
  CodecDev c;
  if (resolve_codec(codec, &c) != TQ_OK) return 0;
  return (size_t)c.rec_bytes;
}

tq_status tq_encode(const tq_codec* codec, const void* src, int64_t n_groups, int64_t n_vec,
                    int64_t src_vec_stride, int64_t src_group_stride, void* dst, int64_t dst_group_stride,
                    int64_t first_vec, void* stream) {
  EncodeParams p;
  tq_status st = resolve_codec(codec, &p.c);
  if (st != TQ_OK) return st;
  if (n_groups < 0 || n_vec < 0 || first_vec < 0) return TQ_ERR_INVALID_ARG;
  if (n_groups == 0 || n_vec == 0) return TQ_OK;
  if (!src || !dst || !aligned(src, 16) || !aligned(dst, 16)) return TQ_ERR_INVALID_ARG;
  if (src_vec_stride < p.c.d || src_vec_stride % 8 || src_group_stride < 0 || src_group_stride % 8 ||
      dst_group_stride < 0 || dst_group_stride % 16)
    return TQ_ERR_INVALID_ARG;
  if (p.c.has_outl && first_vec % TQ_CHUNK) return TQ_ERR_INVALID_ARG;
  p.src = (const uint16_t*)src;
  p.src_vs = src_vec_stride;
  p.src_gs = src_group_stride;
  p.dst = (uint8_t*)dst;
  p.dst_gs = dst_group_stride;
  p.n_groups = n_groups;
  p.n_vec = n_vec;
  p.first_vec = first_vec;
  p.first_chunk = first_vec / TQ_CHUNK;
  p.chunks_per_group = (first_vec + n_vec - 1) / TQ_CHUNK - p.first_chunk + 1;
  // task indices: at most 32 per record (tiles of 16, 8 or 4 vectors), plus a grid's lookahead
  p.small_tasks = p.chunks_per_group < (1ll << 31) && n_groups * p.chunks_per_group * 32 + (1ll << 24) < (1ll << 32);
  p.cpg = make_fast_div(p.small_tasks ? (uint32_t)p.chunks_per_group : 1u);
  // the launcher caps the grid at the number of tasks of the kernel it picks
  return launch_encode(p, 8 * num_sms(), (cudaStream_t)stream) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

tq_status tq_decode(const tq_codec* codec, const void* src, int64_t n_groups, int64_t n_vec,
                    int64_t src_group_stride, int64_t first_vec, float* dst, int64_t dst_vec_stride,
                    int64_t dst_group_stride, void* stream) {
  DecodeParams p;
  tq_status st = resolve_codec(codec, &p.c);
  if (st != TQ_OK) return st;
  if (n_groups < 0 || n_vec < 0 || first_vec < 0) return TQ_ERR_INVALID_ARG;
  if (n_groups == 0 || n_vec == 0) return TQ_OK;
  if (!src || !dst || !aligned(src, 16) || !aligned(dst, 16)) return TQ_ERR_INVALID_ARG;
  if (src_group_stride < 0 || src_group_stride % 16 || dst_vec_stride < p.c.d || dst_vec_stride % 4 ||
      dst_group_stride < 0 || dst_group_stride % 4)
    return TQ_ERR_INVALID_ARG;
  p.src = (const uint8_t*)src;
  p.src_gs = src_group_stride;
  p.dst = dst;
  p.dst_vs = dst_vec_stride;
  p.dst_gs = dst_group_stride;
  p.n_groups = n_groups;
  p.n_vec = n_vec;
  p.first_vec = first_vec;
  p.first_chunk = first_vec / TQ_CHUNK;
  p.chunks_per_group = (first_vec + n_vec - 1) / TQ_CHUNK - p.first_chunk + 1;
  const int64_t tasks = n_groups * p.chunks_per_group;
  // fewer records than SMs: split each over up to 4 CTAs (the codec round trip's
  // 32 records then take 128 CTAs instead of 32); head dim 512 keeps one
  p.log2_parts = 0;
  while (p.c.d < 512 && p.log2_parts < 2 && (tasks << p.log2_parts) < num_sms()) ++p.log2_parts;
  const int grid = (int)std::min<int64_t>(tasks << p.log2_parts, 8LL * num_sms());
  return launch_decode(p, grid, (cudaStream_t)stream) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

tq_status tq_evict(const tq_codec* k_codec, const tq_codec* v_codec, const tq_evict_args* a, void* stream) {
  if (!a) return TQ_ERR_INVALID_ARG;
  CodecDev kc, vc;
  tq_status st = resolve_codec(k_codec, &kc);
  if (st != TQ_OK) return st;
  const bool shared = a->v_rec == a->k_rec;
  if (shared) {
    if (v_codec && std::memcmp(k_codec, v_codec, sizeof(tq_codec)) != 0) return TQ_ERR_INVALID_ARG;
    vc = kc;
  } else {
    st = resolve_codec(v_codec, &vc);
    if (st != TQ_OK) return st;
  }
  const int D = kc.d;
  if (vc.d != D) return TQ_ERR_INVALID_ARG;
  if (a->n_layers <= 0 || a->n_layers > 65535 || a->batch <= 0 || a->n_kv_heads <= 0 ||
      (int64_t)a->batch * a->n_kv_heads > 65535 || a->max_evict <= 0 || a->max_evict > 65535)
    return TQ_ERR_INVALID_ARG;
  if (!a->k_rec || !a->v_rec || !a->k_tail || !a->v_tail || !a->n_chunks || !a->tail_start || !a->tail_len)
    return TQ_ERR_INVALID_ARG;
  if (!aligned(a->k_rec, 16) || !aligned(a->v_rec, 16) || !aligned(a->k_tail, 16) || !aligned(a->v_tail, 16) ||
      a->k_rec_layer_stride % 16 || a->v_rec_layer_stride % 16 || a->tail_layer_stride % 8)
    return TQ_ERR_INVALID_ARG;
  if (a->rec_cap <= 0 || a->tail_cap <= 0 || a->window < 0 || a->margin < 0 || a->t_q < 1)
    return TQ_ERR_INVALID_ARG;
  if (a->block_table && (!aligned(a->block_table, 4) || a->table_stride <= 0)) return TQ_ERR_INVALID_ARG;
  // the retention floor; a ring that cannot hold floor + one chunk never evicts
  const int64_t floor64 = (int64_t)a->window + std::max<int64_t>((int64_t)a->t_q - 1, a->margin);
  if ((int64_t)a->tail_cap < floor64 + TQ_CHUNK) return TQ_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const int floor_ = (int)floor64;
  EvictParams p;
  p.rec_cap = a->rec_cap;
  p.table = a->block_table;
  p.table_stride = a->block_table ? a->table_stride : 0;
  p.rec_limit = a->block_table ? a->table_stride : a->rec_cap;
  p.tail_ls = a->tail_layer_stride;
  p.tail_cap = a->tail_cap;
  p.n_chunks = a->n_chunks;
  p.tail_start = a->tail_start;
  p.tail_len = a->tail_len;
  p.L = a->n_layers;
  p.B = a->batch;
  p.Hkv = a->n_kv_heads;
  p.floor_ = floor_;
  p.max_evict = a->max_evict;
  p.c = kc;
  p.rec = (uint8_t*)a->k_rec;
  p.rec_ls = a->k_rec_layer_stride;
  p.tail = (const uint16_t*)a->k_tail;
  if (launch_evict(p, s) != cudaSuccess) return TQ_ERR_CUDA;
  if (!shared) {
    p.c = vc;
    p.rec = (uint8_t*)a->v_rec;
    p.rec_ls = a->v_rec_layer_stride;
    p.tail = (const uint16_t*)a->v_tail;
    if (launch_evict(p, s) != cudaSuccess) return TQ_ERR_CUDA;
  }
  EvictCommitParams cp;
  cp.n_chunks = a->n_chunks;
  cp.tail_start = a->tail_start;
  cp.tail_len = a->tail_len;
  cp.LB = a->n_layers * a->batch;
  cp.floor_ = floor_;
  cp.max_evict = a->max_evict;
  cp.tail_cap = a->tail_cap;
  cp.rec_limit = p.rec_limit;
  return launch_evict_commit(cp, s) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

tq_status tq_rollback(const tq_codec* k_codec, const tq_codec* v_codec, const tq_evict_args* a,
                      const int32_t* new_len, void* stream) {
  if (!a || !new_len || !aligned(new_len, 4)) return TQ_ERR_INVALID_ARG;
  CodecDev kc, vc;
  tq_status st = resolve_codec(k_codec, &kc);
  if (st != TQ_OK) return st;
  const bool shared = a->v_rec == a->k_rec;
  if (shared) {
    if (v_codec && std::memcmp(k_codec, v_codec, sizeof(tq_codec)) != 0) return TQ_ERR_INVALID_ARG;
    if (a->v_tail != a->k_tail) return TQ_ERR_INVALID_ARG;  // shared records come from one ring
    vc = kc;
  } else {
    st = resolve_codec(v_codec, &vc);
    if (st != TQ_OK) return st;
  }
  if (vc.d != kc.d) return TQ_ERR_INVALID_ARG;
  if (a->n_layers <= 0 || a->n_layers > 65535 || a->batch <= 0 || a->n_kv_heads <= 0 ||
      (int64_t)a->batch * a->n_kv_heads > 2147483647ll)
    return TQ_ERR_INVALID_ARG;
  if (!a->k_rec || !a->v_rec || !a->k_tail || !a->v_tail || !a->n_chunks || !a->tail_start || !a->tail_len)
    return TQ_ERR_INVALID_ARG;
  if (!aligned(a->k_rec, 16) || !aligned(a->v_rec, 16) || !aligned(a->k_tail, 16) || !aligned(a->v_tail, 16) ||
      a->k_rec_layer_stride % 16 || a->v_rec_layer_stride % 16 || a->tail_layer_stride % 8)
    return TQ_ERR_INVALID_ARG;
  // the decoded tokens of one record (at most 127) must fit the ring
  if (a->rec_cap <= 0 || a->tail_cap < TQ_CHUNK) return TQ_ERR_INVALID_ARG;
  if (a->block_table && (!aligned(a->block_table, 4) || a->table_stride <= 0)) return TQ_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  RollbackParams p;
  std::memset(&p, 0, sizeof(p));
  p.rec_cap = a->rec_cap;
  p.table = a->block_table;
  p.table_stride = a->block_table ? a->table_stride : 0;
  p.rec_limit = a->block_table ? a->table_stride : a->rec_cap;
  p.tail_ls = a->tail_layer_stride;
  p.tail_cap = a->tail_cap;
  p.n_chunks = a->n_chunks;
  p.tail_start = a->tail_start;
  p.tail_len = a->tail_len;
  p.new_len = new_len;
  p.L = a->n_layers;
  p.B = a->batch;
  p.Hkv = a->n_kv_heads;
  p.c = kc;
  p.rec = (const uint8_t*)a->k_rec;
  p.rec_ls = a->k_rec_layer_stride;
  p.tail = (uint16_t*)a->k_tail;
  if (launch_rollback(p, s) != cudaSuccess) return TQ_ERR_CUDA;
  if (!shared) {
    p.c = vc;
    p.rec = (const uint8_t*)a->v_rec;
    p.rec_ls = a->v_rec_layer_stride;
    p.tail = (uint16_t*)a->v_tail;
    if (launch_rollback(p, s) != cudaSuccess) return TQ_ERR_CUDA;
  }
  return launch_rollback_commit(p, s) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

size_t tq_decode_attn_workspace_size(const tq_attn_args* args, const tq_codec* k_codec,
                                     const tq_codec* v_codec) {
  Plan pl;
  if (make_plan(args, k_codec, v_codec, &pl) != TQ_OK) return 0;
  return pl.ws_bytes;
}

tq_status tq_decode_attn_plan(const tq_attn_args* args, const tq_codec* k_codec, const tq_codec* v_codec,
                              tq_attn_plan* plan) {
  if (!plan) return TQ_ERR_INVALID_ARG;
  Plan pl;
  const tq_status st = make_plan(args, k_codec, v_codec, &pl);
  if (st != TQ_OK) return st;
  std::memset(plan, 0, sizeof(*plan));
  const int St = pl.S - pl.Sc;
  int ck = TQ_ATTN_KERNEL_CUDA_CORE, dk = TQ_ATTN_KERNEL_CUDA_CORE, dense_gt = pl.GT, launches = 2, warps = 4;
  switch (route_of(pl)) {
    case Route::kMma:
      ck = dk = TQ_ATTN_KERNEL_MMA;
      if (pl.has_rec && pl.groups > 1 && St > 0) ++launches;
      warps = 4 * (pl.has_rec ? pl.groups : 1);
      break;
    case Route::kD512:
      ck = pl.umma512 ? TQ_ATTN_KERNEL_TCGEN05 : TQ_ATTN_KERNEL_MMA512;
      if (pl.dense512) dk = TQ_ATTN_KERNEL_MMA512;
      dense_gt = pl.dense512 ? 16 : std::min(pl.GT, 8);
      if (St > 0) ++launches;
      break;
    case Route::kWarp:
      ck = dk = TQ_ATTN_KERNEL_CUDA_CORE_WARP;
      break;
    case Route::kGeneral:
      break;
  }
  plan->compressed_kernel = pl.Sc > 0 ? ck : TQ_ATTN_KERNEL_NONE;
  plan->dense_kernel = St > 0 ? dk : TQ_ATTN_KERNEL_NONE;
  plan->compressed_splits = pl.Sc;
  plan->dense_splits = St;
  plan->records_per_split = pl.Sc > 0 ? pl.cps : 0;
  plan->dense_tokens_per_split = St > 0 ? pl.tps : 0;
  plan->heads_per_cta = pl.GT;
  plan->dense_heads_per_cta = dense_gt;
  plan->launches = launches;
  plan->workspace_bytes = pl.ws_bytes;
  plan->warps_per_cta = warps;
  return TQ_OK;
}

tq_status tq_decode_attn(const tq_attn_args* a, const tq_codec* k_codec, const tq_codec* v_codec,
                         void* workspace, size_t workspace_bytes, void* stream) {
  Plan pl;
  tq_status st = make_plan(a, k_codec, v_codec, &pl);
  if (st != TQ_OK) return st;
  if (!workspace || !aligned(workspace, 256)) return TQ_ERR_INVALID_ARG;
  if (workspace_bytes < pl.ws_bytes) return TQ_ERR_WORKSPACE;
  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  p.L = a->n_layers;
  p.B = a->batch;
  p.Hq = a->n_q_heads;
  p.Hkv = a->n_kv_heads;
  p.G = pl.G;
  p.n_hg = pl.n_hg;
  p.sscale = (float)((double)a->scale * 1.4426950408889634074);
  p.scap = a->softcap > 0.f ? (float)((double)a->softcap * 1.4426950408889634074) : 0.f;
  p.sv_log2eps = a->sparse_v_eps > 0.f ? (float)std::log2((double)a->sparse_v_eps) : 0.f;
  p.iscap = a->softcap > 0.f ? (float)(1.0 / ((double)a->softcap * 1.4426950408889634074)) : 0.f;
  p.q = (const uint16_t*)a->q;
  p.q_ls = a->q_layer_stride;
  p.q_bs = a->q_batch_stride;
  if (pl.has_rec) {
    p.krec = (const uint8_t*)a->k_rec;
    p.vrec = (const uint8_t*)a->v_rec;
    p.krec_ls = a->k_rec_layer_stride;
    p.vrec_ls = a->v_rec_layer_stride;
    p.rec_cap = a->rec_cap;
    p.table = a->block_table;
    p.table_stride = a->block_table ? a->table_stride : 0;
    p.rec_limit = a->block_table ? a->table_stride : a->rec_cap;
    p.krec_bytes = pl.kc.rec_bytes;
    p.vrec_bytes = pl.vc.rec_bytes;
    p.kb = pl.kc.bits;
    p.vb = pl.vc.bits;
    p.kout = pl.kc.has_outl;
    p.vout = pl.vc.has_outl;
    p.kcap = pl.kc.cap;
    p.vcap = pl.vc.cap;
    p.shared_kv = pl.shared ? 1 : 0;
    p.k_off_norm = pl.kc.off_norm;
    p.v_off_norm = pl.vc.off_norm;
    p.k_off_count = pl.kc.off_count;
    p.v_off_count = pl.vc.off_count;
    p.k_off_ent = pl.kc.off_entries;
    p.v_off_ent = pl.vc.off_entries;
    p.k_main = pl.kc.off_count + (pl.kc.has_outl ? TQ_CHUNK : 0);
    p.v_main = pl.vc.off_count + (pl.vc.has_outl ? TQ_CHUNK : 0);
    std::memcpy(p.kc, pl.kc.centroids, sizeof(p.kc));
    std::memcpy(p.vc, pl.vc.centroids, sizeof(p.vc));
    std::memcpy(p.ksign, pl.kc.signs, sizeof(p.ksign));
    p.n_chunks = a->n_chunks;
  }
  if (pl.has_tail) {
    p.ktail = (const uint16_t*)a->k_tail;
    p.vtail = (const uint16_t*)a->v_tail;
    p.tail_ls = a->tail_layer_stride;
    p.tail_cap = a->tail_cap;
    p.tail_start = a->tail_start;
    p.tail_len = a->tail_len;
  }
  p.S = pl.S;
  p.Sc = pl.Sc;
  p.cps = pl.cps;
  p.tps = pl.tps;
  p.ws_acc = (float*)workspace;
  p.ws_ml = (float*)((char*)workspace + pl.ws_acc_bytes);
  cudaStream_t s = (cudaStream_t)stream;
  const int units_y = a->batch * a->n_kv_heads * pl.n_hg;
  const Route route = route_of(pl);
  const int* status = nullptr;
  if (route == Route::kMma) {
    // tensor cores: compressed and dense splits in one launch of 4-warp
    // CTAs; with CTAs of several groups the dense splits (4-warp work) take
    // a second launch of single-group CTAs
    AttnParams pm = p;
    if (!pl.has_rec) pm.kb = pm.vb = 1;  // dense only: any instantiation (its tables go unused)
    if (pl.has_rec) {
      pm.k_main = mma_stage_bytes(pl.kc);
      pm.v_main = mma_stage_bytes(pl.vc);
    }
    pm.groups = pl.has_rec ? pl.groups : 1;
    attn_mma_smem_layout(pm, pl.D);
    if (pm.sm_total > max_dyn_smem()) return TQ_ERR_UNSUPPORTED;
    const bool wide = pm.groups > 1;
    const int gx = wide ? pl.Sc : pl.S;
    if (gx > 0 && launch_attn_mma(pm, pl.D, dim3(gx, units_y, a->n_layers), s) != cudaSuccess) return TQ_ERR_CUDA;
    if (wide && pl.S > pl.Sc) {
      AttnParams pd = p;
      pd.kb = pd.vb = 1;
      pd.kout = pd.vout = 0;
      pd.k_main = pd.v_main = 0;
      pd.groups = 1;
      pd.split_base = pl.Sc;
      attn_mma_smem_layout(pd, pl.D);
      if (pd.sm_total > max_dyn_smem()) return TQ_ERR_UNSUPPORTED;
      if (launch_attn_mma(pd, pl.D, dim3(pl.S - pl.Sc, units_y, a->n_layers), s) != cudaSuccess) return TQ_ERR_CUDA;
    }
  } else if (route == Route::kD512) {
    // compressed splits on a d-512 tensor-core kernel, dense splits (if any)
    // in a second launch: on the tensor cores for groups of a multiple of 16
    // heads, else on the general kernel (groups of at most 8 heads)
    AttnParams pm = p;
    if (pl.umma512) {
      pm.status = (int*)((char*)workspace + pl.ws_status_off);
      if (cudaMemsetAsync(pm.status, 0, sizeof(int), s) != cudaSuccess) return TQ_ERR_CUDA;
      if (launch_attn_umma512(pm, dim3(pl.Sc, units_y, a->n_layers), s) != cudaSuccess) return TQ_ERR_CUDA;
      status = pm.status;
    } else {
      attn_mma512_smem_layout(pm);
      if (pm.sm_total > max_dyn_smem()) return TQ_ERR_UNSUPPORTED;
      if (launch_attn_mma512(pm, dim3(pl.Sc, units_y, a->n_layers), s) != cudaSuccess) return TQ_ERR_CUDA;
    }
    if (pl.S > pl.Sc && pl.dense512) {
      AttnParams pd = p;
      pd.split_base = pl.Sc;
      pd.n_hg = pl.G / 16;
      const int uy = a->batch * a->n_kv_heads * pd.n_hg;
      if (launch_attn_dense512(pd, dim3(pl.S - pl.Sc, uy, a->n_layers), s) != cudaSuccess) return TQ_ERR_CUDA;
    } else if (pl.S > pl.Sc) {
      AttnParams pd = p;
      pd.split_base = pl.Sc;
      int gt = pl.GT;
      if (gt > 8) {
        gt = 8;
        pd.n_hg = pl.G / 8;
      }
      attn_smem_layout(pd, pl.D, gt);
      if (pd.sm_total > max_dyn_smem()) return TQ_ERR_UNSUPPORTED;
      const int uy = a->batch * a->n_kv_heads * pd.n_hg;
      if (launch_attn(pd, pl.D, gt, dim3(pl.S - pl.Sc, uy, a->n_layers), s) != cudaSuccess) return TQ_ERR_CUDA;
    }
  } else if (route == Route::kWarp) {
    // compressed splits on the warp-local path, dense splits on the general
    // dense path, one launch
    attn_rec_smem_layout(p, pl.D, pl.GT);
    if (p.sm_total > max_dyn_smem()) return TQ_ERR_UNSUPPORTED;
    if (launch_attn_rec(p, pl.D, pl.GT, dim3(pl.S, units_y, a->n_layers), s) != cudaSuccess) return TQ_ERR_CUDA;
  } else {
    attn_smem_layout(p, pl.D, pl.GT);
    if (p.sm_total > max_dyn_smem()) return TQ_ERR_UNSUPPORTED;
    if (launch_attn(p, pl.D, pl.GT, dim3(pl.S, units_y, a->n_layers), s) != cudaSuccess) return TQ_ERR_CUDA;
  }
  MergeParams m;
  m.ws_acc = p.ws_acc;
  m.ws_ml = p.ws_ml;
  m.out = a->out;
  m.rows = (int)pl.rows;
  m.S = pl.S;
  m.Sc = pl.Sc;
  m.status = status;
  m.inv_sqrt_d = (float)(1.0 / std::sqrt((double)pl.D));
  std::memcpy(m.vsign, pl.vc.signs, sizeof(m.vsign));
  return launch_merge(m, pl.D, s) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // extern "C"
