/*
 * tq_oracle.c -- plain, slow, obviously-correct CPU oracle for the rotated
 * Lloyd-Max KV-cache codec and the decode attention that reads it.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no source, header, table or
 * helper with the CUDA path.
 *
 * Every floating-point step runs in fp64 unless the method fixes a narrower
 * type (the stored norm is f32, the centroid table is f32, outlier values are
 * bf16).  Loops are plain scalar loops in the order the method states them.
 *
 * Sources (web pages; cited by title and section):
 *   [P1] "v1.3 PPL on vLLM: production cell + per-channel attribution"
 *        (LLM-KV--Cache-compress PR #15): the M4 Phase A/A.2/B and M5
 *        commits -- rotate = H.D.x and its inverse, per-row scale, Lloyd-Max
 *        argmin, (u16 idx, value) outlier overrides replaced before the
 *        inverse WHT.
 *   [P3] larql PR #196, turbo-quant fix note -- one N(0,1) Lloyd-Max table per
 *        bit width scaled by 1/sqrt(d); append-only encode.
 *   [P4] "feat(v4): TurboQuant KV storage for DeepSeek-V4" (arc PR #98),
 *        "What landed" and its bytes-per-token table (256 packed + one f32
 *        norm = 260 B at head_dim 512), "Eviction is chunked, on purpose"
 *        (EVICT_CHUNK = 128, tail bound window + max(t_q-1, margin) + chunk),
 *        and its softcapping fix (the cap applied after the scale multiply,
 *        before the logits are stored and their maximum taken).
 *
 * Readings where the pages are silent (each is a stated choice):
 *   - sign diagonal: SplitMix64 (Steele, Lea & Flood, OOPSLA 2014), top bit
 *     of each output -> -1;
 *   - Hadamard: Sylvester natural order, orthonormal (1/sqrt(d));
 *   - tie rule: code = number of boundaries strictly below y;
 *   - boundaries: fp32 midpoints of the fp32 scaled centroids;
 *   - outlier test |y_j| > T / sqrt(d)  (rms(y) = 1/sqrt(d) since ||y|| = 1);
 *   - packing: per token an LSB-first little-endian bitstream, code j in bits
 *     [j*b, (j+1)*b); 128-token chunk records (layout in tq_record_layout()).
 *
 * Parity pinned by tests against closed forms (b = 1), Max's 1960 table
 * (b = 2..4), scipy quadrature, scipy's Hadamard matrix, the published
 * SplitMix64 vectors, brute-force nearest-centroid search, and attention
 * special cases; see tests/test_oracle_*.py.  The sign generator's choice and
 * the packing bit order are this project's own definitions: pinned only by
 * hand-worked examples, not by the pages.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_CHUNK 128

/* ------------------------------------------------------------------------- */
/* Standard normal density, distribution and tail                            */
/* ------------------------------------------------------------------------- */
static double norm_pdf(double x) {
  if (isinf(x)) return 0.0;
  return exp(-0.5 * x * x) / sqrt(2.0 * M_PI);
}
static double norm_cdf(double x) { return 0.5 * erfc(-x / sqrt(2.0)); }
static double norm_sf(double x) { return 0.5 * erfc(x / sqrt(2.0)); }
/* x * pdf(x), with the limits at +-infinity equal to 0 */
static double x_pdf(double x) { return isinf(x) ? 0.0 : x * norm_pdf(x); }

/* N(0,1) probability of the cell (a, b], a < b; upper tail differences are
 * used on the positive side to avoid cancellation. */
static double cell_mass(double a, double b) {
  if (a >= 0.0) return norm_sf(a) - norm_sf(b);
  return norm_cdf(b) - norm_cdf(a);
}

/*
 * Gaussian Lloyd-Max quantizer with 2^bits levels for N(0,1), by the 1-D Lloyd
 * iteration [P1 "centroids_gaussian(bits)"; P3 turbo-quant note]:
 *   boundaries  t_k = (c_k + c_{k+1}) / 2
 *   centroids   c_k = E[X | t_{k-1} < X <= t_k]
 *                   = (pdf(t_{k-1}) - pdf(t_k)) / (Phi(t_k) - Phi(t_{k-1}))
 * iterated from evenly spaced centroids until no centroid moves by more than
 * 1e-14 (the N(0,1) density is log-concave, so the fixed point is unique).
 * Writes c[2^bits], t[2^bits - 1] and the distortion E[(X - Q(X))^2];
 * returns the number of iterations.
 */
int orc_lloyd_max_gaussian(int bits, double* c, double* t, double* mse) {
  const int K = 1 << bits;
  for (int k = 0; k < K; ++k) c[k] = (k - 0.5 * (K - 1)) * (4.0 / K);
  int it = 0;
  for (it = 1; it <= 100000; ++it) {
    for (int k = 0; k + 1 < K; ++k) t[k] = 0.5 * (c[k] + c[k + 1]);
    double moved = 0.0;
    for (int k = 0; k < K; ++k) {
      double a = (k == 0) ? -INFINITY : t[k - 1];
      double b = (k == K - 1) ? INFINITY : t[k];
      double ck = (norm_pdf(a) - norm_pdf(b)) / cell_mass(a, b);
      if (fabs(ck - c[k]) > moved) moved = fabs(ck - c[k]);
      c[k] = ck;
    }
    if (moved < 1e-14) break;
  }
  for (int k = 0; k + 1 < K; ++k) t[k] = 0.5 * (c[k] + c[k + 1]);
  /* distortion: sum over cells of int_a^b (x - c)^2 pdf(x) dx, using
   *   int x^2 pdf = P - [x pdf],  int x pdf = pdf(a) - pdf(b). */
  double D = 0.0;
  for (int k = 0; k < K; ++k) {
    double a = (k == 0) ? -INFINITY : t[k - 1];
    double b = (k == K - 1) ? INFINITY : t[k];
    double P = cell_mass(a, b);
    double m2 = P - (x_pdf(b) - x_pdf(a));
    double m1 = norm_pdf(a) - norm_pdf(b);
    D += m2 - 2.0 * c[k] * m1 + c[k] * c[k] * P;
  }
  if (mse) *mse = D;
  return it;
}

/*
 * Boundaries of a caller-supplied ascending f32 centroid table (a calibrated
 * table, P1's calibrated Lloyd-Max commit: a 2^b sorted f32 table loaded in
 * place of the Gaussian one): the f32 midpoints of consecutive centroids,
 * computed in fp64 and rounded, as for the Gaussian table below.
 */
void orc_midpoints_f32(int bits, const float* c32, float* t32) {
  const int K = 1 << bits;
  for (int k = 0; k + 1 < K; ++k) t32[k] = (float)(0.5 * ((double)c32[k] + (double)c32[k + 1]));
}

/*
 * The table a codec of head dimension d uses: the unit-variance table scaled
 * by 1/sqrt(d) [P3], rounded to f32; boundaries are the f32 midpoints of the
 * f32 centroids (computed in fp64, then rounded).
 */
void orc_codebook_f32(int bits, int d, float* c32, float* t32) {
  double c[16], t[15];
  orc_lloyd_max_gaussian(bits, c, t, NULL);
  const int K = 1 << bits;
  for (int k = 0; k < K; ++k) c32[k] = (float)(c[k] / sqrt((double)d));
  for (int k = 0; k + 1 < K; ++k) t32[k] = (float)(0.5 * ((double)c32[k] + (double)c32[k + 1]));
}

/* ------------------------------------------------------------------------- */
/* Sign diagonal: SplitMix64                                                 */
/* ------------------------------------------------------------------------- */
uint64_t orc_splitmix64_next(uint64_t* state) {
  *state += 0x9E3779B97F4A7C15ull;
  uint64_t z = *state;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* s_j = -1 when the top bit of the j-th SplitMix64 output is set, else +1. */
void orc_signs(uint64_t seed, int d, int8_t* s) {
  uint64_t state = seed;
  for (int j = 0; j < d; ++j) s[j] = (orc_splitmix64_next(&state) >> 63) ? -1 : 1;
}

/* ------------------------------------------------------------------------- */
/* Orthonormal Walsh-Hadamard transform (Sylvester order), in place          */
/* ------------------------------------------------------------------------- */
void orc_fwht(double* v, int d) {
  for (int h = 1; h < d; h *= 2)
    for (int i = 0; i < d; i += 2 * h)
      for (int j = i; j < i + h; ++j) {
        double a = v[j], b = v[j + h];
        v[j] = a + b;
        v[j + h] = a - b;
      }
  const double inv = 1.0 / sqrt((double)d);
  for (int j = 0; j < d; ++j) v[j] *= inv;
}

/* ------------------------------------------------------------------------- */
/* bf16                                                                      */
/* ------------------------------------------------------------------------- */
double orc_bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a finite double to the nearest bf16 (8 significant bits), ties to
 * even, directly from the exact value (no intermediate f32 rounding). */
uint16_t orc_double_to_bf16(double y) {
  if (y == 0.0) return signbit(y) ? 0x8000 : 0x0000;
  int e;
  double m = frexp(y, &e);               /* y = m * 2^e, 0.5 <= |m| < 1 */
  double r = nearbyint(ldexp(m, 8));     /* 8 significant bits, ties to even */
  float f = (float)ldexp(r, e - 8);      /* exactly representable */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* bf16 of each of n doubles (orc_double_to_bf16 applied elementwise). */
void orc_bf16_round_array(const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_double_to_bf16(x[i]);
}

/* ------------------------------------------------------------------------- */
/* Record layout                                                             */
/* ------------------------------------------------------------------------- */
/*
 * One record holds 128 consecutive tokens of one (layer, batch, kv-head)
 * stream [P4 "What landed": packed records with the norm inside the record;
 * "Eviction is chunked": EVICT_CHUNK = 128]:
 *   codes   128 rows of d*b/8 bytes (row = token slot, LSB-first bitstream)
 *   norms   128 x f32
 *   when outliers are on:
 *   ocount  128 x u8   (entries stored for each slot)
 *   entries cap x {u16 index, u16 bf16 value}, in (slot, index) order
 * Offsets are returned through the pointers; the function returns the size.
 */
int64_t orc_record_layout(int d, int bits, int has_outliers, int cap, int64_t* off_norm,
                          int64_t* off_count, int64_t* off_entries) {
  int64_t row = (int64_t)d * bits / 8;
  int64_t on = ORC_CHUNK * row;
  int64_t oc = on + 4 * ORC_CHUNK;
  int64_t oe = oc + ORC_CHUNK;
  if (off_norm) *off_norm = on;
  if (off_count) *off_count = oc;
  if (off_entries) *off_entries = oe;
  return has_outliers ? oe + 4 * (int64_t)cap : oc;
}

/* ------------------------------------------------------------------------- */
/* Encode                                                                    */
/* ------------------------------------------------------------------------- */
/*
 * Encode one vector x (d bf16 values) [P1 M4 Phase A/B; problem statement]:
 *   n = ||x|| (fp64, stored as f32); u = x / n; y = H (s . u) / sqrt(d);
 *   code_j = #{k : y_j > t_k};
 *   outlier_j = (T > 0) and |y_j| > T / sqrt(d), value bf16(y_j).
 * A zero vector gives y = 0.  y (fp64) is returned for boundary accounting.
 *
 * The stored per-vector scale S (the record's f32 "norm" field, by which
 * decode multiplies H(yhat)) is chosen by scale_mode [P2, the EDEN-scale
 * commits and their Appendix A note; P1's matched-norm operating point].
 * With chat the dequantised rotated vector (centroids c32[code_j], replaced by
 * the bf16 value at every outlier coordinate of the vector) and the decoded
 * vector xhat = S s.H(chat)/sqrt(d):
 *   0  S = ||x||                                    (the plain codec)
 *   1  S = ||x|| / ||chat||                         matched norm: ||xhat|| = ||x||
 *   2  S = ||x|| / <chat, y>  = ||x||^2 / <c, x>    inner-product preserving: <xhat, x> = ||x||^2
 *   3  S = ||x|| <chat, y> / ||chat||^2 = <c, x> / ||c||^2
 *                                                   least squares: min over S of ||x - xhat||^2
 * (c = s.H(chat)/sqrt(d), the unit-scale reconstruction in the original basis;
 * the transform is orthonormal, so <c, x> = ||x|| <chat, y> and ||c|| = ||chat||.)
 * Modes 2 and 3 multiply to the square of mode 1.  A zero vector stores 0.
 */
void orc_encode_vector(const uint16_t* x, int d, int bits, const float* c32, const float* t32,
                       const int8_t* s, double T, int scale_mode, uint8_t* code, float* norm,
                       uint8_t* is_out, uint16_t* oval, double* y_out) {
  double y[512];
  double ss = 0.0;
  for (int j = 0; j < d; ++j) {
    double xj = orc_bf16_to_double(x[j]);
    ss += xj * xj;
  }
  double n = sqrt(ss);
  *norm = (float)n;
  for (int j = 0; j < d; ++j) y[j] = (n > 0.0) ? s[j] * (orc_bf16_to_double(x[j]) / n) : 0.0;
  orc_fwht(y, d);
  const int nb = (1 << bits) - 1;
  const double thr = T / sqrt((double)d);
  for (int j = 0; j < d; ++j) {
    int c = 0;
    for (int k = 0; k < nb; ++k)
      if (y[j] > (double)t32[k]) ++c;
    code[j] = (uint8_t)c;
    int o = (T > 0.0) && (fabs(y[j]) > thr);
    is_out[j] = (uint8_t)o;
    oval[j] = o ? orc_double_to_bf16(y[j]) : 0;
    if (y_out) y_out[j] = y[j];
  }
  if (scale_mode != 0 && n > 0.0) {
    double cc = 0.0, cy = 0.0;
    for (int j = 0; j < d; ++j) {
      const double cj = is_out[j] ? orc_bf16_to_double(oval[j]) : (double)c32[code[j]];
      cc += cj * cj;
      cy += cj * y[j];
    }
    double S = n;
    if (scale_mode == 1) S = n / sqrt(cc);
    else if (scale_mode == 2) S = n / cy;
    else if (scale_mode == 3) S = n * cy / cc;
    *norm = (float)S;
  }
}

/* Encode n vectors (row stride in elements) into per-coordinate arrays. */
void orc_encode_vectors(const uint16_t* x, int64_t n, int d, int64_t stride, int bits,
                        const float* c32, const float* t32, const int8_t* s, double T, int scale_mode,
                        uint8_t* codes, float* norms, uint8_t* is_out, uint16_t* oval, double* y) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i)
    orc_encode_vector(x + i * stride, d, bits, c32, t32, s, T, scale_mode, codes + i * d, norms + i,
                      is_out + i * d, oval + i * d, y ? y + i * d : NULL);
}

/*
 * Pack n_tok (<= 128) encoded tokens into one record.  Slots beyond n_tok
 * keep whatever the buffer holds.  Outlier entries are appended in (slot,
 * index) order; a slot stores at most 255 and the record at most cap; the
 * rest keep their ordinary codes (the code is written at every coordinate).
 */
void orc_pack_record(int d, int bits, int has_outliers, int cap, int n_tok, const uint8_t* codes,
                     const float* norms, const uint8_t* is_out, const uint16_t* oval, uint8_t* rec) {
  int64_t off_norm, off_count, off_ent;
  orc_record_layout(d, bits, has_outliers, cap, &off_norm, &off_count, &off_ent);
  const int64_t row = (int64_t)d * bits / 8;
  for (int i = 0; i < n_tok; ++i) {
    uint8_t* r = rec + i * row;
    memset(r, 0, (size_t)row);
    for (int j = 0; j < d; ++j) {
      int64_t pos = (int64_t)j * bits;
      for (int q = 0; q < bits; ++q)
        if ((codes[i * d + j] >> q) & 1) r[(pos + q) / 8] |= (uint8_t)(1u << ((pos + q) % 8));
    }
    memcpy(rec + off_norm + 4 * i, &norms[i], 4);
  }
  if (!has_outliers) return;
  int total = 0;
  for (int i = 0; i < n_tok; ++i) {
    int cnt = 0;
    for (int j = 0; j < d; ++j) {
      if (!is_out[i * d + j]) continue;
      if (cnt < 255 && total < cap) {
        uint8_t* e = rec + off_ent + 4 * total;
        uint16_t idx = (uint16_t)j, v = oval[i * d + j];
        e[0] = (uint8_t)(idx & 0xff);
        e[1] = (uint8_t)(idx >> 8);
        e[2] = (uint8_t)(v & 0xff);
        e[3] = (uint8_t)(v >> 8);
        ++cnt;
        ++total;
      }
    }
    rec[off_count + i] = (uint8_t)cnt;
  }
}

/* ------------------------------------------------------------------------- */
/* Decode                                                                    */
/* ------------------------------------------------------------------------- */
int orc_read_code(const uint8_t* row, int j, int bits) {
  int64_t pos = (int64_t)j * bits;
  int c = 0;
  for (int q = 0; q < bits; ++q) c |= ((row[(pos + q) / 8] >> ((pos + q) % 8)) & 1) << q;
  return c;
}

/*
 * Decode slot `slot` of a record [P1 M5 commit: dequantise, replace outliers,
 * inverse WHT, rescale]:  yhat_j = c[code_j], replaced by the stored bf16
 * value at outlier coordinates;  xhat = n * s . H(yhat) / sqrt(d).
 * With rotated != 0 the result stays in the rotated basis: n * yhat.
 */
void orc_decode_slot(const uint8_t* rec, int slot, int d, int bits, int has_outliers, int cap,
                     const float* c32, const int8_t* s, int rotated, double* out) {
  int64_t off_norm, off_count, off_ent;
  orc_record_layout(d, bits, has_outliers, cap, &off_norm, &off_count, &off_ent);
  const int64_t row = (int64_t)d * bits / 8;
  double yh[512];
  for (int j = 0; j < d; ++j) yh[j] = (double)c32[orc_read_code(rec + slot * row, j, bits)];
  if (has_outliers) {
    int first = 0;
    for (int i = 0; i < slot; ++i) first += rec[off_count + i];
    for (int e = 0; e < rec[off_count + slot]; ++e) {
      const uint8_t* p = rec + off_ent + 4 * (first + e);
      int idx = p[0] | (p[1] << 8);
      uint16_t v = (uint16_t)(p[2] | (p[3] << 8));
      yh[idx] = orc_bf16_to_double(v);
    }
  }
  float nf;
  memcpy(&nf, rec + off_norm + 4 * slot, 4);
  const double n = (double)nf;
  if (rotated) {
    for (int j = 0; j < d; ++j) out[j] = n * yh[j];
    return;
  }
  orc_fwht(yh, d);
  for (int j = 0; j < d; ++j) out[j] = n * s[j] * yh[j];
}

/* Decode tokens [0, n) of a record array (record i/128 holds token i). */
void orc_decode_records(const uint8_t* recs, int64_t rec_bytes, int64_t n, int d, int bits,
                        int has_outliers, int cap, const float* c32, const int8_t* s, int rotated,
                        double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i)
    orc_decode_slot(recs + (i / ORC_CHUNK) * rec_bytes, (int)(i % ORC_CHUNK), d, bits,
                    has_outliers, cap, c32, s, rotated, out + i * d);
}

/* ------------------------------------------------------------------------- */
/* Attention                                                                 */
/* ------------------------------------------------------------------------- */
/*
 * Logit soft cap [P4, the softcapping fix]: s -> cap * tanh(s / cap), applied
 * to s = scale * q . k before the logit is stored and before the maximum is
 * taken.  cap = 0 means no cap (the pages' own kernel uses 1.0 as its "off"
 * value; here 1.0 is an ordinary cap).
 */
static double soft_cap(double s, double cap) { return cap > 0.0 ? cap * tanh(s / cap) : s; }

/*
 * Brute-force softmax attention of G query rows over n keys/values, all in the
 * original basis and fp64:  out_g = sum_i softmax_i(cap(scale * q_g . k_i)) v_i.
 * With n = 0 the output is zero.
 */
void orc_attention(const double* q, int G, const double* K, const double* V, int64_t n, int d,
                   double scale, double softcap, double* out) {
#pragma omp parallel for schedule(static)
  for (int g = 0; g < G; ++g) {
    double* o = out + (int64_t)g * d;
    for (int j = 0; j < d; ++j) o[j] = 0.0;
    if (n == 0) continue;
    double* logit = (double*)malloc(sizeof(double) * (size_t)n);
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
      double acc = 0.0;
      for (int j = 0; j < d; ++j) acc += q[(int64_t)g * d + j] * K[i * d + j];
      logit[i] = soft_cap(scale * acc, softcap);
      if (logit[i] > m) m = logit[i];
    }
    double Z = 0.0;
    for (int64_t i = 0; i < n; ++i) {
      double p = exp(logit[i] - m);
      Z += p;
      for (int j = 0; j < d; ++j) o[j] += p * V[i * d + j];
    }
    for (int j = 0; j < d; ++j) o[j] /= Z;
    free(logit);
  }
}

/*
 * Attention with sparse-V dequantisation [P2, turboquant_plus commit log:
 * "safer-asym + sparse-V dequant", value work skipped where the post-softmax
 * weight is negligible].  Tokens 0 .. n_blk_tokens-1 are partitioned into
 * blocks [blk_begin[b], blk_end[b]); each block belongs to sequence blk_seq[b],
 * and the blocks of a sequence are visited in the order they are listed,
 * sharing per query head the running maximum M_h of the logits of the blocks
 * visited before (-inf at the start).  Query heads are taken in groups of
 * `group` consecutive heads; a block's values are skipped for a group when
 * every logit of every head of the group in the block lies below
 * M_h + ln(eps).  Skipped tokens still count in the softmax denominator; tokens
 * outside the blocks are never skipped.  Every logit is computed in fp64 as in
 * orc_attention.  Writes the number of (group, token) pairs skipped.
 */
void orc_attention_sparse_v(const double* q, int G, const double* K, const double* V, int64_t n, int d,
                            double scale, double softcap, double eps, int group, const int64_t* blk_begin,
                            const int64_t* blk_end, const int* blk_seq, int n_blk, int n_seq, double* out,
                            int64_t* skipped) {
  const int n_grp = (G + group - 1) / group;
  double* logit = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * (size_t)G);
  unsigned char* skip = (unsigned char*)calloc((size_t)n_grp * (size_t)(n > 0 ? n : 1), 1);
  for (int g = 0; g < G; ++g)
    for (int64_t i = 0; i < n; ++i) {
      double acc = 0.0;
      for (int j = 0; j < d; ++j) acc += q[(int64_t)g * d + j] * K[i * d + j];
      logit[(int64_t)g * n + i] = soft_cap(scale * acc, softcap);
    }
  int64_t n_skip = 0;
  const double lne = eps > 0.0 ? log(eps) : -INFINITY;
  double* M = (double*)malloc(sizeof(double) * (size_t)G);
  for (int sq = 0; sq < n_seq; ++sq) {
    for (int g = 0; g < G; ++g) M[g] = -INFINITY;
    for (int b = 0; b < n_blk; ++b) {
      if (blk_seq[b] != sq) continue;
      for (int hg = 0; hg < n_grp; ++hg) {
        int all_low = 1;
        for (int g = hg * group; g < G && g < (hg + 1) * group; ++g)
          for (int64_t i = blk_begin[b]; i < blk_end[b]; ++i)
            if (!(logit[(int64_t)g * n + i] < M[g] + lne)) all_low = 0;
        if (all_low && eps > 0.0)
          for (int64_t i = blk_begin[b]; i < blk_end[b]; ++i) {
            skip[(int64_t)hg * n + i] = 1;
            ++n_skip;
          }
      }
      for (int g = 0; g < G; ++g)
        for (int64_t i = blk_begin[b]; i < blk_end[b]; ++i)
          if (logit[(int64_t)g * n + i] > M[g]) M[g] = logit[(int64_t)g * n + i];
    }
  }
  for (int g = 0; g < G; ++g) {
    double* o = out + (int64_t)g * d;
    for (int j = 0; j < d; ++j) o[j] = 0.0;
    if (n == 0) continue;
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i)
      if (logit[(int64_t)g * n + i] > m) m = logit[(int64_t)g * n + i];
    double Z = 0.0;
    for (int64_t i = 0; i < n; ++i) {
      const double p = exp(logit[(int64_t)g * n + i] - m);
      Z += p;
      if (skip[(int64_t)(g / group) * n + i]) continue;
      for (int j = 0; j < d; ++j) o[j] += p * V[i * d + j];
    }
    for (int j = 0; j < d; ++j) o[j] /= Z;
  }
  if (skipped) *skipped = n_skip;
  free(M);
  free(skip);
  free(logit);
}

/*
 * The same attention evaluated the way the fused kernel organises it (a
 * cross-check of the oracle, not a second reference): the query is rotated
 * once, q~ = H(s_k . q)/sqrt(d); a compressed key scores as n_i * q~ . yhat_i;
 * compressed values accumulate n_i * yhat_i in the rotated basis, and one
 * inverse transform s_v . H(acc)/sqrt(d) brings them back; dense (bf16) keys
 * and values are used as they are.
 *   Kr, Vr: compressed keys/values in the rotated basis (n_i * yhat_i) [nc][d]
 *   Kd, Vd: dense keys/values [nd][d]
 */
void orc_attention_rotated(const double* q, int G, const double* Kr, const double* Vr, int64_t nc,
                           const double* Kd, const double* Vd, int64_t nd, int d, double scale,
                           double softcap, const int8_t* sk, const int8_t* sv, double* out) {
  for (int g = 0; g < G; ++g) {
    double qt[512], acc_r[512], acc_d[512];
    for (int j = 0; j < d; ++j) qt[j] = sk[j] * q[(int64_t)g * d + j];
    orc_fwht(qt, d);
    for (int j = 0; j < d; ++j) acc_r[j] = acc_d[j] = 0.0;
    const int64_t n = nc + nd;
    double* o = out + (int64_t)g * d;
    if (n == 0) {
      for (int j = 0; j < d; ++j) o[j] = 0.0;
      continue;
    }
    double* logit = (double*)malloc(sizeof(double) * (size_t)n);
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
      double acc = 0.0;
      if (i < nc)
        for (int j = 0; j < d; ++j) acc += qt[j] * Kr[i * d + j];
      else
        for (int j = 0; j < d; ++j) acc += q[(int64_t)g * d + j] * Kd[(i - nc) * d + j];
      logit[i] = soft_cap(scale * acc, softcap);
      if (logit[i] > m) m = logit[i];
    }
    double Z = 0.0;
    for (int64_t i = 0; i < n; ++i) {
      double p = exp(logit[i] - m);
      Z += p;
      if (i < nc)
        for (int j = 0; j < d; ++j) acc_r[j] += p * Vr[i * d + j];
      else
        for (int j = 0; j < d; ++j) acc_d[j] += p * Vd[(i - nc) * d + j];
    }
    orc_fwht(acc_r, d);
    for (int j = 0; j < d; ++j) o[j] = (sv[j] * acc_r[j] + acc_d[j]) / Z;
    free(logit);
  }
}

/* ------------------------------------------------------------------------- */
/* Chunked eviction bound                                                    */
/* ------------------------------------------------------------------------- */
/*
 * [P4 "What landed" / "Eviction is chunked, on purpose" / "Mutation runs"]:
 * the dense tail is bounded by window + max(t_q - 1, margin) + EVICT_CHUNK.
 * retention floor = window + max(t_q - 1, margin): tokens the tail must keep.
 * Number of whole chunks that leave a tail of `tail_len` tokens: the largest
 * k with tail_len - k * chunk >= retention floor (0 when none).
 */
/*
 * Rollback of one stream to new_len tokens [P4 "What landed": the cache reports
 * its length in tokens and maps truncation onto both time bases, the packed
 * records and the dense tail; a deep rollback has to dequantise].  Given
 * n_chunks, tail_len and new_len, writes the new counters and the number of
 * leading tokens of record n_chunks' that must be decoded into the tail:
 *   T = clamp(new_len, 0, 128 n + len);
 *   T >= 128 n: n' = n, len' = T - 128 n, start kept, nothing decoded;
 *   T <  128 n: n' = T / 128, len' = T mod 128, start' = 0, len' tokens of
 *               record n' decoded.
 * Returns the number of tokens to decode.
 */
int orc_rollback_counts(int n_chunks, int tail_len, int new_len, int* n_out, int* len_out, int* start_reset) {
  const int total = ORC_CHUNK * n_chunks + tail_len;
  const int T = new_len < 0 ? 0 : (new_len > total ? total : new_len);
  if (T >= ORC_CHUNK * n_chunks) {
    *n_out = n_chunks;
    *len_out = T - ORC_CHUNK * n_chunks;
    *start_reset = 0;
    return 0;
  }
  *n_out = T / ORC_CHUNK;
  *len_out = T % ORC_CHUNK;
  *start_reset = 1;
  return *len_out;
}

int orc_retention_floor(int window, int t_q, int margin) {
  return window + ((t_q - 1) > margin ? (t_q - 1) : margin);
}

int orc_chunks_to_evict(int tail_len, int window, int t_q, int margin, int chunk) {
  int floor_ = orc_retention_floor(window, t_q, margin);
  if (tail_len < floor_ + chunk) return 0;
  return (tail_len - floor_) / chunk;
}
