/*
 * pa_oracle.c -- plain fp64 CPU oracle for paged-attention decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or constant with the CUDA path.
 *
 * What it computes (the plain definition; tiling, online softmax and
 * split-context partitions only reorder it):
 *
 *   For sequence s, query position i, query head h, KV head hkv = h / G and
 *   L = context_lens[s]:
 *     L == 0  -> out = 0        ("[FlyDSL] pa_decode: MXFP4 K/V in the shared
 *                                 PA tile kernel", plan-free commit: context-0
 *                                 rows are zero-filled on both paths)
 *     for t in [0, L): blk = block_tables[s, t / S], slot = t mod S
 *        (only owned rows are read: "[FlyDSL] pa_decode: zero V rows past the
 *         context before PV", Root cause / Fix -- rows at or past the context
 *         length never reach the output)
 *     x_t = softmax_scale * q_scale * sum_d q[d] * k_t[d]
 *     out = sum_t exp(x_t - M) v_t / sum_t exp(x_t - M),  M = max_t x_t
 *   computed in two passes, in double precision.
 *   With causal set (query length > 1; the first page notes a causal option that a later
 *   change adds next to the masking flag), query position i sees only the tokens
 *   t < L - qlen + 1 + i: the context ends with the qlen query tokens themselves, and
 *   each sees itself and what precedes it.  A position that sees no token gives zeros.
 *   With a sliding window W > 0 (the first page lists sliding-window plans among the
 *   variants its probe covers; the pages do not define it further), query position i,
 *   whose own place in the context is p = L - qlen + i, sees only the tokens t > p - W:
 *   the W tokens ending at itself, cut further by causal masking when that is set.
 *   Tokens before every position's window (t < L - qlen - W + 1) are never read.
 *   With sinks (one fp32 logit per query head, in the units of the softmax-scaled scores;
 *   the pages list "sinks" beside sliding window among what the MXFP4 path refuses,
 *   without defining them), every row's softmax takes one more term with a zero value:
 *   out = sum_t exp(x_t - M) v_t / (sum_t exp(x_t - M) + exp(s_h - M)),
 *   M = max(max_t x_t, s_h); a row that sees no token gives zeros.
 *   With trans_v set, the value cache stores each page head-dim major: [NB, Hkv, D, S],
 *   the S tokens of one head dim contiguous (the first page's probe covers fp8
 *   per-tensor caches in a trans_v layout as well as with plain V, without defining it; this
 *   is the plain transposed reading, and the layout of vLLM's classic value cache).
 *
 * Storage formats are decoded from their definitions:
 *   bf16      : the high half of an IEEE binary32
 *   e4m3 (OCP): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0
 *               is subnormal m/8 * 2^-6; S.1111.111 is NaN; there is no Inf
 *               (the first page's Tests section: the "inf" fill of e4m3 is the
 *               finite +-448)
 *   e2m1      : 1 sign, 2 exponent bits (bias 1), 1 mantissa bit
 *   e8m0      : 2^(b - 127); b = 255 is NaN
 *   MXFP4 row : "[FlyDSL] pa_decode: MXFP4 K/V ...", Summary: data uint8
 *               [pages, kv_heads, 128, 64] (two e2m1 per byte), scales uint8
 *               e8m0 [pages, kv_heads, 128, 4], one scale per 32 values along
 *               head_dim.  Element 2j is the low nibble of byte j, 2j+1 the
 *               high nibble (the OCP MX packing; the pages do not say).
 *
 * All tensors are dense and contiguous:
 *   query        [B, qlen, Hq, D]        bf16 or e4m3 bytes.  A bf16 query may also be read
 *                as the MXFP4 page quantises it ("[FlyDSL] pa_decode: MXFP4 K/V ...",
 *                Summary: bf16 Q is quantised to e4m3 per head row in the kernel): per
 *                row, s = amax / 448 and y = q / s in fp32 (round to nearest), y rounded
 *                to the nearest e4m3 value (ties to even, finite at +-448), read back as
 *                e4m3(y) * s; a zero row stays zero.
 *   q_scale      scalar or [B, qlen, Hq] fp32 (e4m3 query only)
 *   key/value    [NB, Hkv, S, row_bytes] (row_bytes = 2D bf16, D e4m3, D/2 MXFP4);
 *                value [NB, Hkv, D, S] elements with trans_v
 *   scales       per-tensor: fp32 [1]; per-token: fp32 [NB, Hkv, S];
 *                e8m0: uint8 [NB, Hkv, S, D/32]
 *   block_tables [B, max_blocks_per_seq] int32; context_lens [B] int32
 *   out          [B, qlen, Hq, D] double
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_KV_BF16 = 0, ORC_KV_E4M3 = 1, ORC_KV_MXFP4 = 2 };
enum { ORC_SCALE_NONE = 0, ORC_SCALE_TENSOR = 1, ORC_SCALE_TOKEN = 2, ORC_SCALE_E8M0 = 3 };
enum { ORC_Q_BF16 = 0, ORC_Q_E4M3 = 1, ORC_Q_BF16_TO_E4M3 = 2 };

typedef struct {
  int32_t batch, qlen, num_q_heads, num_kv_heads, head_dim, page_size;
  int32_t num_blocks, max_blocks_per_seq;
  int32_t kv_format, scale_kind, q_format, q_scale_per_row;
  double softmax_scale;
  const void* query;
  const float* q_scale;
  const void* key_cache;
  const void* value_cache;
  const void* key_scale;
  const void* value_scale;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int32_t causal;
  int32_t window; /* sliding window W (0: none) */
  int32_t trans_v; /* value cache [NB, Hkv, D, S] (bf16 / e4m3 only) */
  const float* sinks; /* [Hq] or NULL */
} orc_args;

/* ---- format decoders ---------------------------------------------------- */

double orc_bf16(uint16_t bits) {
  uint32_t w = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

double orc_e4m3(uint8_t b) {
  int sign = b >> 7;
  int e = (b >> 3) & 15;
  int m = b & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -mag : mag;
}

double orc_e2m1(uint8_t nibble) {
  int sign = (nibble >> 3) & 1;
  int e = (nibble >> 1) & 3;
  int m = nibble & 1;
  double mag;
  if (e == 0)
    mag = 0.5 * (double)m;
  else
    mag = ldexp(1.0 + 0.5 * (double)m, e - 1);
  return sign ? -mag : mag;
}

double orc_e8m0(uint8_t b) {
  if (b == 255) return NAN;
  return ldexp(1.0, (int)b - 127);
}

/* Nearest e4m3 (OCP) value to y, ties to even, saturating at +-448 (the largest finite
 * e4m3); the spacing is 2^(E-3) in the binade [2^E, 2^(E+1)), E >= -6 (below 2^-6 the
 * subnormal spacing 2^-9 continues). */
double orc_e4m3_round(float y) {
  if (isnan(y)) return NAN;
  double a = fabs((double)y);
  if (a >= 448.0) return y < 0 ? -448.0 : 448.0;
  if (a == 0.0) return (double)y;
  int e;
  (void)frexp(a, &e); /* a = f * 2^e, f in [0.5, 1): binade E = e - 1 */
  int E = e - 1 < -6 ? -6 : e - 1;
  double quantum = ldexp(1.0, E - 3);
  double r = rint(a / quantum) * quantum; /* rint: nearest, ties to even */
  if (r > 448.0) r = 448.0;
  return y < 0 ? -r : r;
}

/* ---- element access ------------------------------------------------------ */

static int64_t row_bytes(const orc_args* a) {
  if (a->kv_format == ORC_KV_BF16) return 2 * (int64_t)a->head_dim;
  if (a->kv_format == ORC_KV_E4M3) return a->head_dim;
  return a->head_dim / 2;
}

/* Dequantized element d of token slot `slot` in page `blk`, KV head `hkv`. */
static double kv_elem(const orc_args* a, const void* cache, const void* scale, int64_t blk,
                      int hkv, int slot, int d, int transposed) {
  const int64_t rb = row_bytes(a);
  const int64_t token = (blk * a->num_kv_heads + hkv) * a->page_size + slot;
  const uint8_t* row = (const uint8_t*)cache + token * rb;
  /* transposed page: element (d, slot) of the [D, S] page of (blk, hkv) */
  const int64_t tel = ((blk * a->num_kv_heads + hkv) * a->head_dim + d) * a->page_size + slot;
  double v;
  if (a->kv_format == ORC_KV_BF16) {
    uint16_t bits;
    if (transposed)
      memcpy(&bits, (const uint8_t*)cache + 2 * tel, 2);
    else
      memcpy(&bits, row + 2 * d, 2);
    v = orc_bf16(bits);
  } else if (a->kv_format == ORC_KV_E4M3) {
    v = orc_e4m3(transposed ? ((const uint8_t*)cache)[tel] : row[d]);
  } else {
    uint8_t byte = row[d / 2];
    uint8_t nib = (d % 2 == 0) ? (byte & 15) : (byte >> 4);
    v = orc_e2m1(nib);
  }
  switch (a->scale_kind) {
    case ORC_SCALE_TENSOR:
      v *= (double)((const float*)scale)[0];
      break;
    case ORC_SCALE_TOKEN:
      v *= (double)((const float*)scale)[token];
      break;
    case ORC_SCALE_E8M0: {
      const int nblk = a->head_dim / 32;
      v *= orc_e8m0(((const uint8_t*)scale)[token * nblk + d / 32]);
      break;
    }
    default:
      break;
  }
  return v;
}

static double q_elem(const orc_args* a, int s, int i, int h, int d) {
  const int64_t qrow = ((int64_t)s * a->qlen + i) * a->num_q_heads + h;
  if (a->q_format == ORC_Q_BF16 || a->q_format == ORC_Q_BF16_TO_E4M3) {
    uint16_t bits;
    memcpy(&bits, (const uint8_t*)a->query + 2 * (qrow * a->head_dim + d), 2);
    return orc_bf16(bits);
  }
  double q = orc_e4m3(((const uint8_t*)a->query)[qrow * a->head_dim + d]);
  double qs = a->q_scale_per_row ? (double)a->q_scale[qrow] : (double)a->q_scale[0];
  return q * qs;
}

/* ---- attention over a token range ---------------------------------------- */

/*
 * Softmax attention of one (s, hkv) group over owned tokens [t0, t1), for every
 * query row of the group (qlen * G rows).  Writes, per row r:
 *   m[r] = max_t x_t, l[r] = sum_t exp(x_t - m[r]), o[r][:] = sum_t exp(x_t - m) v_t / l.
 * A row that sees no token of the range (an empty range, or causal masking) gives
 * m = -inf, l = 0, o = 0.
 */
static void attend_range(const orc_args* a, int s, int hkv, int t0, int t1, double* m,
                         double* l, double* o, double* x, double* qv, double* kv) {
  const int G = a->num_q_heads / a->num_kv_heads;
  const int R = a->qlen * G;
  const int D = a->head_dim;
  const int S = a->page_size;
  const int32_t* bt = a->block_tables + (int64_t)s * a->max_blocks_per_seq;
  const int n = t1 - t0;
  const int L = a->context_lens[s];

  for (int r = 0; r < R; ++r) {
    int i = r / G, h = hkv * G + r % G;
    for (int d = 0; d < D; ++d) qv[(int64_t)r * D + d] = q_elem(a, s, i, h, d);
    if (a->q_format == ORC_Q_BF16_TO_E4M3) { /* quantise the row (see the header) */
      float amax = 0.0f;
      for (int d = 0; d < D; ++d) {
        float q = (float)qv[(int64_t)r * D + d];
        if (fabsf(q) > amax) amax = fabsf(q);
      }
      float sc = amax / 448.0f;
      for (int d = 0; d < D; ++d) {
        float q = (float)qv[(int64_t)r * D + d];
        qv[(int64_t)r * D + d] = amax > 0.0f ? orc_e4m3_round(q / sc) * (double)sc : 0.0;
      }
    }
  }
  /* pass 1: scores */
  for (int r = 0; r < R; ++r) m[r] = -INFINITY;
  for (int j = 0; j < n; ++j) {
    int t = t0 + j;
    int64_t blk = bt[t / S];
    for (int d = 0; d < D; ++d)
      kv[d] = kv_elem(a, a->key_cache, a->key_scale, blk, hkv, t % S, d, 0);
    for (int r = 0; r < R; ++r) {
      if (a->causal && t >= L - a->qlen + 1 + r / G) {  /* after query position r / G */
        x[(int64_t)r * n + j] = -INFINITY;
        continue;
      }
      if (a->window > 0 && t <= L - a->qlen + r / G - a->window) { /* before its window */
        x[(int64_t)r * n + j] = -INFINITY;
        continue;
      }
      double dot = 0.0;
      for (int d = 0; d < D; ++d) dot += qv[(int64_t)r * D + d] * kv[d];
      double xs = a->softmax_scale * dot;
      x[(int64_t)r * n + j] = xs;
      if (xs > m[r]) m[r] = xs;
    }
  }
  /* pass 2: weights and the weighted sum of V */
  for (int r = 0; r < R; ++r) {
    l[r] = 0.0;
    for (int d = 0; d < D; ++d) o[(int64_t)r * D + d] = 0.0;
  }
  for (int j = 0; j < n; ++j) {
    int t = t0 + j;
    int64_t blk = bt[t / S];
    for (int d = 0; d < D; ++d)
      kv[d] = kv_elem(a, a->value_cache, a->value_scale, blk, hkv, t % S, d, a->trans_v);
    for (int r = 0; r < R; ++r) {
      if (x[(int64_t)r * n + j] == -INFINITY) continue; /* not seen by this row */
      double w = exp(x[(int64_t)r * n + j] - m[r]);
      l[r] += w;
      for (int d = 0; d < D; ++d) o[(int64_t)r * D + d] += w * kv[d];
    }
  }
  for (int r = 0; r < R; ++r)
    if (l[r] > 0.0)
      for (int d = 0; d < D; ++d) o[(int64_t)r * D + d] /= l[r];
}

static int check_args(const orc_args* a) {
  if (a->batch < 0 || a->qlen < 1 || a->num_kv_heads < 1 || a->num_q_heads < 1) return -1;
  if (a->causal != 0 && a->causal != 1) return -1;
  if (a->window < 0) return -1;
  if (a->trans_v != 0 && (a->trans_v != 1 || a->kv_format == ORC_KV_MXFP4)) return -1;
  if (a->num_q_heads % a->num_kv_heads) return -1;
  if (a->head_dim < 1 || a->page_size < 1) return -1;
  if (a->kv_format == ORC_KV_MXFP4 && (a->head_dim % 32 || a->scale_kind != ORC_SCALE_E8M0))
    return -1;
  for (int s = 0; s < a->batch; ++s) {
    int L = a->context_lens[s];
    if (L < 0) return -1;
    if ((int64_t)(L + a->page_size - 1) / a->page_size > a->max_blocks_per_seq) return -1;
    for (int p = 0; p < (L + a->page_size - 1) / a->page_size; ++p) {
      int32_t blk = a->block_tables[(int64_t)s * a->max_blocks_per_seq + p];
      if (blk < 0 || blk >= a->num_blocks) return -1;
    }
  }
  return 0;
}

static int max_context(const orc_args* a) {
  int mx = 0;
  for (int s = 0; s < a->batch; ++s)
    if (a->context_lens[s] > mx) mx = a->context_lens[s];
  return mx;
}

/*
 * Full decode.  out: [B, qlen, Hq, D] doubles.  nthreads <= 0 uses the OpenMP
 * default.  Returns 0, or -1 on malformed arguments, -2 on allocation failure.
 */
int orc_pa_decode(const orc_args* a, double* out, int nthreads) {
  if (check_args(a)) return -1;
  const int G = a->num_q_heads / a->num_kv_heads;
  const int R = a->qlen * G;
  const int D = a->head_dim;
  const int Lmax = max_context(a);
  const int units = a->batch * a->num_kv_heads;
  int err = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel
  {
    double* m = malloc(sizeof(double) * R);
    double* l = malloc(sizeof(double) * R);
    double* o = malloc(sizeof(double) * (size_t)R * D);
    double* x = malloc(sizeof(double) * (size_t)R * (Lmax > 0 ? Lmax : 1));
    double* qv = malloc(sizeof(double) * (size_t)R * D);
    double* kv = malloc(sizeof(double) * D);
    if (!m || !l || !o || !x || !qv || !kv) {
#pragma omp atomic write
      err = -2;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int u = 0; u < units; ++u) {
        int s = u / a->num_kv_heads, hkv = u % a->num_kv_heads;
        const int L = a->context_lens[s];
        int t0 = 0; /* first token any query position's window holds */
        if (a->window > 0 && L - a->qlen - a->window + 1 > 0) t0 = L - a->qlen - a->window + 1;
        attend_range(a, s, hkv, t0, L, m, l, o, x, qv, kv);
        for (int r = 0; r < R; ++r) {
          int i = r / G, h = hkv * G + r % G;
          double* dst = out + ((((int64_t)s * a->qlen + i) * a->num_q_heads + h) * D);
          double f = 1.0; /* o = sum_t exp(x_t - m) v_t / l; with a sink the denominator grows */
          if (a->sinks && l[r] > 0.0) {
            const double sk = (double)a->sinks[h];
            const double Mp = m[r] > sk ? m[r] : sk; /* M = max(max_t x_t, s_h) */
            const double num = l[r] * exp(m[r] - Mp);
            f = num / (num + exp(sk - Mp));
          }
          for (int d = 0; d < D; ++d) dst[d] = o[(int64_t)r * D + d] * f;
        }
      }
    }
    free(m); free(l); free(o); free(x); free(qv); free(kv);
  }
  return err;
}

/*
 * Attention of one (s, hkv) group over tokens [t0, t1) of sequence s; t1 must
 * not exceed context_lens[s].  Writes m, l: [qlen*G]; o: [qlen*G, D]; row
 * r = i*G + (h mod G).  Used to check the partition merge identity.
 */
int orc_pa_decode_range(const orc_args* a, int s, int hkv, int t0, int t1, double* m, double* l,
                        double* o) {
  if (check_args(a)) return -1;
  if (s < 0 || s >= a->batch || hkv < 0 || hkv >= a->num_kv_heads) return -1;
  if (t0 < 0 || t1 < t0 || t1 > a->context_lens[s]) return -1;
  const int G = a->num_q_heads / a->num_kv_heads;
  const int R = a->qlen * G;
  const int D = a->head_dim;
  int n = t1 - t0;
  double* x = malloc(sizeof(double) * (size_t)R * (n > 0 ? n : 1));
  double* qv = malloc(sizeof(double) * (size_t)R * D);
  double* kv = malloc(sizeof(double) * D);
  int rc = 0;
  if (!x || !qv || !kv)
    rc = -2;
  else
    attend_range(a, s, hkv, t0, t1, m, l, o, x, qv, kv);
  free(x); free(qv); free(kv);
  return rc;
}

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---- MXFP4 quantisation: the cache write whose pages the decode reads ------------
 *
 * "[FlyDSL] pa_decode: MXFP4 K/V ...", Dependencies: the MXFP4 pages come from a KV write
 * kernel.  The pages name the format (e2m1 values, one e8m0 scale per 32 along head_dim,
 * element 2j in the low nibble of byte j) but not the conversion into it; the conversion
 * here is the OCP MX one.  Per block of 32 values: the shared scale is
 * X = 2^(floor(log2 amax) - 2) (2 = the largest exponent of e2m1, whose largest value is
 * 6 = 1.5 * 2^2), and each value becomes the e2m1 value nearest to x / X, ties to the code
 * with an even mantissa bit, saturating at +-6, keeping the sign (a negative value that
 * rounds to zero is the code of -0).  Where the format leaves a choice: an all-zero block
 * takes scale byte 127 (X = 1); the exponent is clamped to [-126, 127], so scale bytes
 * stay in 1..254 (the decode takes 0 and 255 as undefined in owned rows); a block holding
 * a NaN or an infinity takes byte 255 (NaN) and zero codes.
 */
static uint8_t orc_e2m1_nearest(double y) {
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  const double a = fabs(y);
  int best = 0;
  for (int c = 1; c < 8; ++c) {
    const double dc = fabs(a - mag[c]), db = fabs(a - mag[best]);
    if (dc < db || (dc == db && (c & 1) == 0)) best = c; /* a tie goes to the even code */
  }
  return (uint8_t)(best | (signbit(y) ? 8 : 0));
}

/* Quantises n values (n a multiple of 32) into n/2 data bytes and n/32 scale bytes.
 * Returns 0, or -1 if n is not a multiple of 32. */
int orc_mxfp4_quantize(const float* x, int n, uint8_t* data, uint8_t* scales) {
  if (n <= 0 || n % 32) return -1;
  memset(data, 0, (size_t)n / 2);
  for (int b = 0; b < n / 32; ++b) {
    const float* v = x + 32 * b;
    double amax = 0.0;
    int finite = 1;
    for (int i = 0; i < 32; ++i) {
      if (!isfinite(v[i])) finite = 0;
      else if (fabs((double)v[i]) > amax) amax = fabs((double)v[i]);
    }
    uint8_t sb = 127;
    double X = 1.0;
    if (!finite) {
      sb = 255;
    } else if (amax > 0.0) {
      int e;
      (void)frexp(amax, &e); /* amax = f * 2^e, f in [0.5, 1): floor(log2 amax) = e - 1 */
      int E = (e - 1) - 2;
      E = E < -126 ? -126 : (E > 127 ? 127 : E);
      sb = (uint8_t)(E + 127);
      X = ldexp(1.0, E);
    }
    scales[b] = sb;
    for (int i = 0; i < 32; ++i) {
      const uint8_t code = finite ? orc_e2m1_nearest((double)v[i] / X) : 0;
      const int j = 32 * b + i;
      data[j / 2] |= (uint8_t)(j % 2 == 0 ? code : code << 4);
    }
  }
  return 0;
}
