/*
 * pgd_oracle_fp8.c -- the oracle for the 8-bit KV cache: FP8 E4M3 codes with
 * one fp32 scale per (block, KV head, slot), i.e. per (token, head).
 *
 * TEST INFRASTRUCTURE, like pgd_oracle.c: only the test suite, the package
 * smoke check and the benchmark's CPU-baseline leg may load or call it.  It
 * shares no code with the CUDA library.
 *
 * Sources (page title, section):
 *  - "Module 10: inference and serving", section "Quantize the cache,
 *    evaluate the final artifact": a one-byte cache halves the cache's memory
 *    and its read traffic, at the price of scale metadata and quantisation
 *    work.
 *  - "Ch. 6 Inference efficiency and serving", 6.6.1: x is approximated by
 *    s * round(x / s); symmetric quantisation fixes the zero point and takes
 *    the scale from the largest absolute value; an all-zero tensor takes any
 *    positive scale (never s = 0).  6.6.2: the scale's granularity, with the
 *    KV cache as one quantised object.
 *  - "The math of Transformer inference", section 11 (quantisation of weights
 *    and KV): int8/fp8 KV halves the time to read the cache; KV scales are
 *    usually taken per head and per token; dequantisation is fused into the
 *    attention kernel.
 *  - The E4M3 format itself (sign, 4 exponent bits with bias 7, 3 mantissa
 *    bits; no infinities; S.1111.111 is NaN; largest finite 448) is the OCP
 *    8-bit floating point specification's, as implemented by the GPU's
 *    e4m3 conversions.
 *
 * Readings (listed in the design notes):
 *  - quantisation of one (token, KV head) row x[0..d): amax = max_i |x_i|,
 *    scale = amax / 448 in binary32 (1 when amax is 0), code_i =
 *    E4M3(x_i / scale) with the division in binary32 and the conversion
 *    rounding to nearest, ties to even, saturating finite values to +-448;
 *  - the dequantised value of a code c in a row with scale s is E4M3(c) * s,
 *    exactly;
 *  - attention over the 8-bit cache is the attention of pgd_oracle.c over the
 *    dequantised K and V (the query stays bf16).
 *
 * Physical layout of an 8-bit pool (the library's choice): [NB][n_kv][bs/8]
 * groups of 8 tokens, each group 8*d + 32 bytes -- the codes of its 8 tokens
 * as 8-row x 16-byte core matrices (code of group slot r, dim i at
 * (i / 16) * 128 + r * 16 + i % 16), then the 8 tokens' fp32 scales (scale
 * of group slot r at 8*d + 4*r, little-endian binary32).
 *
 * Mutations (tests plant them here to check the pins): 9 K scales ignored,
 * 10 V scales ignored, 11 codes read in 16-bit core-matrix order (8 x 8),
 * 12 quantiser truncates instead of rounding to nearest.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ---------------------------------------------------------------- E4M3 */

/* Value of an E4M3 code: subnormals m/8 * 2^-6, normals (1 + m/8) *
 * 2^(e - 7), S.1111.111 is NaN. */
double oracle_e4m3_decode(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  double v = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/* Nearest E4M3 code to x (binary32), ties to even, finite values beyond the
 * largest code saturate to +-448; NaN gives the NaN code S.1111.111. */
uint8_t oracle_e4m3_encode_mode(float x, int truncate) {
  if (isnan(x)) return 0x7F;
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (a >= 448.0) return sign | 0x7E;
  double (*rnd)(double) = truncate ? trunc : nearbyint; /* nearbyint: ties to even */
  if (a < ldexp(1.0, -6)) {
    /* subnormal grid, spacing 2^-9; a count of 8 is the smallest normal */
    int q = (int)rnd(a / ldexp(1.0, -9));
    return sign | (uint8_t)q;
  }
  int k;
  frexp(a, &k);            /* a = f * 2^k, f in [0.5, 1) */
  int e = k - 1;           /* 2^e <= a < 2^(e+1) */
  int q = (int)rnd(a / ldexp(1.0, e - 3)); /* in [8, 16] */
  if (q == 16) {
    q = 8;
    e += 1;
  }
  return sign | (uint8_t)(((e + 7) << 3) | (q - 8));
}

uint8_t oracle_e4m3_encode(float x) { return oracle_e4m3_encode_mode(x, 0); }

/* The 256 code values, filled from oracle_e4m3_decode before any worker
 * thread starts (a plain cache of the definition above). */
static double e4m3_value[256];
static void fill_e4m3_values(void) {
  for (int c = 0; c < 256; ++c) e4m3_value[c] = oracle_e4m3_decode((uint8_t)c);
}

/* Bytes of one 8-token group: codes, then scales. */
static size_t group_bytes(int d) { return (size_t)8 * d + 32; }

/* Byte offset of the group holding `slot` of (block, head) in the pool. */
static size_t group_base(int blk, int g, int slot, int n_kv, int bs, int d) {
  return (((size_t)blk * n_kv + g) * (size_t)(bs >> 3) + (size_t)(slot >> 3)) * group_bytes(d);
}

/* Offset of the code of dim i of group slot r inside its group. */
static size_t code_offset(int r, int i) {
  return (size_t)(i >> 4) * 128 + (size_t)r * 16 + (size_t)(i & 15);
}

/* Offset under the 16-bit (8 x 8) core-matrix order -- mutation 11 only. */
static size_t code_offset16(int r, int i) {
  return (size_t)(i >> 3) * 64 + (size_t)r * 8 + (size_t)(i & 7);
}

static float load_scale(const uint8_t *group, int d, int r) {
  float f;
  memcpy(&f, group + (size_t)8 * d + (size_t)4 * r, sizeof f);
  return f;
}

static void store_scale(uint8_t *group, int d, int r, float f) {
  memcpy(group + (size_t)8 * d + (size_t)4 * r, &f, sizeof f);
}

static float bf16_bits_to_float(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Quantise one row of d bf16 values: codes[i] and the row's scale. */
void oracle_quantize_row(const uint16_t *x, int d, uint8_t *codes, float *scale_out,
                         int mutation) {
  float amax = 0.0f;
  for (int i = 0; i < d; ++i) {
    float a = fabsf(bf16_bits_to_float(x[i]));
    if (a > amax) amax = a;
  }
  volatile float num = amax, den = 448.0f;
  float scale = (amax > 0.0f) ? num / den : 1.0f;
  for (int i = 0; i < d; ++i) {
    volatile float xi = bf16_bits_to_float(x[i]), sc = scale;
    float y = xi / sc;
    codes[i] = oracle_e4m3_encode_mode(y, mutation == 12);
  }
  *scale_out = scale;
}

/* ------------------------------------------------------------ kv_append */

/* For every sequence b and KV head g: quantise k_new[b][g][:] and
 * v_new[b][g][:] and store the codes and the scale at slot positions[b] % bs
 * of block table[b][positions[b] / bs].  Returns 0, or 1 if a position or
 * block id is out of range (that sequence is skipped). */
int oracle_kv_append_fp8(uint8_t *k_cache, uint8_t *v_cache, const uint16_t *k_new,
                         const uint16_t *v_new, const int32_t *block_tables,
                         const int32_t *positions, int B, int n_kv, int d, int bs, int MB,
                         int NB, int mutation) {
  int status = 0;
  uint8_t *row = (uint8_t *)malloc((size_t)d);
  if (!row) return 2;
  for (int b = 0; b < B; ++b) {
    int32_t pos = positions[b];
    if (pos < 0 || pos >= MB * bs) { status = 1; continue; }
    int32_t blk = block_tables[(size_t)b * MB + pos / bs];
    if (blk < 0 || blk >= NB) { status = 1; continue; }
    int slot = pos % bs, r = slot & 7;
    for (int g = 0; g < n_kv; ++g) {
      size_t base = group_base(blk, g, slot, n_kv, bs, d);
      size_t src = ((size_t)b * n_kv + g) * d;
      float sc;
      oracle_quantize_row(k_new + src, d, row, &sc, mutation);
      for (int i = 0; i < d; ++i) k_cache[base + code_offset(r, i)] = row[i];
      store_scale(k_cache + base, d, r, sc);
      oracle_quantize_row(v_new + src, d, row, &sc, mutation);
      for (int i = 0; i < d; ++i) v_cache[base + code_offset(r, i)] = row[i];
      store_scale(v_cache + base, d, r, sc);
    }
  }
  free(row);
  return status;
}

/* ------------------------------------------------------------ attention */

typedef struct {
  double *out;
  const uint16_t *q;
  const uint8_t *k_cache, *v_cache;
  const int32_t *tables, *ctx;
  int B, n_q, n_kv, d, bs, MB, NB;
  double scale;
  int mutation;
  long row_begin, row_end;
  int status;
} job8;

/* Dequantised element i of token t (sequence b, KV head g) from `cache`;
 * 0 on success, 1 on a bad block id. */
static int elem8(const job8 *J, const uint8_t *cache, int use_scale, int b, int g, int t, int i,
                 double *v) {
  int32_t blk = J->tables[(size_t)b * J->MB + t / J->bs];
  if (blk < 0 || blk >= J->NB) return 1;
  int slot = t % J->bs, r = slot & 7;
  const uint8_t *group = cache + group_base(blk, g, slot, J->n_kv, J->bs, J->d);
  size_t off = (J->mutation == 11) ? code_offset16(r, i) : code_offset(r, i);
  double s = use_scale ? (double)load_scale(group, J->d, r) : 1.0;
  *v = e4m3_value[group[off]] * s;
  return 0;
}

/* One (b, h) row: the definition over dequantised K and V, in double. */
static int attend_row8(const job8 *J, int b, int h) {
  const int d = J->d, G = J->n_q / J->n_kv, g = h / G;
  const int ctx = J->ctx[b];
  if (ctx < 1 || ctx > J->MB * J->bs) return 1;
  const uint16_t *qrow = J->q + ((size_t)b * J->n_q + h) * d;
  double *orow = J->out + ((size_t)b * J->n_q + h) * d;
  double *s = (double *)malloc(sizeof(double) * (size_t)ctx);
  if (!s) return 2;
  double smax = -INFINITY;
  for (int t = 0; t < ctx; ++t) {
    double acc = 0.0;
    for (int i = 0; i < d; ++i) {
      double kv;
      if (elem8(J, J->k_cache, J->mutation != 9, b, g, t, i, &kv)) {
        free(s);
        return 1;
      }
      acc += (double)bf16_bits_to_float(qrow[i]) * kv;
    }
    s[t] = J->scale * acc;
    if (s[t] > smax) smax = s[t];
  }
  double denom = 0.0;
  for (int t = 0; t < ctx; ++t) {
    s[t] = exp(s[t] - smax);
    denom += s[t];
  }
  for (int i = 0; i < d; ++i) orow[i] = 0.0;
  for (int t = 0; t < ctx; ++t) {
    double w = s[t] / denom;
    for (int i = 0; i < d; ++i) {
      double vv;
      elem8(J, J->v_cache, J->mutation != 10, b, g, t, i, &vv);
      orow[i] += w * vv;
    }
  }
  free(s);
  return 0;
}

static void *worker8(void *arg) {
  job8 *J = (job8 *)arg;
  for (long r = J->row_begin; r < J->row_end; ++r) {
    int st = attend_row8(J, (int)(r / J->n_q), (int)(r % J->n_q));
    if (st && !J->status) J->status = st;
  }
  return NULL;
}

/* out[b][h][:] = sum_t softmax_t(scale * q[b][h] . k~_t) v~_t over t <
 * context_lens[b], where k~, v~ are the dequantised codes (code value times
 * the token's scale) of KV head h / G.
 * n_threads <= 0: one per online core.  Returns 0, or 1 on an invalid
 * context length or block id. */
int oracle_paged_attention_fp8(double *out, const uint16_t *q, const uint8_t *k_cache,
                               const uint8_t *v_cache, const int32_t *block_tables,
                               const int32_t *context_lens, int B, int n_q, int n_kv, int d,
                               int bs, int MB, int NB, double scale, int n_threads,
                               int mutation) {
  if (B < 0 || n_q <= 0 || n_kv <= 0 || n_q % n_kv || d <= 0 || d % 16 || bs <= 0 || bs % 8 ||
      MB <= 0 || NB <= 0)
    return 1;
  long rows = (long)B * n_q;
  if (rows == 0) return 0;
  if (n_threads <= 0) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    n_threads = n > 0 ? (int)n : 1;
  }
  if (n_threads > 256) n_threads = 256;
  if (rows < n_threads) n_threads = (int)rows;
  fill_e4m3_values();
  job8 base = {out, q, k_cache, v_cache, block_tables, context_lens,
               B, n_q, n_kv, d, bs, MB, NB, scale, mutation, 0, 0, 0};
  job8 *jobs = (job8 *)calloc((size_t)n_threads, sizeof(job8));
  pthread_t *th = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
  if (!jobs || !th) { free(jobs); free(th); return 2; }
  for (int i = 0; i < n_threads; ++i) {
    jobs[i] = base;
    jobs[i].row_begin = rows * i / n_threads;
    jobs[i].row_end = rows * (i + 1) / n_threads;
  }
  for (int i = 1; i < n_threads; ++i) pthread_create(&th[i], NULL, worker8, &jobs[i]);
  worker8(&jobs[0]);
  int status = jobs[0].status;
  for (int i = 1; i < n_threads; ++i) {
    pthread_join(th[i], NULL);
    if (jobs[i].status && !status) status = jobs[i].status;
  }
  free(jobs);
  free(th);
  return status;
}
