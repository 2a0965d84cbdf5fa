/*
 * pgd_oracle.c -- the oracle: a plain, slow, float64 CPU statement of what the
 * paged GQA decode path computes.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load or call this code.  It shares no code,
 * header, table or helper with the CUDA library, and it never reads anything
 * the CUDA library produced: it takes the same bf16 bit patterns and the same
 * block tables as plain host arrays.
 *
 * Sources (page title, section):
 *  - "Module 10: inference and serving" (wrwei.github.io), section "Attention
 *    reads a different cache per sequence": one decode position of one layer
 *    scores the query against every cached key of its own sequence and sums
 *    the values; Lab 2 (toy decoder): the new position attends to all old
 *    positions and to itself (mask arange(k_len) <= old + i), scores are the
 *    scaled dot product with the default 1/sqrt(d_head) scale, and KV head g
 *    is repeated G times along the head axis (repeat_interleave), so query
 *    head h reads KV head floor(h / G).
 *  - same page, section "Mapping logical positions to physical blocks": a
 *    per-sequence block table maps logical block j to a physical block of a
 *    shared pool; token t lives in block table[t / bs] at slot t % bs.
 *  - "Ch. 6 Inference efficiency and serving" (glenzli.com), section 6.4
 *    (paged KV management): same mapping, blocks need not be adjacent.
 *  - "LLM inference systems engineering" (jasonzhang109.github.io), section
 *    2.1.3 (computation graph and generation loop): the step writes the
 *    pending token's K/V into the cache, and the cache then holds exactly the
 *    positions already forwarded.
 *  - same book, section 2.8.3 (what FlashAttention reduces): the running
 *    (m, l, o) state of a softmax-weighted sum and its block update.
 *  - "The math of Transformer inference" (hs-black.github.io), section 8,
 *    "the KV cache must be sharded too": split the sequence, compute local
 *    attention per part, merge the parts by log-sum-exp.
 *
 * Physical layout of the pool (the pages fix only the logical shape
 * (B, n_kv, T, d_head) and the block table, so this is the library's choice):
 * [NB][n_kv][tile], one tile per (block, KV head) holding bs x d bf16 values
 * as 8 x 8 core matrices -- element (slot s, dim i) of a tile is at
 * ((s / 8) * (d / 8) + i / 8) * 64 + (s % 8) * 8 + i % 8.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - context_lens[b] counts every cached position including the token just
 *    appended; a decode query attends to all of them.
 *  - scale is a caller argument (1/sqrt(d_head) in every workload).
 *  - a context length below 1, or one that needs more blocks than the table
 *    row holds, is an error (the oracle returns a nonzero code).
 *
 * Arithmetic: every bf16 input is widened exactly to double; everything after
 * that is double.  No blocking or reordering beyond the definitions above.
 *
 * The `mutation` argument exists only so that tests can plant a known mistake
 * here (on the CPU) and check that the pins catch it; 0 means the oracle as
 * defined.  Mutations: 1 slot off by one, 2 head map h % n_kv, 3 partial last
 * block dropped, 4 one slot past the context read, 5 no 1/sqrt(d) scale,
 * 6 no softmax normalisation, 7 K and V swapped, 8 score sign flipped.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Offset of element (slot, i) inside one (block, head) tile. */
static size_t tile_offset(int slot, int i, int d) {
  return ((size_t)(slot >> 3) * (size_t)(d >> 3) + (size_t)(i >> 3)) * 64 +
         (size_t)(slot & 7) * 8 + (size_t)(i & 7);
}

/* ------------------------------------------------------------------ */
/* kv_append: place one new token per sequence into its paged slot.   */
/* ------------------------------------------------------------------ */

/* For every sequence b, the new token sits at logical position
 * positions[b]; its block is table[b][positions[b] / bs] and its slot is
 * positions[b] % bs.  K and V of every KV head are copied bit for bit.
 * Cache layout: [NB][n_kv][tile] as above.  New-token layout: [B][n_kv][d].
 * Returns 0, or 1 if a position or a block id is out of range (nothing is
 * written for that sequence). */
int oracle_kv_append(uint16_t *k_cache, uint16_t *v_cache, const uint16_t *k_new,
                     const uint16_t *v_new, const int32_t *block_tables,
                     const int32_t *positions, int B, int n_kv, int d, int bs, int MB,
                     int NB) {
  int status = 0;
  for (int b = 0; b < B; ++b) {
    int32_t pos = positions[b];
    if (pos < 0 || pos >= MB * bs) { status = 1; continue; }
    int32_t blk = block_tables[(size_t)b * MB + pos / bs];
    if (blk < 0 || blk >= NB) { status = 1; continue; }
    int slot = pos % bs;
    for (int g = 0; g < n_kv; ++g) {
      size_t tile = ((size_t)blk * n_kv + g) * (size_t)bs * d;
      size_t src = ((size_t)b * n_kv + g) * d;
      for (int i = 0; i < d; ++i) {
        k_cache[tile + tile_offset(slot, i, d)] = k_new[src + i];
        v_cache[tile + tile_offset(slot, i, d)] = v_new[src + i];
      }
    }
  }
  return status;
}

/* ------------------------------------------------------------------ */
/* paged decode attention                                              */
/* ------------------------------------------------------------------ */

typedef struct {
  double *out;            /* [B][n_q][d] */
  const uint16_t *q;      /* [B][n_q][d] */
  const uint16_t *k_cache, *v_cache;
  const int32_t *tables;  /* [B][MB] */
  const int32_t *ctx;     /* [B] */
  int B, n_q, n_kv, d, bs, MB, NB;
  double scale;
  int mutation;
  /* work split: rows (b, h) in [row_begin, row_end) */
  long row_begin, row_end;
  int status;
} attn_job;

/* Resolve logical token t of sequence b, KV head g, through the block
 * table: the element offset of its tile and its slot in the tile.  Returns
 * -1 when the table entry is not a valid block id. */
static long token_tile(const attn_job *J, int b, int g, int t, int *slot_out) {
  int j = t / J->bs;
  int slot = t % J->bs;
  if (J->mutation == 1) slot = (t + 1) % J->bs;
  int32_t blk = J->tables[(size_t)b * J->MB + j];
  if (blk < 0 || blk >= J->NB) return -1;
  *slot_out = slot;
  return (long)(((size_t)blk * J->n_kv + g) * (size_t)J->bs * J->d);
}

/* One (sequence b, query head h): scores over every cached position,
 * softmax, weighted sum of values -- the definition, in double. */
static int attend_row(const attn_job *J, int b, int h) {
  const int d = J->d;
  const int G = J->n_q / J->n_kv;
  int g = h / G;
  if (J->mutation == 2) g = h % J->n_kv;
  int ctx = J->ctx[b];
  if (ctx < 1 || ctx > J->MB * J->bs) return 1;
  int n_tok = ctx;
  if (J->mutation == 3) n_tok = (ctx / J->bs) * J->bs;
  if (J->mutation == 4 && ctx < J->MB * J->bs) n_tok = ctx + 1;
  double scale = (J->mutation == 5) ? 1.0 : J->scale;
  const uint16_t *Kc = (J->mutation == 7) ? J->v_cache : J->k_cache;
  const uint16_t *Vc = (J->mutation == 7) ? J->k_cache : J->v_cache;

  const uint16_t *qrow = J->q + ((size_t)b * J->n_q + h) * d;
  double *orow = J->out + ((size_t)b * J->n_q + h) * d;
  double *s = (double *)malloc(sizeof(double) * (size_t)(n_tok > 0 ? n_tok : 1));
  if (!s) return 2;

  /* scores s_t = scale * sum_i q_i k_{t,i} */
  double smax = -INFINITY;
  for (int t = 0; t < n_tok; ++t) {
    int slot = 0;
    long r = token_tile(J, b, g, t, &slot);
    if (r < 0) { free(s); return 1; }
    double acc = 0.0;
    for (int i = 0; i < d; ++i)
      acc += bf16_bits_to_double(qrow[i]) * bf16_bits_to_double(Kc[r + tile_offset(slot, i, d)]);
    s[t] = scale * acc;
    if (J->mutation == 8) s[t] = -s[t];
    if (s[t] > smax) smax = s[t];
  }
  /* softmax weights w_t = exp(s_t - max) / sum_u exp(s_u - max) */
  double denom = 0.0;
  for (int t = 0; t < n_tok; ++t) {
    s[t] = exp(s[t] - smax);
    denom += s[t];
  }
  if (J->mutation == 6) denom = 1.0;
  /* out = sum_t w_t v_t */
  for (int i = 0; i < d; ++i) orow[i] = 0.0;
  for (int t = 0; t < n_tok; ++t) {
    int slot = 0;
    long r = token_tile(J, b, g, t, &slot);
    double w = s[t] / denom;
    for (int i = 0; i < d; ++i) orow[i] += w * bf16_bits_to_double(Vc[r + tile_offset(slot, i, d)]);
  }
  free(s);
  return 0;
}

static void *attn_worker(void *arg) {
  attn_job *J = (attn_job *)arg;
  for (long r = J->row_begin; r < J->row_end; ++r) {
    int b = (int)(r / J->n_q), h = (int)(r % J->n_q);
    int st = attend_row(J, b, h);
    if (st && !J->status) J->status = st;
  }
  return NULL;
}

static int resolve_threads(int n_threads, long rows) {
  if (n_threads <= 0) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    n_threads = (n > 0) ? (int)n : 1;
  }
  if (n_threads > 256) n_threads = 256;
  if (rows < n_threads) n_threads = (int)(rows > 0 ? rows : 1);
  return n_threads;
}

/* Number of threads oracle_paged_attention will use for `rows` rows. */
int oracle_threads_used(int n_threads, long rows) { return resolve_threads(n_threads, rows); }

/* out[b][h][:] = sum_t softmax_t(scale * q[b][h] . k[b][h/G][t]) v[b][h/G][t]
 * over t in [0, context_lens[b]), K/V read through block_tables.
 * Returns 0 on success, 1 on an invalid context length or block id. */
int oracle_paged_attention(double *out, const uint16_t *q, const uint16_t *k_cache,
                           const uint16_t *v_cache, const int32_t *block_tables,
                           const int32_t *context_lens, int B, int n_q, int n_kv, int d,
                           int bs, int MB, int NB, double scale, int n_threads,
                           int mutation) {
  if (B < 0 || n_q <= 0 || n_kv <= 0 || n_q % n_kv || d <= 0 || bs <= 0 || MB <= 0 || NB <= 0 ||
      d % 8 || bs % 8)
    return 1;
  long rows = (long)B * n_q;
  if (rows == 0) return 0;
  int nt = resolve_threads(n_threads, rows);
  attn_job base = {out, q, k_cache, v_cache, block_tables, context_lens, B, n_q, n_kv, d,
                   bs, MB, NB, scale, mutation, 0, 0, 0};
  attn_job *jobs = (attn_job *)calloc((size_t)nt, sizeof(attn_job));
  pthread_t *th = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
  if (!jobs || !th) { free(jobs); free(th); return 2; }
  for (int i = 0; i < nt; ++i) {
    jobs[i] = base;
    jobs[i].row_begin = rows * i / nt;
    jobs[i].row_end = rows * (i + 1) / nt;
  }
  for (int i = 1; i < nt; ++i) pthread_create(&th[i], NULL, attn_worker, &jobs[i]);
  attn_worker(&jobs[0]);
  int status = jobs[0].status;
  for (int i = 1; i < nt; ++i) {
    pthread_join(th[i], NULL);
    if (jobs[i].status && !status) status = jobs[i].status;
  }
  free(jobs);
  free(th);
  return status;
}

/* Softmax weights of one (b, h) row: w[t] for t < context_lens[b].  Exposed so
 * tests can check that they are a probability vector. */
int oracle_attention_weights(double *w, const uint16_t *q, const uint16_t *k_cache,
                             const int32_t *block_tables, const int32_t *context_lens,
                             int b, int h, int n_q, int n_kv, int d, int bs, int MB, int NB,
                             double scale) {
  attn_job J = {NULL, q, k_cache, k_cache, block_tables, context_lens, b + 1, n_q, n_kv, d,
                bs, MB, NB, scale, 0, 0, 0, 0};
  int G = n_q / n_kv, g = h / G, ctx = context_lens[b];
  if (ctx < 1 || ctx > MB * bs) return 1;
  const uint16_t *qrow = q + ((size_t)b * n_q + h) * d;
  double smax = -INFINITY;
  for (int t = 0; t < ctx; ++t) {
    int slot = 0;
    long r = token_tile(&J, b, g, t, &slot);
    if (r < 0) return 1;
    double acc = 0.0;
    for (int i = 0; i < d; ++i)
      acc += bf16_bits_to_double(qrow[i]) * bf16_bits_to_double(k_cache[r + tile_offset(slot, i, d)]);
    w[t] = scale * acc;
    if (w[t] > smax) smax = w[t];
  }
  double denom = 0.0;
  for (int t = 0; t < ctx; ++t) { w[t] = exp(w[t] - smax); denom += w[t]; }
  for (int t = 0; t < ctx; ++t) w[t] /= denom;
  return 0;
}

/* ------------------------------------------------------------------ */
/* sequence split + log-sum-exp merge                                  */
/* ------------------------------------------------------------------ */

/* Local attention of one (b, h) row over the token range [t0, t1): the
 * running state of the block update -- m = max score, l = sum exp(s - m),
 * o = sum exp(s - m) v (unnormalised).  An empty range gives m = -inf,
 * l = 0, o = 0. */
int oracle_attention_part(double *m_out, double *l_out, double *o_out, const uint16_t *q,
                          const uint16_t *k_cache, const uint16_t *v_cache,
                          const int32_t *block_tables, int b, int h, int t0, int t1,
                          int n_q, int n_kv, int d, int bs, int MB, int NB, double scale) {
  attn_job J = {NULL, q, k_cache, v_cache, block_tables, NULL, b + 1, n_q, n_kv, d,
                bs, MB, NB, scale, 0, 0, 0, 0};
  int G = n_q / n_kv, g = h / G;
  const uint16_t *qrow = q + ((size_t)b * n_q + h) * d;
  double m = -INFINITY, l = 0.0;
  for (int i = 0; i < d; ++i) o_out[i] = 0.0;
  if (t1 > t0) {
    for (int t = t0; t < t1; ++t) {
      int slot = 0;
      long r = token_tile(&J, b, g, t, &slot);
      if (r < 0) return 1;
      double acc = 0.0;
      for (int i = 0; i < d; ++i)
        acc += bf16_bits_to_double(qrow[i]) * bf16_bits_to_double(k_cache[r + tile_offset(slot, i, d)]);
      double s = scale * acc;
      if (s > m) m = s;
    }
    for (int t = t0; t < t1; ++t) {
      int slot = 0;
      long r = token_tile(&J, b, g, t, &slot);
      double acc = 0.0;
      for (int i = 0; i < d; ++i)
        acc += bf16_bits_to_double(qrow[i]) * bf16_bits_to_double(k_cache[r + tile_offset(slot, i, d)]);
      double p = exp(scale * acc - m);
      l += p;
      for (int i = 0; i < d; ++i) o_out[i] += p * bf16_bits_to_double(v_cache[r + tile_offset(slot, i, d)]);
    }
  }
  *m_out = m;
  *l_out = l;
  return 0;
}

/* Merge n_parts local states (m_i, l_i, o_i[d]) of one row into the
 * normalised output: M = max_i m_i, out = sum_i e^{m_i - M} o_i /
 * sum_i e^{m_i - M} l_i.  Parts with m_i = -inf (empty) contribute nothing.
 * Returns 1 if every part is empty. */
int oracle_lse_merge(double *out, const double *m, const double *l, const double *o,
                     int n_parts, int d) {
  double M = -INFINITY;
  for (int i = 0; i < n_parts; ++i)
    if (m[i] > M) M = m[i];
  if (M == -INFINITY) return 1;
  double L = 0.0;
  for (int k = 0; k < d; ++k) out[k] = 0.0;
  for (int i = 0; i < n_parts; ++i) {
    if (m[i] == -INFINITY) continue;
    double c = exp(m[i] - M);
    L += c * l[i];
    for (int k = 0; k < d; ++k) out[k] += c * o[(size_t)i * d + k];
  }
  for (int k = 0; k < d; ++k) out[k] /= L;
  return 0;
}
