/*
 * pgd_oracle_mla.c -- the oracle for decode attention over an MLA latent
 * cache (multi-head latent attention, the absorbed form).
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load or call this code.  It shares no code,
 * header, table or helper with the CUDA library and never reads anything the
 * CUDA library produced.
 *
 * Sources (page title, section):
 *  - "The math of Transformer inference" (hs-black.github.io), section on
 *    MLA ("store one low-rank latent vector"): per layer and token the cache
 *    holds the latent c_t^KV (d_c = 512) and a decoupled RoPE key k_t^R
 *    (d_h^R = 64), 576 elements shared by all n_h = 128 heads; W^UK is
 *    absorbed into the query (each head's query mapped into the 512-d latent
 *    space and dotted with the cached latent), the RoPE part adds the dot
 *    product of the head's RoPE query with k_t^R, and W^UV is absorbed into
 *    the output projection, so attention returns a 512-d latent output per
 *    head; after absorption decode is MQA with G = n_h.
 *  - "LLM inference systems engineering" (jasonzhang109.github.io), 2.8.2:
 *    q_j^T W_j^K c_t = (W_j^{K T} q_j)^T c_t and sum_t a_t W_j^V c_t =
 *    W_j^V sum_t a_t c_t -- the identities behind the absorbed form; 2.4.2:
 *    (d_c + d_r) elements per layer and token.
 *  - Paged storage as for the decode oracle ("Module 10", "Mapping logical
 *    positions to physical blocks"): token t of sequence b lives in block
 *    table[b][t / bs], slot t % bs.
 *
 * Definition, for sequence b and head h, with D = d_c + d_r cached values
 * per token and the first Dv = d_c of them the latent:
 *     s_t = scale * sum_{i < D} q[b][h][i] * c_t[i]        (t < ctx_b)
 *     out[b][h][j] = sum_t softmax(s)_t * c_t[j]           (j < Dv)
 * q[b][h] is the absorbed query [W_h^{UK T} q_h^C ; q_h^R].
 *
 * Pool layout (the library's choice): [NB][tile], one tile of bs x D bf16 per
 * block as 8 x 8 core matrices, element (slot s, dim i) at
 * ((s / 8) * (D / 8) + i / 8) * 64 + (s % 8) * 8 + i % 8.
 *
 * Arithmetic: bf16 widened exactly to double, then double throughout.
 * `mutation` (tests only): 1 the RoPE part left out of the score, 2 the value
 * read from the last Dv cached dims, 3 no scale.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

static double mla_widen(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static size_t mla_elem(int s, int i, int D) {
  return ((size_t)(s / 8) * (size_t)(D / 8) + (size_t)(i / 8)) * 64 + (size_t)(s % 8) * 8 +
         (size_t)(i % 8);
}

/* Write the new token's cached row c_new[b][0 .. D) at position
 * positions[b] (block table[b][p / bs], slot p % bs).  A bit copy.  Returns 0,
 * or 1 if a position or block id is out of range (that row is skipped). */
int oracle_mla_append(uint16_t *cache, const uint16_t *c_new, const int32_t *block_tables,
                      const int32_t *positions, int B, int D, int bs, int MB, int NB) {
  int status = 0;
  for (int b = 0; b < B; ++b) {
    long p = positions[b];
    if (p < 0 || p >= (long)MB * bs) { status = 1; continue; }
    int32_t blk = block_tables[(size_t)b * MB + p / bs];
    if (blk < 0 || blk >= NB) { status = 1; continue; }
    size_t tile = (size_t)blk * (size_t)bs * D;
    for (int i = 0; i < D; ++i)
      cache[tile + mla_elem((int)(p % bs), i, D)] = c_new[(size_t)b * D + i];
  }
  return status;
}

typedef struct {
  double *out;
  const uint16_t *q, *cache;
  const int32_t *tables, *ctx;
  int B, H, D, Dv, bs, MB, NB;
  double scale;
  int mutation;
  long row_begin, row_end;
  int status;
} mla_job;

static int mla_row(const mla_job *J, int b, int h) {
  const int D = J->D, Dv = J->Dv;
  int ctx = J->ctx[b];
  if (ctx < 1 || ctx > J->MB * J->bs) return 1;
  const uint16_t *qr = J->q + ((size_t)b * J->H + h) * D;
  double *orow = J->out + ((size_t)b * J->H + h) * Dv;
  double *w = (double *)malloc(sizeof(double) * (size_t)ctx);
  if (!w) return 2;
  const int n_dot = (J->mutation == 1) ? Dv : D;
  const double scale = (J->mutation == 3) ? 1.0 : J->scale;
  const int v0 = (J->mutation == 2) ? D - Dv : 0;
  double wmax = -INFINITY;
  for (int t = 0; t < ctx; ++t) {
    int32_t blk = J->tables[(size_t)b * J->MB + t / J->bs];
    if (blk < 0 || blk >= J->NB) { free(w); return 1; }
    size_t tile = (size_t)blk * (size_t)J->bs * D;
    double acc = 0.0;
    for (int i = 0; i < n_dot; ++i)
      acc += mla_widen(qr[i]) * mla_widen(J->cache[tile + mla_elem(t % J->bs, i, D)]);
    w[t] = scale * acc;
    if (w[t] > wmax) wmax = w[t];
  }
  double den = 0.0;
  for (int t = 0; t < ctx; ++t) {
    w[t] = exp(w[t] - wmax);
    den += w[t];
  }
  for (int j = 0; j < Dv; ++j) orow[j] = 0.0;
  for (int t = 0; t < ctx; ++t) {
    int32_t blk = J->tables[(size_t)b * J->MB + t / J->bs];
    size_t tile = (size_t)blk * (size_t)J->bs * D;
    double a = w[t] / den;
    for (int j = 0; j < Dv; ++j)
      orow[j] += a * mla_widen(J->cache[tile + mla_elem(t % J->bs, v0 + j, D)]);
  }
  free(w);
  return 0;
}

static void *mla_worker(void *arg) {
  mla_job *J = (mla_job *)arg;
  for (long r = J->row_begin; r < J->row_end; ++r) {
    int st = mla_row(J, (int)(r / J->H), (int)(r % J->H));
    if (st && !J->status) J->status = st;
  }
  return NULL;
}

/* out[B][H][Dv] of latent decode attention (definition above).  Returns 0,
 * or 1 on an invalid argument, context length or block id. */
int oracle_mla_attention(double *out, const uint16_t *q, const uint16_t *cache,
                         const int32_t *block_tables, const int32_t *context_lens, int B, int H,
                         int D, int Dv, int bs, int MB, int NB, double scale, int n_threads,
                         int mutation) {
  if (B < 0 || H <= 0 || D <= 0 || D % 8 || Dv <= 0 || Dv > D || bs <= 0 || bs % 8 || MB <= 0 ||
      NB <= 0)
    return 1;
  long rows = (long)B * H;
  if (rows == 0) return 0;
  if (n_threads <= 0) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    n_threads = n > 0 ? (int)n : 1;
  }
  if (n_threads > 256) n_threads = 256;
  if (rows < n_threads) n_threads = (int)rows;
  mla_job base = {out, q, cache, block_tables, context_lens, B, H, D, Dv, bs, MB, NB,
                  scale, mutation, 0, 0, 0};
  mla_job *jobs = (mla_job *)calloc((size_t)n_threads, sizeof(mla_job));
  pthread_t *th = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
  if (!jobs || !th) { free(jobs); free(th); return 2; }
  for (int k = 0; k < n_threads; ++k) {
    jobs[k] = base;
    jobs[k].row_begin = rows * k / n_threads;
    jobs[k].row_end = rows * (k + 1) / n_threads;
  }
  for (int k = 1; k < n_threads; ++k) pthread_create(&th[k], NULL, mla_worker, &jobs[k]);
  mla_worker(&jobs[0]);
  int status = jobs[0].status;
  for (int k = 1; k < n_threads; ++k) {
    pthread_join(th[k], NULL);
    if (jobs[k].status && !status) status = jobs[k].status;
  }
  free(jobs);
  free(th);
  return status;
}
