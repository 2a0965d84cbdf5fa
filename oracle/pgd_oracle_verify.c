/*
 * pgd_oracle_verify.c -- the oracle for multi-query (speculative verify)
 * paged attention and for appending several tokens per sequence.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load or call this code.  It shares no code,
 * header, table or helper with the CUDA library (nor with the other oracle
 * files: each states its own formulas) and never reads anything the CUDA
 * library produced.
 *
 * Sources (page title, section):
 *  - "Module 10: inference and serving" (wrwei.github.io), section "Verify a
 *    chain, then roll back uncommitted state": the draft proposes gamma
 *    tokens; the target runs one forward over the last committed token and
 *    the proposals, each position scored on the proposed prefix before it;
 *    rejected positions are cut from the caches afterwards.  Lab 2 (toy
 *    decoder): t new positions are concatenated to the cached K/V and
 *    position i attends under the mask arange(k_len) <= old + i, with the
 *    default 1/sqrt(d_head) scale and KV head g repeated G times
 *    (repeat_interleave: query head h reads KV head floor(h / G)).
 *  - "The math of Transformer inference" (hs-black.github.io), section 10
 *    (speculative decoding, greedy version): one target forward over the
 *    prefix plus k proposed tokens gives the k + 1 positions' logits, and the
 *    output equals plain greedy decoding by the target.
 *  - "LLM inference systems engineering" (jasonzhang109.github.io), 2.1.3:
 *    verify_target(target_cache, [pending] + drafts) writes the provisional
 *    K/V; only the consumed prefix is kept.
 *  - Paged storage ("Module 10", "Mapping logical positions to physical
 *    blocks"; "Ch. 6 Inference efficiency and serving", 6.4): token t of
 *    sequence b lives in block table[b][t / bs], slot t % bs.
 *
 * Physical layout of the pool (the library's choice; the pages fix only the
 * logical shape and the block table): [NB][n_kv][tile], each tile bs x d
 * bf16 values as 8 x 8 core matrices, element (slot s, dim i) at
 * ((s / 8) * (d / 8) + i / 8) * 64 + (s % 8) * 8 + i % 8.
 *
 * Readings where the pages are silent (listed in the design notes):
 *  - q and out are [B][T][n_q][d]: T = gamma + 1 query tokens per sequence,
 *    the same T for every sequence of a call;
 *  - context_lens[b] counts the cached positions including the T new tokens,
 *    which are the last T positions: query token i sits at position
 *    context_lens[b] - T + i and sees positions 0 .. context_lens[b] - T + i;
 *  - new tokens are written at positions[b] + j, positions[b] being the
 *    number of positions cached before them.
 *
 * Arithmetic: bf16 inputs widened exactly to double; everything after in
 * double.  No blocking or reordering beyond the definitions.
 *
 * `mutation` plants a known mistake for the tests (0: the oracle as
 * defined): 1 no causal mask among the new tokens (every query sees the
 * whole context), 2 the mask shifted by one (query i sees one position
 * fewer), 3 query tokens in reverse order.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double widen_bf16(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Element offset of (slot s, dim i) inside one tile. */
static size_t elem_in_tile(int s, int i, int d) {
  return ((size_t)(s / 8) * (size_t)(d / 8) + (size_t)(i / 8)) * 64 + (size_t)(s % 8) * 8 +
         (size_t)(i % 8);
}

/* Append T tokens per sequence: token j of sequence b (k_new / v_new
 * [B][T][n_kv][d]) goes to logical position positions[b] + j, i.e. block
 * block_tables[b][pos / bs], slot pos % bs, for every KV head; a bit copy.
 * Returns 0, or 1 if a position or block id is out of range (that token is
 * skipped). */
int oracle_kv_append_tokens(uint16_t *k_cache, uint16_t *v_cache, const uint16_t *k_new,
                            const uint16_t *v_new, const int32_t *block_tables,
                            const int32_t *positions, int B, int T, int n_kv, int d, int bs,
                            int MB, int NB) {
  int status = 0;
  for (int b = 0; b < B; ++b) {
    for (int j = 0; j < T; ++j) {
      long pos = (long)positions[b] + j;
      if (pos < 0 || pos >= (long)MB * bs) { status = 1; continue; }
      int32_t blk = block_tables[(size_t)b * MB + pos / bs];
      if (blk < 0 || blk >= NB) { status = 1; continue; }
      int slot = (int)(pos % bs);
      for (int g = 0; g < n_kv; ++g) {
        size_t tile = ((size_t)blk * n_kv + g) * (size_t)bs * d;
        size_t src = (((size_t)b * T + j) * n_kv + g) * d;
        for (int i = 0; i < d; ++i) {
          k_cache[tile + elem_in_tile(slot, i, d)] = k_new[src + i];
          v_cache[tile + elem_in_tile(slot, i, d)] = v_new[src + i];
        }
      }
    }
  }
  return status;
}

typedef struct {
  double *out;           /* [B][T][n_q][d] */
  const uint16_t *q;     /* [B][T][n_q][d] */
  const uint16_t *k_cache, *v_cache;
  const int32_t *tables; /* [B][MB] */
  const int32_t *ctx;    /* [B] */
  int B, T, n_q, n_kv, d, bs, MB, NB;
  double scale;
  int mutation;
  long row_begin, row_end; /* rows (b, i, h) */
  int status;
} verify_job;

/* Tile offset of token t (sequence b, KV head g) and its slot; -1 for an
 * invalid block id. */
static long locate_token(const verify_job *J, int b, int g, int t, int *slot) {
  int32_t blk = J->tables[(size_t)b * J->MB + t / J->bs];
  if (blk < 0 || blk >= J->NB) return -1;
  *slot = t % J->bs;
  return (long)(((size_t)blk * J->n_kv + g) * (size_t)J->bs * J->d);
}

/* One (sequence b, query token i, query head h): the causal decode
 * definition over positions 0 .. ctx - T + i. */
static int verify_row(const verify_job *J, int b, int i, int h) {
  const int d = J->d, T = J->T;
  const int G = J->n_q / J->n_kv;
  const int g = h / G;
  const int ctx = J->ctx[b];
  if (ctx < T || ctx > J->MB * J->bs) return 1;
  int qi = (J->mutation == 3) ? T - 1 - i : i;
  int n_tok = ctx - T + i + 1;               /* mask: position <= old + i */
  if (J->mutation == 1) n_tok = ctx;
  if (J->mutation == 2) n_tok = ctx - T + i;
  if (n_tok < 1) n_tok = 1;
  const uint16_t *qrow = J->q + (((size_t)b * T + qi) * J->n_q + h) * d;
  double *orow = J->out + (((size_t)b * T + i) * J->n_q + h) * d;
  double *w = (double *)malloc(sizeof(double) * (size_t)n_tok);
  if (!w) return 2;
  double wmax = -INFINITY;
  for (int t = 0; t < n_tok; ++t) {
    int slot = 0;
    long r = locate_token(J, b, g, t, &slot);
    if (r < 0) { free(w); return 1; }
    double acc = 0.0;
    for (int c = 0; c < d; ++c)
      acc += widen_bf16(qrow[c]) * widen_bf16(J->k_cache[r + elem_in_tile(slot, c, d)]);
    w[t] = J->scale * acc;
    if (w[t] > wmax) wmax = w[t];
  }
  double den = 0.0;
  for (int t = 0; t < n_tok; ++t) {
    w[t] = exp(w[t] - wmax);
    den += w[t];
  }
  for (int c = 0; c < d; ++c) orow[c] = 0.0;
  for (int t = 0; t < n_tok; ++t) {
    int slot = 0;
    long r = locate_token(J, b, g, t, &slot);
    double wt = w[t] / den;
    for (int c = 0; c < d; ++c)
      orow[c] += wt * widen_bf16(J->v_cache[r + elem_in_tile(slot, c, d)]);
  }
  free(w);
  return 0;
}

static void *verify_worker(void *arg) {
  verify_job *J = (verify_job *)arg;
  for (long r = J->row_begin; r < J->row_end; ++r) {
    int h = (int)(r % J->n_q);
    long bi = r / J->n_q;
    int i = (int)(bi % J->T), b = (int)(bi / J->T);
    int st = verify_row(J, b, i, h);
    if (st && !J->status) J->status = st;
  }
  return NULL;
}

/* out[b][i][h][:] = sum_{t <= ctx_b - T + i} softmax_t(scale q[b][i][h] . k_t) v_t.
 * Returns 0, or 1 on an invalid context length or block id. */
int oracle_paged_verify_attention(double *out, const uint16_t *q, const uint16_t *k_cache,
                                  const uint16_t *v_cache, const int32_t *block_tables,
                                  const int32_t *context_lens, int B, int T, int n_q, int n_kv,
                                  int d, int bs, int MB, int NB, double scale, int n_threads,
                                  int mutation) {
  if (B < 0 || T < 1 || n_q <= 0 || n_kv <= 0 || n_q % n_kv || d <= 0 || d % 8 || bs <= 0 ||
      bs % 8 || MB <= 0 || NB <= 0)
    return 1;
  long rows = (long)B * T * n_q;
  if (rows == 0) return 0;
  if (n_threads <= 0) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    n_threads = n > 0 ? (int)n : 1;
  }
  if (n_threads > 256) n_threads = 256;
  if (rows < n_threads) n_threads = (int)rows;
  verify_job base = {out, q, k_cache, v_cache, block_tables, context_lens, B, T, n_q, n_kv, d,
                     bs, MB, NB, scale, mutation, 0, 0, 0};
  verify_job *jobs = (verify_job *)calloc((size_t)n_threads, sizeof(verify_job));
  pthread_t *th = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
  if (!jobs || !th) { free(jobs); free(th); return 2; }
  for (int k = 0; k < n_threads; ++k) {
    jobs[k] = base;
    jobs[k].row_begin = rows * k / n_threads;
    jobs[k].row_end = rows * (k + 1) / n_threads;
  }
  for (int k = 1; k < n_threads; ++k) pthread_create(&th[k], NULL, verify_worker, &jobs[k]);
  verify_worker(&jobs[0]);
  int status = jobs[0].status;
  for (int k = 1; k < n_threads; ++k) {
    pthread_join(th[k], NULL);
    if (jobs[k].status && !status) status = jobs[k].status;
  }
  free(jobs);
  free(th);
  return status;
}
