/*
 * pgd.h -- C ABI of libpgd: paged GQA decode attention and KV append on one
 * GB300 GPU (sm_103a).
 *
 * Terms (page title, section):
 *   B      sequences in the batch
 *   n_q    query heads; n_kv KV heads; G = n_q / n_kv query heads share one KV
 *          head, query head h reading KV head h / G ("Module 10: inference and
 *          serving", section "Deriving capacity from the configuration" and
 *          Lab 2's repeat_interleave; "The math of Transformer inference",
 *          section 5: MHA G = 1, MQA n_kv = 1, GQA in between)
 *   d      head width (d_head); this library supports d = 128
 *   bs     block size in tokens; a block holds bs consecutive positions of one
 *          sequence ("Module 10", section "Mapping logical positions to
 *          physical blocks"; "Ch. 6 Inference efficiency and serving", 6.4)
 *   NB     physical blocks in the pool; MB = width of a block-table row
 *
 * Layouts (all device memory unless marked host):
 *   k_cache, v_cache  bf16 pools of NB blocks: [NB][n_kv][tile], one tile per
 *                     (block, KV head), a contiguous bs*d*2-byte run holding
 *                     the bs tokens x d dims as 8 x 8 core matrices --
 *                     element (slot s, dim i) at ((s/8)*(d/8) + i/8)*64 +
 *                     (s%8)*8 + i%8, i.e. [bs/8][d/8][8][8].  The pages fix
 *                     only the logical shape (B, n_kv, T, d) and the block
 *                     table; this tiling lets one bulk copy per tile land
 *                     directly as a tensor-core operand.  bs must be a
 *                     multiple of 8.
 *   block_tables      int32 [B][MB]  logical block j of sequence b lives in
 *                     physical block block_tables[b][j]; entries past the
 *                     sequence's last block are never read
 *   context_lens      int32 [B]      cached positions of sequence b, counting
 *                     the token appended in this step
 *   q, out            bf16 [B][n_q][d]
 *   k_new, v_new      bf16 [B][n_kv][d]
 *
 * Conventions:
 *   - Ownership: the caller owns every buffer, including workspaces; no entry
 *     point here allocates device memory.  Pointers to bf16 arrays must be
 *     16-byte aligned; the workspace must be 256-byte aligned.
 *   - Asynchrony: GPU entry points only enqueue work on `stream` (a
 *     cudaStream_t passed as void*; NULL = the legacy default stream) and
 *     return.  Argument errors are detected on the host before any launch.
 *   - Device-side checks: kernels never read or write outside the pool.  A
 *     block id outside [0, NB), a context length outside [1, MB*bs] or an
 *     append position outside [0, MB*bs) skips the affected work and sets a
 *     bit in the per-device error word (pgd_device_errors); outputs of the
 *     affected sequences are then unspecified.
 *   - Threading: entry points are thread-safe except that one pgd_alloc
 *     handle must not be used from two threads at once.
 */
#ifndef PGD_H_
#define PGD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pgd_status {
  PGD_OK = 0,
  PGD_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size or shape */
  PGD_ERR_UNSUPPORTED = 2,   /* valid but not built: d != 128, bs, G, batch */
  PGD_ERR_OUT_OF_BLOCKS = 3, /* allocator: not enough free blocks; no change made */
  PGD_ERR_WORKSPACE = 4,     /* workspace missing, too small or misaligned */
  PGD_ERR_CUDA = 5,          /* a CUDA runtime call failed (see detail) */
  PGD_ERR_BLOCK_STATE = 6    /* allocator: block not held, double release, table gap */
} pgd_status;

/* Bits of the per-device error word written by the kernels. */
#define PGD_DEVERR_BAD_BLOCK_ID 1 /* a needed table entry was outside [0, NB) */
#define PGD_DEVERR_BAD_CONTEXT 2  /* a context length was < 1 or > MB*bs */
#define PGD_DEVERR_BAD_POSITION 4 /* a kv_append position was outside [0, MB*bs) */
#define PGD_DEVERR_TIMEOUT 8      /* a bounded wait inside a kernel gave up */

/* Largest batch one attention call accepts (larger batches: split the call). */
#define PGD_MAX_BATCH 2048

/* Static description of a status code.  Never NULL. */
const char *pgd_status_string(pgd_status s);

/* Detail of the last non-OK status returned on the calling thread ("" if
 * none).  Valid until the next call on that thread. */
const char *pgd_last_error_detail(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t pgd_version(void);

/* ---------------------------------------------------------------------- */
/* kv_append                                                              */
/* ---------------------------------------------------------------------- */
/* Write the new token of every sequence into its paged slot.  The decode
 * step forwards the pending token and commits its K/V to the cache, after
 * which the cache holds exactly the positions already forwarded ("LLM
 * inference systems engineering", 2.1.3 computation graph and generation
 * loop; "The math of Transformer inference", section 1, decode bullet; the
 * toy decoder of "Module 10", Lab 2, concatenates the new K/V before it
 * attends).
 *
 * For every b < B and KV head g < n_kv, with p = positions[b] (the number of
 * positions cached before this token):
 *     k_cache[block_tables[b][p / bs]][g][p % bs][:] = k_new[b][g][:]
 *     v_cache[...same slot...]                       = v_new[b][g][:]
 * A bit-for-bit copy.  positions is a device array [B].  The caller must not
 * append into a block that other sequences share (refcount > 1): take the
 * copy-on-write path first (pgd_alloc_append_slot + pgd_copy_blocks).
 * Returns PGD_OK after enqueueing; B == 0 is a no-op. */
pgd_status pgd_kv_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                         const int32_t *block_tables, const int32_t *positions, int32_t B,
                         int32_t n_kv, int32_t d, int32_t bs, int32_t MB, int32_t NB,
                         void *stream);

/* ---------------------------------------------------------------------- */
/* paged decode attention                                                 */
/* ---------------------------------------------------------------------- */
/* Single-query attention of every sequence over its own paged cache ("Module
 * 10", section "Attention reads a different cache per sequence"; "The math
 * of Transformer inference", section 4):
 *     out[b][h][:] = sum_t softmax_t(scale * q[b][h] . k_t) v_t,
 *     t in [0, context_lens[b]), k_t/v_t = KV head h / G of token t read
 *     through block_tables[b] at block t / bs, slot t % bs.
 * Only the valid positions of each sequence are read (section 9 of "The math
 * of Transformer inference": ragged reads).  Each K/V tile is read once per
 * (sequence, KV head) and serves all G query heads.  The context may be split
 * into parts whose (max, sum, weighted-sum) states are merged by log-sum-exp
 * ("The math of Transformer inference", section 8, sharding the KV cache
 * along the sequence; "LLM inference systems engineering", 2.8.3).
 * Arithmetic: bf16 inputs, fp32 accumulation, fp32 softmax, bf16 output
 * rounded to nearest even.
 *
 * num_splits: 0 = automatic: one CTA per SM; the kernel reads the context
 *   lengths and either gives each (sequence, KV head) to one CTA whole (when
 *   there are no more of them than CTAs and the longest is short enough to
 *   hide behind the total HBM traffic) or cuts all blocks into one part of
 *   (nearly) equal size per CTA;
 *   k > 0 = k * B * n_kv parts of (nearly) equal size in blocks, fixed.
 * workspace: device scratch of at least pgd_attention_workspace_size(...)
 *   bytes, 256-byte aligned, zero-filled before its first use (cudaMemset);
 *   every completed call leaves its counters at zero again, so one workspace
 *   can serve any number of calls in stream order.  Concurrent calls on
 *   different streams need separate workspaces.
 * Supported: d = 128, bs in {16, 32}, G in {1, 2, 4, 8}, 0 <= B <=
 * PGD_MAX_BATCH, B * MB < 2^31.  Returns PGD_OK after enqueueing. */
size_t pgd_attention_workspace_size(int32_t B, int32_t n_q, int32_t n_kv, int32_t d,
                                    int32_t num_splits);

pgd_status pgd_paged_decode_attention(void *out, const void *q, const void *k_cache,
                                      const void *v_cache, const int32_t *block_tables,
                                      const int32_t *context_lens, int32_t B, int32_t n_q,
                                      int32_t n_kv, int32_t d, int32_t bs, int32_t MB,
                                      int32_t NB, float scale, int32_t num_splits,
                                      void *workspace, size_t workspace_bytes, void *stream);

/* Number of CTAs one pgd_paged_decode_attention call launches with these
 * arguments on the current device when it runs the tensor-core kernel (0 on
 * invalid arguments); a call routed to the short-context kernel (see
 * pgd_set_short_context_tokens) launches 8 * B * n_kv. */
int32_t pgd_attention_grid(int32_t B, int32_t n_q, int32_t n_kv, int32_t bs, int32_t num_splits);

/* Size of the library's own device scratch array used by
 * pgd_paged_decode_attention_noalloc (16 MiB on every GPU that loads the
 * library, held until the process exits). */
#define PGD_NOALLOC_SCRATCH_BYTES (16u << 20)

/* pgd_paged_decode_attention for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point; it exists for callers
 * such as plugins or callbacks running inside another runtime's execution
 * step, which receive inputs and outputs but no scratch and must not call
 * cudaMalloc/cudaFree there (those calls can synchronize the device, fail
 * under the host runtime's memory budget, and compete with its allocator).
 * Same arguments, semantics and results as pgd_paged_decode_attention, minus
 * the workspace: the split-merge scratch lives in a fixed __device__ array of
 * PGD_NOALLOC_SCRATCH_BYTES inside the library.  Sizes whose workspace
 * (pgd_attention_workspace_size) exceeds that array are rejected with
 * PGD_ERR_WORKSPACE.  No device memory is allocated by this call.
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress); make that first call before any stream
 * capture.  Every call on a device shares the one array and leaves its
 * contents behind; the call clears the part that must start at zero (with
 * cudaMemsetAsync on `stream`) before launching.  Calls that overlap on the
 * same GPU -- on different streams, say -- race on the array and must be
 * serialised by the caller. */
pgd_status pgd_paged_decode_attention_noalloc(void *out, const void *q, const void *k_cache,
                                              const void *v_cache, const int32_t *block_tables,
                                              const int32_t *context_lens, int32_t B, int32_t n_q,
                                              int32_t n_kv, int32_t d, int32_t bs, int32_t MB,
                                              int32_t NB, float scale, int32_t num_splits,
                                              void *stream);

/* ---------------------------------------------------------------------- */
/* append, then attend (device buffers)                                   */
/* ---------------------------------------------------------------------- */
/* The decode step of one layer on device buffers: the new token's K/V
 * (k_new, v_new: bf16 [B][n_kv][d]) are written at position
 * context_lens[b] - 1 exactly as pgd_kv_append does ("LLM inference systems
 * engineering", 2.1.3: the step commits the pending token's K/V), then
 * out = pgd_paged_decode_attention over the updated caches.  Same shapes,
 * rules, results and errors as those two calls made one after the other;
 * every argument is checked before anything is enqueued.  The attention
 * kernel is launched with programmatic stream serialization and, knowing
 * that the kernel before it writes only the caches, runs its prologue (block
 * counts, split choice, Q and block-table loads) while kv_append runs and
 * waits for it only before its first cache read.  The block holding position
 * context_lens[b] - 1 must be private to sequence b (copy-on-write), as for
 * pgd_kv_append. */
pgd_status pgd_append_decode_attention(void *out, const void *q, const void *k_new,
                                       const void *v_new, void *k_cache, void *v_cache,
                                       const int32_t *block_tables, const int32_t *context_lens,
                                       int32_t B, int32_t n_q, int32_t n_kv, int32_t d, int32_t bs,
                                       int32_t MB, int32_t NB, float scale, int32_t num_splits,
                                       void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------- */
/* multi-query (speculative verify) attention                              */
/* ---------------------------------------------------------------------- */
/* A draft proposes gamma tokens; the target model scores the pending token
 * and the gamma proposals in one forward, each position conditioned on the
 * proposed prefix before it, and the caches are cut back to the committed
 * boundary afterwards ("Module 10", section "Verify a chain, then roll back
 * uncommitted state"; "The math of Transformer inference", section 10,
 * greedy version: one target forward over prefix + k tokens gives k + 1
 * positions' logits; "LLM inference systems engineering", 2.1.3, the
 * verify_target interface).  At the attention level of one layer that is T =
 * gamma + 1 query tokens per sequence over the paged cache with the causal
 * mask of "Module 10", Lab 2 (new position i sees every cached position up to
 * and including its own).
 *
 * pgd_kv_append_tokens: write T new tokens per sequence, k_new / v_new bf16
 * [B][T][n_kv][d], token j at position positions[b] + j (positions: device
 * int32 [B], the number of positions cached before them); otherwise exactly
 * pgd_kv_append (bit-for-bit, same layout, same rules on shared blocks).
 * Rolling back rejected tokens needs no device work: the caller lowers the
 * sequence's length (and may release blocks past it); slots past a context
 * length are never read.
 *
 * pgd_paged_verify_attention: for every b < B, query token i < T, query head
 * h < n_q, with c = context_lens[b] (which counts the T new tokens, already
 * appended: c >= T, else PGD_DEVERR_BAD_CONTEXT) and g = h / (n_q / n_kv):
 *     out[b][i][h][:] = sum_{t <= c - T + i} softmax_t(scale * q[b][i][h] . k_t) v_t
 * with k_t, v_t the cached K/V of token t of sequence b, KV head g (as in
 * pgd_paged_decode_attention, which is the case T = 1).  q and out: bf16
 * [B][T][n_q][d].  T * (n_q / n_kv) <= 16 (the query rows served per KV
 * head and pass over the cache), else PGD_ERR_UNSUPPORTED; bf16 pools only.
 * Same arithmetic, tolerance, workspace rules and errors as
 * pgd_paged_decode_attention; workspace: pgd_verify_workspace_size(...) bytes.
 * Each KV tile is read once per call for all T x G query rows of its head. */
pgd_status pgd_kv_append_tokens(const void *k_new, const void *v_new, void *k_cache,
                                void *v_cache, const int32_t *block_tables,
                                const int32_t *positions, int32_t B, int32_t T, int32_t n_kv,
                                int32_t d, int32_t bs, int32_t MB, int32_t NB, void *stream);
size_t pgd_verify_workspace_size(int32_t B, int32_t T, int32_t n_q, int32_t n_kv, int32_t d,
                                 int32_t num_splits);
pgd_status pgd_paged_verify_attention(void *out, const void *q, const void *k_cache,
                                      const void *v_cache, const int32_t *block_tables,
                                      const int32_t *context_lens, int32_t B, int32_t T,
                                      int32_t n_q, int32_t n_kv, int32_t d, int32_t bs,
                                      int32_t MB, int32_t NB, float scale, int32_t num_splits,
                                      void *workspace, size_t workspace_bytes, void *stream);

/* pgd_append_verify_attention: one verify step in one call -- the T new
 * tokens of every sequence appended at positions context_lens[b] - T + j
 * (pgd_kv_append_tokens with positions = context_lens - T), then
 * pgd_paged_verify_attention over the updated caches; the attention's CTAs
 * run their prologue while the append runs.  Same arguments, layouts, rules
 * and errors as those two calls; every argument is checked before the first
 * launch.
 *
 * pgd_verify_step: the same step for a caller whose per-step tensors live in
 * host memory -- q_h, k_new_h, v_new_h, context_lens_h in, out_h out -- with
 * the handling of pgd_decode_step: page-locked host buffers that the device
 * addresses (16-byte aligned) are read and written in place by the kernels
 * over the host link, any other goes through its device buffer (q_d,
 * k_new_d, v_new_d, context_lens_d, out_d) and a copy (inputs all read in
 * place must hold the step's values when the call is made, as there);
 * everything is enqueued on `stream`, and the host buffers must stay
 * untouched until the stream has completed the step.  The cache, block
 * tables and workspace stay on the device. */
pgd_status pgd_append_verify_attention(void *out, const void *q, const void *k_new,
                                       const void *v_new, void *k_cache, void *v_cache,
                                       const int32_t *block_tables, const int32_t *context_lens,
                                       int32_t B, int32_t T, int32_t n_q, int32_t n_kv, int32_t d,
                                       int32_t bs, int32_t MB, int32_t NB, float scale,
                                       int32_t num_splits, void *workspace,
                                       size_t workspace_bytes, void *stream);
pgd_status pgd_verify_step(void *out_h, const void *q_h, const void *k_new_h, const void *v_new_h,
                           const int32_t *context_lens_h, void *out_d, void *q_d, void *k_new_d,
                           void *v_new_d, int32_t *context_lens_d, void *k_cache, void *v_cache,
                           const int32_t *block_tables, int32_t B, int32_t T, int32_t n_q,
                           int32_t n_kv, int32_t d, int32_t bs, int32_t MB, int32_t NB,
                           float scale, int32_t num_splits, void *workspace,
                           size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------- */
/* MLA latent cache (multi-head latent attention, absorbed form)           */
/* ---------------------------------------------------------------------- */
/* A latent cache stores, per layer and token, the latent c_t (d_c = 512) and
 * a decoupled RoPE key k_t^R (d_r = 64): 576 values shared by every head
 * ("The math of Transformer inference", MLA section; "LLM inference systems
 * engineering", 2.4.2).  With W^UK absorbed into the query and W^UV into the
 * output projection (same book, 2.8.2), decode attention of head h is
 *     s_t = scale * q[b][h] . c_t       (all 576 values; q = [W_h^{UK T} q_h^C ; q_h^R])
 *     out[b][h][j] = sum_t softmax(s)_t c_t[j]     (j < 512, t < context_lens[b])
 * -- MQA with every head reading the one cache.
 *
 * Latent pool: bf16 [NB][bs/8][72][8][8] (block tiles of bs x 576 values as
 * 8 x 8 core matrices: element (slot s, value i) at
 * ((s / 8) * 72 + i / 8) * 64 + (s % 8) * 8 + i % 8); bs in {16, 32, 64};
 * block tables and context lengths as for the GQA cache.  q: bf16 [B][H][576];
 * out: bf16 [B][H][512].  d must be 576 and dv 512 (else UNSUPPORTED).
 * pgd_mla_append writes c_new[b] (bf16 [B][576]) at position positions[b]
 * (bit exact).  pgd_mla_decode_attention: fp32 scores and softmax, bf16
 * probabilities and latent values on the tensor cores, fp32 accumulation,
 * bf16 output; num_splits = parts of each context (0 = automatic); with more
 * than one part it needs pgd_mla_workspace_size(B, H, num_splits) bytes of
 * 256-byte-aligned workspace (no zeroing needed), else workspace may be NULL.
 * Device errors as for pgd_paged_decode_attention. */
size_t pgd_mla_workspace_size(int32_t B, int32_t H, int32_t num_splits);
pgd_status pgd_mla_append(const void *c_new, void *cache, const int32_t *block_tables,
                          const int32_t *positions, int32_t B, int32_t d, int32_t bs, int32_t MB,
                          int32_t NB, void *stream);
pgd_status pgd_mla_decode_attention(void *out, const void *q, const void *cache,
                                    const int32_t *block_tables, const int32_t *context_lens,
                                    int32_t B, int32_t H, int32_t d, int32_t dv, int32_t bs,
                                    int32_t MB, int32_t NB, float scale, int32_t num_splits,
                                    void *workspace, size_t workspace_bytes, void *stream);
/* The decode step of one layer over a latent cache: c_new[b] (bf16 [B][576])
 * written at position context_lens[b] - 1 exactly as pgd_mla_append does,
 * then pgd_mla_decode_attention over the updated cache -- the same shapes,
 * rules, results and errors as those two calls one after the other, every
 * argument checked before anything is enqueued.  The attention kernel knows
 * that the kernel before it writes only the cache: its prologue (queries,
 * tensor memory, barriers) runs while the append does, and only its copies
 * wait for it. */
pgd_status pgd_mla_append_decode_attention(void *out, const void *q, const void *c_new,
                                           void *cache, const int32_t *block_tables,
                                           const int32_t *context_lens, int32_t B, int32_t H,
                                           int32_t d, int32_t dv, int32_t bs, int32_t MB,
                                           int32_t NB, float scale, int32_t num_splits,
                                           void *workspace, size_t workspace_bytes,
                                           void *stream);

/* pgd_mla_step: pgd_mla_append_decode_attention for a caller whose per-step
 * tensors live in host memory -- q_h (bf16 [B][H][576]), c_new_h (bf16
 * [B][576]), context_lens_h in, out_h (bf16 [B][H][512]) out.  q_h is always
 * copied to q_d (every context part of a head group reads it); c_new_h,
 * context_lens_h and out_h, when page-locked host memory that the device
 * addresses, are read and written in place by the kernels over the host
 * link, otherwise through c_new_d, context_lens_d, out_d and a copy each.
 * Everything is enqueued on `stream`; the host buffers must stay untouched
 * until the stream has completed the step.  The cache, tables and workspace
 * stay on the device; arguments and errors as for the device-buffer call. */
pgd_status pgd_mla_step(void *out_h, const void *q_h, const void *c_new_h,
                        const int32_t *context_lens_h, void *out_d, void *q_d, void *c_new_d,
                        int32_t *context_lens_d, void *cache, const int32_t *block_tables,
                        int32_t B, int32_t H, int32_t d, int32_t dv, int32_t bs, int32_t MB,
                        int32_t NB, float scale, int32_t num_splits, void *workspace,
                        size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------- */
/* cascade: shared prefixes read once per group                            */
/* ---------------------------------------------------------------------- */
/* pgd_paged_decode_attention for a batch in which groups of sequences share
 * their leading blocks ("Module 10", section "Share only identical state":
 * sequences point at the same read-only prefix blocks; same page: sharing
 * the storage does not by itself share the traffic).  Same definition,
 * arguments, rules and result; the work is split in two passes merged by
 * log-sum-exp ("The math of Transformer inference", section 8; "LLM
 * inference systems engineering", 2.8.3):
 *   1. for each group and KV head, each shared prefix tile is read once and
 *      multiplied against all of the group's query rows together on the
 *      tensor cores (up to 128 rows = sequences x G per pass; larger groups
 *      take several), giving a partial state per (sequence, query head);
 *   2. each sequence's own suffix is attended as pgd_paged_decode_attention
 *      does, giving partial states too;
 *   3. a combine kernel merges both passes' partial states of every
 *      (sequence, query head) into the output.
 * Groups (device int32 arrays of n_groups entries): sequences
 * group_first[i] .. group_first[i] + group_size[i] - 1 (consecutive; a
 * sequence in at most one group) share their first group_blocks[i] block
 * table entries (the same physical block ids, read from the table of
 * group_first[i]).  seq_prefix_blocks (device int32 [B]) gives each
 * sequence's shared block count: group_blocks of its group, or 0.  Every
 * sequence must keep at least one block after its shared ones
 * (context_lens[b] > seq_prefix_blocks[b] * bs; else PGD_DEVERR_BAD_CONTEXT).
 * max_group_size and max_group_blocks are host upper bounds of group_size
 * and group_blocks (they size the grid and the workspace).  workspace: at
 * least pgd_cascade_workspace_size(...) bytes, 256-byte aligned, zero-filled
 * before first use.  bf16 pools only.  Three kernels on `stream`: the
 * shared-prefix pass runs on about a quarter of the SMs and lets the suffix
 * pass start at once on the others (with num_splits = 0 the suffix pass's
 * grid shrinks by the prefix pass's CTAs); the suffix pass completes only
 * after the prefix pass, and the combine kernel waits for both. */
size_t pgd_cascade_workspace_size(int32_t B, int32_t n_q, int32_t n_kv, int32_t d, int32_t bs,
                                  int32_t num_splits, int32_t max_group_size,
                                  int32_t max_group_blocks);
pgd_status pgd_cascade_decode_attention(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, const int32_t *seq_prefix_blocks,
    const int32_t *group_first, const int32_t *group_size, const int32_t *group_blocks,
    int32_t n_groups, int32_t max_group_size, int32_t max_group_blocks, int32_t B, int32_t n_q,
    int32_t n_kv, int32_t d, int32_t bs, int32_t MB, int32_t NB, float scale, int32_t num_splits,
    void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------- */
/* 8-bit KV cache: FP8 E4M3 codes with one fp32 scale per (token, head)    */
/* ---------------------------------------------------------------------- */
/* Storing the cache in 8 bits halves its memory and the bytes a decode step
 * reads ("Module 10", section "Quantize the cache, evaluate the final
 * artifact"; "The math of Transformer inference", section 11: KV in int8 /
 * fp8, scales per head and per token, dequantisation fused into the kernel).
 *
 * Pool layout (k_cache, v_cache; the library's choice): uint8
 * [NB][n_kv][bs/8][1056] -- each (block, KV head) tile is bs/8 groups of 8
 * tokens; a group holds the 8 tokens' E4M3 codes (1024 bytes: code of group
 * slot r, dim i at (i / 16) * 128 + r * 16 + i % 16) followed by their 8
 * fp32 scales (byte 1024 + 4 r).  Token t of a sequence is code row
 * t % bs of block block_tables[b][t / bs]; its value is E4M3(code) * scale.
 * The pool must be 16-byte aligned.
 *
 * Quantisation (pgd_kv_append_fp8; "Ch. 6 Inference efficiency and
 * serving", 6.6.1: symmetric, scale from the largest absolute value, never a
 * zero scale): for each (sequence, KV head) row x of d = 128 bf16 values,
 * scale = max_i |x_i| / 448 (1 when that max is 0) and code_i =
 * E4M3(x_i / scale), both divisions IEEE binary32, the E4M3 conversion
 * rounding to nearest even and saturating to +-448 (OCP E4M3: no
 * infinities; S.1111.111 is NaN).  Same arguments, checks and errors as
 * pgd_kv_append. */
pgd_status pgd_kv_append_fp8(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                             const int32_t *block_tables, const int32_t *positions, int32_t B,
                             int32_t n_kv, int32_t d, int32_t bs, int32_t MB, int32_t NB,
                             void *stream);

/* pgd_paged_decode_attention over an 8-bit pool: the same definition applied
 * to the dequantised K and V, the same arguments (k_cache, v_cache as
 * above), checks, errors and workspace (pgd_attention_workspace_size).
 * Arithmetic: q.k^T on the tensor cores in E4M3 with each query head split
 * into a high and a low E4M3 part after scaling by a power of two -- the
 * bf16 query itself, except that elements more than 2^9 below the head's
 * largest keep an absolute error under 2^-17 of that largest -- the key and
 * query scales applied in fp32; V dequantised to f16 (code times the scale
 * rounded to f16) and probabilities in f16 for the p.v; fp32 softmax and
 * accumulation; bf16 output.  The query must be finite and the dequantised
 * V values within the f16 range (|v| < 65504). */
pgd_status pgd_paged_decode_attention_fp8(void *out, const void *q, const void *k_cache,
                                          const void *v_cache, const int32_t *block_tables,
                                          const int32_t *context_lens, int32_t B, int32_t n_q,
                                          int32_t n_kv, int32_t d, int32_t bs, int32_t MB,
                                          int32_t NB, float scale, int32_t num_splits,
                                          void *workspace, size_t workspace_bytes, void *stream);

/* pgd_append_decode_attention for an 8-bit pool: pgd_kv_append_fp8 at
 * position context_lens[b] - 1, then pgd_paged_decode_attention_fp8, with the
 * same overlap of the attention prologue and the append. */
pgd_status pgd_append_decode_attention_fp8(void *out, const void *q, const void *k_new,
                                           const void *v_new, void *k_cache, void *v_cache,
                                           const int32_t *block_tables,
                                           const int32_t *context_lens, int32_t B, int32_t n_q,
                                           int32_t n_kv, int32_t d, int32_t bs, int32_t MB,
                                           int32_t NB, float scale, int32_t num_splits,
                                           void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------- */
/* one decode step with host inputs and outputs                            */
/* ---------------------------------------------------------------------- */
/* One decode step of one layer for a caller whose per-step tensors live in
 * host memory: pgd_append_decode_attention (append at position
 * context_lens[b] - 1, then attention) on q_h, k_new_h, v_new_h and
 * context_lens_h, with the result in out_h -- all enqueued on `stream`.
 * q_h, k_new_h, v_new_h, context_lens_h and out_h, when page-locked host
 * memory that the device addresses (as the CUDA runtime reports it) and
 * 16-byte aligned, are read and written in place by the kernels over the host
 * link; otherwise they go through the caller's device buffers (q_d, k_new_d,
 * v_new_d, context_lens_d, out_d) and a copy each.  A copy breaks the chain
 * of kernels that start while their predecessor finishes, so in-place buffers
 * save about 5 us a step.  When all four inputs are read in place, the
 * kernels may read them before earlier work in the stream has finished: they
 * must hold the step's values when the call is made (not be filled by work
 * enqueued before it).  The host buffers must stay untouched until the
 * stream has completed the step.
 * The cache, block tables and workspace stay on the device.  Shapes and rules
 * as above. */
pgd_status pgd_decode_step(void *out_h, const void *q_h, const void *k_new_h, const void *v_new_h,
                           const int32_t *context_lens_h, void *out_d, void *q_d, void *k_new_d,
                           void *v_new_d, int32_t *context_lens_d, void *k_cache, void *v_cache,
                           const int32_t *block_tables, int32_t B, int32_t n_q, int32_t n_kv,
                           int32_t d, int32_t bs, int32_t MB, int32_t NB, float scale,
                           int32_t num_splits, void *workspace, size_t workspace_bytes,
                           void *stream);

/* pgd_decode_step for an 8-bit pool: the same handling of the host buffers
 * around pgd_append_decode_attention_fp8. */
pgd_status pgd_decode_step_fp8(void *out_h, const void *q_h, const void *k_new_h,
                               const void *v_new_h, const int32_t *context_lens_h, void *out_d,
                               void *q_d, void *k_new_d, void *v_new_d, int32_t *context_lens_d,
                               void *k_cache, void *v_cache, const int32_t *block_tables,
                               int32_t B, int32_t n_q, int32_t n_kv, int32_t d, int32_t bs,
                               int32_t MB, int32_t NB, float scale, int32_t num_splits,
                               void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------- */
/* copy-on-write block copy                                               */
/* ---------------------------------------------------------------------- */
/* For i < n: copy physical block src_ids[i] to dst_ids[i] (all KV heads, all
 * bs slots, K and V).  The device half of copy-on-write: a sequence that must
 * write into a block other sequences share first gets a private copy ("Module
 * 10", section "Share only identical state"; "Ch. 6", 6.4).  src_ids and
 * dst_ids are device arrays; a pair with an id outside [0, NB) is skipped and
 * flagged.  Source and destination blocks must not overlap. */
pgd_status pgd_copy_blocks(void *k_cache, void *v_cache, const int32_t *src_ids,
                           const int32_t *dst_ids, int32_t n, int32_t n_kv, int32_t d,
                           int32_t bs, int32_t NB, void *stream);

/* ---------------------------------------------------------------------- */
/* measurement: read-only streaming bandwidth                              */
/* ---------------------------------------------------------------------- */
/* One pass that reads every byte of src[0 .. bytes) once from device memory
 * and discards it: the bandwidth a kernel that only reads can reach on this
 * GPU, to be timed in the same job as the attention kernels so that their
 * fractions of the HBM roofline have a denominator of their own kind beside
 * a copy's ("LLM inference systems engineering", 3.8.2: keep peak and
 * sustained bandwidth apart and calibrate on the access pattern measured).
 *   mode 0  16-byte vector loads by a grid of four 512-thread CTAs per SM;
 *           bytes a multiple of 16.
 *   mode 1  the attention kernels' pattern: one CTA per SM streams its share
 *           as 4 KiB bulk copies (TMA engine) into a three-stage ring of
 *           64 KiB shared-memory stages; bytes a multiple of 4096.
 * src is a device pointer, 16-byte aligned, owned by the caller and left
 * unchanged.  Returns PGD_ERR_INVALID_ARG for another mode, a null or
 * misaligned src or a size that is not a multiple of the mode's unit (0 bytes
 * is a no-op); a wait that gives up sets PGD_DEVERR_TIMEOUT.  Only enqueues
 * on `stream`.  Not part of the attention path. */
pgd_status pgd_read_stream(const void *src, size_t bytes, int32_t mode, void *stream);

/* ---------------------------------------------------------------------- */
/* wait limit of the kernels' bounded waits (for tests of the exit path)  */
/* ---------------------------------------------------------------------- */
/* Every wait of a kernel's role on another role of its CTA (an mbarrier
 * phase) gives up after a limit; the kernel then sets PGD_DEVERR_TIMEOUT,
 * stops issuing copies and MMAs, lets every role run to the end of its walk
 * with its remaining waits returning at once, waits (with the fixed 4 s
 * limit) for the copies already in flight, frees its tensor memory and
 * exits; its outputs are then unspecified, the caller's workspace counters
 * are left at zero and the next call runs normally.  The limit is 4 s
 * (4e9 ns); pgd_set_wait_limit_ns sets it, process-wide, for the launches
 * made after the call (0 restores 4 s) -- a short limit makes the waits run
 * out on purpose, which is what a test of that exit path needs; nothing else
 * should change it.  Thread-safe; pgd_wait_limit_ns returns the value in
 * force.  No counterpart on the pages. */
void pgd_set_wait_limit_ns(uint64_t ns);
uint64_t pgd_wait_limit_ns(void);

/* ---------------------------------------------------------------------- */
/* short-context path                                                     */
/* ---------------------------------------------------------------------- */
/* A single-query call with num_splits = 0 of pgd_paged_decode_attention,
 * pgd_append_decode_attention, pgd_decode_step, their 8-bit counterparts
 * (_fp8), pgd_paged_decode_attention_noalloc or pgd_cascade_decode_attention
 * without groups, whose every possible context is short -- MB * bs at most
 * the limit below, itself at most 1024 -- with at most 64 (sequence, KV head)
 * units and B * n_kv * MB * bs at most 40960, runs a latency-first kernel
 * instead of the tensor-core one: such a call is bound by the start-up of a
 * kernel, not by its bytes.  One cluster of 8 CTAs per unit, each taking an
 * eighth of the context; q.k and p.v on the CUDA cores in fp32 (8-bit codes
 * times their scales), exact exp2; the eight (max, sum, output) states merged
 * by log-sum-exp through distributed shared memory ("The math of Transformer
 * inference", section 8); for the append variants the new token's K/V are
 * written by the same launch, bit for bit as pgd_kv_append (pgd_kv_append_fp8)
 * writes them.  The results, errors and rules are those of the documented
 * calls; the workspace is checked but not touched.  The limit is 1024 tokens;
 * pgd_set_short_context_tokens sets it process-wide for the calls made after
 * it (0 sends every call to the tensor-core kernel, a negative value restores
 * 1024) and returns the previous limit; pgd_short_path returns 1 when a call
 * with these sizes would run the short-context kernel now, else 0.
 * Thread-safe.  No counterpart on the pages: a choice between two kernels for
 * the same operation. */
int32_t pgd_set_short_context_tokens(int32_t max_tokens);
int32_t pgd_short_path(int32_t B, int32_t n_kv, int32_t bs, int32_t MB, int32_t num_splits);

/* ---------------------------------------------------------------------- */
/* device error word                                                      */
/* ---------------------------------------------------------------------- */
/* Wait for `stream`, then read the current device's error word (PGD_DEVERR_*
 * bits accumulated by every kernel of this library on that device) into
 * *flags; clear it when `clear` is nonzero. */
pgd_status pgd_device_errors(int32_t *flags, int32_t clear, void *stream);

/* ---------------------------------------------------------------------- */
/* host block allocator (host memory only)                                */
/* ---------------------------------------------------------------------- */
/* A pool of num_blocks physical block ids with a reference count each
 * ("Module 10", sections "Mapping logical positions to physical blocks" and
 * "Share only identical state"; "Ch. 6", 6.4; "The math of Transformer
 * inference", section 9, PagedAttention: reference counts and copy-on-write).
 * Ids are allocated on demand, one block when a sequence grows past a block
 * boundary, so a sequence wastes at most bs - 1 slots. */
typedef struct pgd_alloc pgd_alloc;

/* Create a pool of num_blocks (> 0) free blocks. */
pgd_status pgd_alloc_create(int32_t num_blocks, pgd_alloc **out);
/* Destroy a pool (NULL is a no-op). */
void pgd_alloc_destroy(pgd_alloc *a);
/* Take n free ids (count 1 each) into ids_out[n]; all or nothing
 * (PGD_ERR_OUT_OF_BLOCKS leaves the pool unchanged). */
pgd_status pgd_alloc_allocate(pgd_alloc *a, int32_t n, int32_t *ids_out);
/* Add one reference to each of ids[n] (each must be held). */
pgd_status pgd_alloc_share(pgd_alloc *a, const int32_t *ids, int32_t n);
/* Drop one reference from each of ids[n]; an id whose count reaches 0 is
 * free again.  Checked first, applied only if every drop is valid. */
pgd_status pgd_alloc_release(pgd_alloc *a, const int32_t *ids, int32_t n);
/* Reference count of id (0 = free), or -1 if id is outside the pool. */
int32_t pgd_alloc_refcount(const pgd_alloc *a, int32_t id);
int32_t pgd_alloc_num_free(const pgd_alloc *a);
int32_t pgd_alloc_num_blocks(const pgd_alloc *a);
/* Make the slot of logical position pos writable in one table row (host
 * int32 [MB], -1 = unassigned).  If pos opens a block that the row lacks,
 * allocate it.  If the block holding pos is shared (count > 1), copy on
 * write: allocate a private block, point the row at it, drop one reference to
 * the old block, and return the pair in *cow_src / *cow_dst for the caller to
 * copy on the device (pgd_copy_blocks) before appending.  Otherwise both are
 * -1.  On PGD_ERR_OUT_OF_BLOCKS nothing changes. */
pgd_status pgd_alloc_append_slot(pgd_alloc *a, int32_t *table_row, int32_t MB, int32_t bs,
                                 int32_t pos, int32_t *cow_src, int32_t *cow_dst);
/* Fork: make dst_row (host int32 [MB]) share every block that holds one of
 * the first n_tokens tokens of src_row (a reference each, the partial last
 * block included; its first write takes the copy-on-write path). */
pgd_status pgd_alloc_fork(pgd_alloc *a, const int32_t *src_row, int32_t n_tokens, int32_t bs,
                          int32_t *dst_row, int32_t MB);

/* Host-side check of host copies of block tables and context lengths: every
 * length in [1, MB*bs] and every needed entry in [0, NB).  Returns
 * PGD_ERR_INVALID_ARG with a detail naming the first offender. */
pgd_status pgd_validate_tables(const int32_t *block_tables_h, const int32_t *context_lens_h,
                               int32_t B, int32_t MB, int32_t NB, int32_t bs);

#ifdef __cplusplus
}
#endif

#endif /* PGD_H_ */
