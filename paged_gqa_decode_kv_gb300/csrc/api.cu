// api.cu -- the C ABI declared in include/pgd.h: argument checks on the host,
// workspace layout, kernel launches, the host-buffer decode step and the
// per-device error word.
#include <cuda_runtime.h>

#include <math.h>
#include <stdarg.h>
#include <stdio.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <atomic>

#include "pgd_device.cuh"
#include "short_attention.cuh"

namespace pgd {
int attention_ctas_per_sm(int G, int bs, int B);
cudaError_t attention_launch(const AttnParams &p, int G, int bs, int grid, cudaStream_t stream);
int attention_ctas_per_sm_fp8(int G, int bs, int B);
cudaError_t attention_launch_fp8(const AttnParams &p, int G, int bs, int grid,
                                 cudaStream_t stream);
cudaError_t prefix_attention_launch(const PrefixParams &p, int G, int bs, int grid,
                                    cudaStream_t stream);
cudaError_t cascade_combine_launch(const CombineParams &p, int G, cudaStream_t stream);
cudaError_t mla_attention_launch(const MlaParams &p, cudaStream_t stream);
cudaError_t mla_append_launch(const void *c_new, void *cache, const int32_t *tables,
                              const int32_t *pos, int pos_offset, int B, int bs, int MB, int NB,
                              int32_t *err, cudaStream_t stream);
int mla_heads_per_cta();
cudaError_t kv_append_fp8_launch(const void *k_new, const void *v_new, void *k_cache,
                                 void *v_cache, const int32_t *tables, const int32_t *pos,
                                 int pos_offset, int B, int n_kv, int bs, int MB, int NB,
                                 int32_t *err, cudaStream_t stream);
cudaError_t kv_append_launch(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                             const int32_t *tables, const int32_t *pos, int pos_offset, int B,
                             int T, int n_kv, int bs, int MB, int NB, int32_t *err,
                             cudaStream_t stream);
cudaError_t copy_blocks_launch(void *k_cache, void *v_cache, const int32_t *src_ids,
                               const int32_t *dst_ids, int n, int n_kv, int bs, int NB,
                               int32_t *err, cudaStream_t stream);
cudaError_t read_stream_launch(const void *src, size_t bytes, int mode, int32_t *err,
                               cudaStream_t stream);
void set_error_detail(const char *msg);
void clear_error_detail();
const char *error_detail();
}  // namespace pgd

using namespace pgd;

namespace {

constexpr int kMaxDevices = 64;
// Automatic grids never exceed this many CTAs, so a workspace sized for it
// serves every device.
constexpr int kAutoMaxCtas = 2048;
constexpr size_t kWsAlign = 256;

pgd_status fail(pgd_status s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  set_error_detail(buf);
  return s;
}

pgd_status ok() {
  clear_error_detail();
  return PGD_OK;
}

// Wait limit handed to every launch (0: the kernels' default); set only by
// pgd_set_wait_limit_ns, for tests of the timeout exit.
std::atomic<unsigned long long> g_wait_limit_ns{0};

// Largest MB * bs routed to the short-context kernel (pgd_set_short_context_tokens).
std::atomic<int> g_short_tokens{1024};

pgd_status cuda_fail(cudaError_t e, const char *what) {
  return fail(PGD_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// The per-device error word lives in this translation unit; its device
// address is looked up once per device.
__device__ int32_t g_device_error_word;

std::mutex g_mu;
int32_t *g_err_ptr[kMaxDevices] = {};

pgd_status error_word(int32_t **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PGD_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    g_err_ptr[dev] = static_cast<int32_t *>(p);
  }
  *out = g_err_ptr[dev];
  return PGD_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool supported_group(int G) { return G == 1 || G == 2 || G == 4 || G == 8; }
bool supported_bs(int bs) { return bs == 16 || bs == 32; }

pgd_status check_cache_shape(int32_t n_kv, int32_t d, int32_t bs, int32_t MB, int32_t NB) {
  if (n_kv <= 0 || MB <= 0 || NB <= 0 || bs <= 0)
    return fail(PGD_ERR_INVALID_ARG, "n_kv, bs, MB and NB must be positive");
  if (d != kHeadDim) return fail(PGD_ERR_UNSUPPORTED, "d = %d (only 128 is built)", d);
  if (!supported_bs(bs)) return fail(PGD_ERR_UNSUPPORTED, "block size %d (16 or 32)", bs);
  if ((long long)MB * bs > 0x7fffffffLL)
    return fail(PGD_ERR_INVALID_ARG, "MB * bs overflows int32");
  return PGD_OK;
}

struct WsLayout {
  size_t counters, part_ml, part_o, total;
  long long slots;
};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace: [B*n_kv] int32 per-unit arrival counters, then per partial slot
// (max, sum) and o[G][128].  A slot is unit + part (one part per CTA), so
// slots = units + CTAs.
// Kernel row count for T query tokens of Gh heads each: the next power of
// two of T * Gh, or 0 past 16 rows.
int unit_rows(int T, int Gh) {
  const int r = T * Gh;
  if (T < 1 || r > 16) return 0;
  int g = 1;
  while (g < r) g <<= 1;
  return g;
}

WsLayout ws_layout(int32_t B, int32_t n_q, int32_t n_kv, long long grid) {
  WsLayout L;
  const int G = n_q / n_kv;
  const long long units = (long long)B * n_kv;
  L.slots = units + grid;
  L.counters = 0;
  L.part_ml = round_up((size_t)units * 4, kWsAlign);
  L.part_o = L.part_ml + round_up((size_t)L.slots * G * 2 * 4, kWsAlign);
  L.total = L.part_o + (size_t)L.slots * G * kHeadDim * 4;
  return L;
}

std::map<std::tuple<int, int, int, int, int>, int> g_occ;

pgd_status auto_grid(int G, int bs, int B, int *grid, bool fp8 = false) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  const int bucket = (B + 255) / 256;
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_tuple(dev, G, bs, bucket, fp8 ? 1 : 0);
  auto it = g_occ.find(key);
  if (it == g_occ.end()) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    int per_sm = fp8 ? attention_ctas_per_sm_fp8(G, bs, bucket * 256)
                     : attention_ctas_per_sm(G, bs, bucket * 256);
    if (per_sm <= 0) return fail(PGD_ERR_CUDA, "occupancy query failed for G=%d bs=%d", G, bs);
    long long g = (long long)sms * per_sm;
    if (g > kAutoMaxCtas) g = kAutoMaxCtas;
    it = g_occ.emplace(key, (int)g).first;
  }
  *grid = it->second;
  return PGD_OK;
}

pgd_status check_attention_args(const void *out, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *tables, const int32_t *ctx,
                                 int32_t B, int32_t n_q, int32_t n_kv, int32_t d, int32_t bs,
                                 int32_t MB, int32_t NB, float scale, int32_t num_splits) {
  if (B < 0) return fail(PGD_ERR_INVALID_ARG, "B = %d", B);
  if (B > PGD_MAX_BATCH) return fail(PGD_ERR_UNSUPPORTED, "B = %d > %d", B, PGD_MAX_BATCH);
  pgd_status s = check_cache_shape(n_kv, d, bs, MB, NB);
  if (s != PGD_OK) return s;
  if (n_q <= 0 || n_q % n_kv) return fail(PGD_ERR_INVALID_ARG, "n_q %% n_kv != 0");
  if (!supported_group(n_q / n_kv))
    return fail(PGD_ERR_UNSUPPORTED, "group size G = %d (1, 2, 4 or 8)", n_q / n_kv);
  if ((long long)B * MB >= 0x7fffffffLL) return fail(PGD_ERR_INVALID_ARG, "B * MB >= 2^31");
  if (!(scale > 0.f) || !isfinite(scale)) return fail(PGD_ERR_INVALID_ARG, "scale must be > 0");
  if (num_splits < 0) return fail(PGD_ERR_INVALID_ARG, "num_splits < 0");
  if (num_splits > 0 && (long long)num_splits * B * n_kv > (1LL << 30))
    return fail(PGD_ERR_INVALID_ARG, "num_splits too large");
  if (B == 0) return PGD_OK;
  if (!out || !q || !k_cache || !v_cache || !tables || !ctx)
    return fail(PGD_ERR_INVALID_ARG, "null pointer");
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return fail(PGD_ERR_INVALID_ARG, "bf16 arrays must be 16-byte aligned");
  if (!aligned(tables, 4) || !aligned(ctx, 4))
    return fail(PGD_ERR_INVALID_ARG, "int32 arrays must be 4-byte aligned");
  return PGD_OK;
}

// Host-side half of an attention launch: workspace checks, grid and the
// kernel's parameter block.  Nothing is enqueued.
struct PreparedAttention {
  AttnParams p;
  int G, bs, grid;
  bool fp8;
};

pgd_status prepare_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *tables, const int32_t *ctx, int32_t B, int32_t n_q,
                             int32_t n_kv, int32_t bs, int32_t MB, int32_t NB, float scale,
                             int32_t num_splits, void *workspace, size_t workspace_bytes,
                             PreparedAttention *pa, bool fp8 = false, int32_t T = 1) {
  if (!workspace) return fail(PGD_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(workspace, kWsAlign)) return fail(PGD_ERR_WORKSPACE, "workspace not 256-aligned");
  // query rows per unit: T tokens x the KV head's query heads, padded to a
  // power of two (the kernel's row count)
  const int Gh = n_q / n_kv;
  const int G = unit_rows(T, Gh);
  if (G == 0 || (fp8 && T != 1))
    return fail(PGD_ERR_UNSUPPORTED, "T = %d x %d heads per KV head (at most 16 rows)", T, Gh);
  const int32_t n_rows = G * n_kv;
  if (workspace_bytes < ws_layout(B, n_rows, n_kv, 1).total)
    return fail(PGD_ERR_WORKSPACE, "workspace %zu bytes is too small", workspace_bytes);
  int grid = 0;
  if (num_splits > 0) {
    grid = (int)((long long)num_splits * B * n_kv);
  } else {
    pgd_status s = auto_grid(G, bs, B, &grid, fp8);
    if (s != PGD_OK) return s;
  }
  const WsLayout L = ws_layout(B, n_rows, n_kv, grid);
  if (workspace_bytes < L.total)
    return fail(PGD_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, L.total);
  int32_t *err = nullptr;
  pgd_status s = error_word(&err);
  if (s != PGD_OK) return s;
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  AttnParams p;
  p.out = static_cast<__nv_bfloat16 *>(out);
  p.q = static_cast<const __nv_bfloat16 *>(q);
  p.k_cache = static_cast<const unsigned char *>(k_cache);
  p.v_cache = static_cast<const unsigned char *>(v_cache);
  p.tables = tables;
  p.ctx = ctx;
  p.B = B;
  p.n_q = n_q;
  p.n_kv = n_kv;
  p.MB = MB;
  p.NB = NB;
  p.T = T;
  p.lg_gh = Gh == 1 ? 0 : Gh == 2 ? 1 : Gh == 4 ? 2 : 3;
  p.rows = T * Gh;
  p.qk_scale_log2 = (float)((double)scale * 1.4426950408889634);  // scale * log2(e)
  p.counters = reinterpret_cast<int32_t *>(ws + L.counters);
  p.auto_split = num_splits == 0 ? 1 : 0;
  p.prefetch_units = (num_splits == 0 && (long long)B * n_kv <= grid) ? 1 : 0;
  p.part_ml = reinterpret_cast<float *>(ws + L.part_ml);
  p.part_o = reinterpret_cast<float *>(ws + L.part_o);
  p.err = err;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.wait_late = 0;
  p.seq_prefix_blocks = nullptr;
  p.pre_ml = nullptr;
  p.pre_o = nullptr;
  p.n_tsplit = 0;
  p.part_info = nullptr;
  pa->p = p;
  pa->G = G;
  pa->bs = bs;
  pa->grid = grid;
  pa->fp8 = fp8;
  return PGD_OK;
}

// Whether an automatic single-query call goes to the short-context kernel:
// every context it can hold (MB * bs tokens) is within the limit, and its
// (sequence, KV head) units and units x tokens are small enough for the
// latency-first kernel to win (short_attention.cu gives the measurements).
bool short_rule(long long B, long long n_kv, long long MB, long long bs, int32_t num_splits,
                int T) {
  const long long units = B * n_kv, tokens = MB * bs;
  return T == 1 && num_splits == 0 && units >= 1 && units <= short_max_units() &&
         tokens <= std::min(g_short_tokens.load(), short_max_tokens()) &&
         units * tokens <= short_max_work();
}

bool short_path(const PreparedAttention &pa, int32_t num_splits, int32_t MB, int32_t bs) {
  return short_rule(pa.p.B, pa.p.n_kv, MB, bs, num_splits, pa.p.T);
}

// The short-context kernel on a prepared call's arguments; with k_new and
// v_new it appends the new token first, in the same launch.
pgd_status launch_short(const PreparedAttention &pa, const void *k_new, const void *v_new,
                        void *k_cache, void *v_cache, cudaStream_t stream, bool early = false) {
  ShortParams sp;
  sp.out = pa.p.out;
  sp.q = pa.p.q;
  sp.k_cache = static_cast<unsigned char *>(k_cache);
  sp.v_cache = static_cast<unsigned char *>(v_cache);
  sp.k_new = static_cast<const __nv_bfloat16 *>(k_new);
  sp.v_new = static_cast<const __nv_bfloat16 *>(v_new);
  sp.tables = pa.p.tables;
  sp.ctx = pa.p.ctx;
  sp.B = pa.p.B;
  sp.n_q = pa.p.n_q;
  sp.n_kv = pa.p.n_kv;
  sp.MB = pa.p.MB;
  sp.NB = pa.p.NB;
  sp.qk_scale_log2 = pa.p.qk_scale_log2;
  sp.fp8 = pa.fp8 ? 1 : 0;
  sp.early = early ? 1 : 0;
  sp.err = pa.p.err;
  cudaError_t e = short_attention_launch(sp, pa.G, pa.bs, stream);
  if (e != cudaSuccess) return cuda_fail(e, "short-context attention launch");
  return PGD_OK;
}

pgd_status launch_prepared(const PreparedAttention &pa, cudaStream_t stream) {
  cudaError_t e = pa.fp8 ? attention_launch_fp8(pa.p, pa.G, pa.bs, pa.grid, stream)
                         : attention_launch(pa.p, pa.G, pa.bs, pa.grid, stream);
  if (e != cudaSuccess) return cuda_fail(e, "paged attention launch");
  return PGD_OK;
}

pgd_status launch_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *tables, const int32_t *ctx, int32_t B, int32_t n_q,
                            int32_t n_kv, int32_t bs, int32_t MB, int32_t NB, float scale,
                            int32_t num_splits, void *workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
  PreparedAttention pa;
  pgd_status s = prepare_attention(out, q, k_cache, v_cache, tables, ctx, B, n_q, n_kv, bs, MB,
                                   NB, scale, num_splits, workspace, workspace_bytes, &pa);
  if (s != PGD_OK) return s;
  if (short_path(pa, num_splits, MB, bs))
    return launch_short(pa, nullptr, nullptr, const_cast<void *>(k_cache),
                        const_cast<void *>(v_cache), stream);
  return launch_prepared(pa, stream);
}

// kv_append at position context_lens[b] - 1, then attention over the updated
// caches.  Every check runs before the first launch.  The attention kernel
// is told that the kernel before it (kv_append) writes only the caches, so
// its CTAs run their prologue while kv_append runs and wait only before the
// first cache read.  `early`: q, k_new, v_new and ctx are caller memory that
// no kernel of the stream writes (page-locked host buffers), which the
// short-context kernel may read before the previous kernel has completed.
pgd_status append_then_attend(void *out, const void *q, const void *k_new, const void *v_new,
                              void *k_cache, void *v_cache, const int32_t *tables,
                              const int32_t *ctx, int32_t B, int32_t n_q, int32_t n_kv,
                              int32_t bs, int32_t MB, int32_t NB, float scale, int32_t num_splits,
                              void *workspace, size_t workspace_bytes, cudaStream_t stream,
                              bool fp8 = false, bool early = false) {
  if (!k_new || !v_new) return fail(PGD_ERR_INVALID_ARG, "null pointer");
  if (!aligned(k_new, 16) || !aligned(v_new, 16))
    return fail(PGD_ERR_INVALID_ARG, "bf16 arrays must be 16-byte aligned");
  PreparedAttention pa;
  pgd_status s = prepare_attention(out, q, k_cache, v_cache, tables, ctx, B, n_q, n_kv, bs, MB,
                                   NB, scale, num_splits, workspace, workspace_bytes, &pa, fp8);
  if (s != PGD_OK) return s;
  if (short_path(pa, num_splits, MB, bs))  // one launch: the append is fused
    return launch_short(pa, k_new, v_new, k_cache, v_cache, stream, early);
  // (The append kernels read their inputs only after waiting for the kernel
  // before them and then let the attention launch, so that it never starts
  // before earlier work that may write what its prologue reads: the tables.)
  cudaError_t e = fp8 ? kv_append_fp8_launch(k_new, v_new, k_cache, v_cache, tables, ctx, -1, B,
                                             n_kv, bs, MB, NB, pa.p.err, stream)
                      : kv_append_launch(k_new, v_new, k_cache, v_cache, tables, ctx, -1, B, 1,
                                         n_kv, bs, MB, NB, pa.p.err, stream);
  if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
  pa.p.wait_late = 1;
  return launch_prepared(pa, stream);
}

// Cascade plan: the shared-prefix pass cuts each group's sequences into
// chunks of 128 / G and each group's prefix into n_tsplit parts (at most 16,
// at least one 128-token stage each), so that it takes about a quarter of the
// SMs -- one CTA each -- beside the suffix pass on the rest.
struct CascadePlan {
  int n_tsplit, n_rchunk;
  size_t pre_ml, pre_o, part_info, total;  // byte offsets / size past the decode workspace
};
constexpr int kPrefixSmShare = 4;

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

CascadePlan cascade_plan(int32_t B, int32_t n_q, int32_t n_kv, int32_t bs, int32_t n_groups,
                         int32_t max_group_size, int32_t max_group_blocks, size_t decode_bytes,
                         int sms) {
  CascadePlan c;
  const int G = n_q / n_kv;
  const long long stages = std::max(1LL, ((long long)max_group_blocks * bs + 127) / 128);
  c.n_rchunk = std::max(1, (max_group_size * G + 127) / 128);
  const long long items = std::max(1LL, (long long)std::max(n_groups, 1) * n_kv * c.n_rchunk);
  const long long want = std::max(1LL, (long long)sms / kPrefixSmShare);
  c.n_tsplit = (int)std::max(1LL, std::min({16LL, stages, (want + items - 1) / items}));
  const size_t rows = (size_t)B * n_q * c.n_tsplit;
  c.pre_ml = round_up(decode_bytes, kWsAlign);
  c.pre_o = c.pre_ml + round_up(rows * 2 * 4, kWsAlign);
  c.part_info = c.pre_o + round_up(rows * kHeadDim * 4, kWsAlign);
  c.total = c.part_info + (size_t)B * n_kv * 8;
  return c;
}

}  // namespace

namespace pgd {
// Entry for other translation units of the library: the same checks and
// launch as pgd_paged_decode_attention, with the scratch supplied by the
// caller, and the scratch size the call needs.
pgd_status paged_attention_with_scratch(void *out, const void *q, const void *k_cache,
                                        const void *v_cache, const int32_t *tables,
                                        const int32_t *ctx, int32_t B, int32_t n_q, int32_t n_kv,
                                        int32_t d, int32_t bs, int32_t MB, int32_t NB,
                                        float scale, int32_t num_splits, void *scratch,
                                        size_t scratch_bytes, cudaStream_t stream) {
  pgd_status s = check_attention_args(out, q, k_cache, v_cache, tables, ctx, B, n_q, n_kv, d, bs,
                                      MB, NB, scale, num_splits);
  if (s != PGD_OK || B == 0) return s;
  return launch_attention(out, q, k_cache, v_cache, tables, ctx, B, n_q, n_kv, bs, MB, NB, scale,
                          num_splits, scratch, scratch_bytes, stream);
}

// The argument checks of pgd_paged_decode_attention alone (nothing is
// enqueued), for entry points that must reject a call before they touch
// any device memory.
pgd_status attention_args_status(const void *out, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *tables, const int32_t *ctx,
                                 int32_t B, int32_t n_q, int32_t n_kv, int32_t d, int32_t bs,
                                 int32_t MB, int32_t NB, float scale, int32_t num_splits) {
  return check_attention_args(out, q, k_cache, v_cache, tables, ctx, B, n_q, n_kv, d, bs, MB, NB,
                              scale, num_splits);
}

pgd_status set_status_detail(pgd_status s, const char *msg) {
  set_error_detail(msg);
  return s;
}
}  // namespace pgd

extern "C" {

const char *pgd_status_string(pgd_status s) {
  switch (s) {
    case PGD_OK: return "ok";
    case PGD_ERR_INVALID_ARG: return "invalid argument";
    case PGD_ERR_UNSUPPORTED: return "unsupported configuration";
    case PGD_ERR_OUT_OF_BLOCKS: return "out of blocks";
    case PGD_ERR_WORKSPACE: return "workspace missing or too small";
    case PGD_ERR_CUDA: return "CUDA error";
    case PGD_ERR_BLOCK_STATE: return "invalid block state";
  }
  return "unknown status";
}

const char *pgd_last_error_detail(void) { return error_detail(); }

int32_t pgd_version(void) { return 100; }

pgd_status pgd_kv_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                         const int32_t *block_tables, const int32_t *positions, int32_t B,
                         int32_t n_kv, int32_t d, int32_t bs, int32_t MB, int32_t NB,
                         void *stream) {
  if (B < 0) return fail(PGD_ERR_INVALID_ARG, "B = %d", B);
  pgd_status s = check_cache_shape(n_kv, d, bs, MB, NB);
  if (s != PGD_OK) return s;
  if ((long long)B * n_kv > 0x7fffffffLL) return fail(PGD_ERR_INVALID_ARG, "B * n_kv too large");
  if (B == 0) return ok();
  if (!k_new || !v_new || !k_cache || !v_cache || !block_tables || !positions)
    return fail(PGD_ERR_INVALID_ARG, "null pointer");
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return fail(PGD_ERR_INVALID_ARG, "bf16 arrays must be 16-byte aligned");
  int32_t *err = nullptr;
  s = error_word(&err);
  if (s != PGD_OK) return s;
  cudaError_t e = kv_append_launch(k_new, v_new, k_cache, v_cache, block_tables, positions, 0, B,
                                   1, n_kv, bs, MB, NB, err, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
  return ok();
}

pgd_status pgd_kv_append_tokens(const void *k_new, const void *v_new, void *k_cache,
                                void *v_cache, const int32_t *block_tables,
                                const int32_t *positions, int32_t B, int32_t T, int32_t n_kv,
                                int32_t d, int32_t bs, int32_t MB, int32_t NB, void *stream) {
  if (B < 0 || T < 1) return fail(PGD_ERR_INVALID_ARG, "B = %d, T = %d", B, T);
  pgd_status s = check_cache_shape(n_kv, d, bs, MB, NB);
  if (s != PGD_OK) return s;
  if ((long long)B * T * n_kv > 0x7ffffffcLL)
    return fail(PGD_ERR_INVALID_ARG, "B * T * n_kv too large");
  if (B == 0) return ok();
  if (!k_new || !v_new || !k_cache || !v_cache || !block_tables || !positions)
    return fail(PGD_ERR_INVALID_ARG, "null pointer");
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return fail(PGD_ERR_INVALID_ARG, "bf16 arrays must be 16-byte aligned");
  int32_t *err = nullptr;
  s = error_word(&err);
  if (s != PGD_OK) return s;
  cudaError_t e = kv_append_launch(k_new, v_new, k_cache, v_cache, block_tables, positions, 0, B,
                                   T, n_kv, bs, MB, NB, err, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
  return ok();
}

size_t pgd_attention_workspace_size(int32_t B, int32_t n_q, int32_t n_kv, int32_t d,
                                    int32_t num_splits) {
  if (B < 0 || n_kv <= 0 || n_q <= 0 || n_q % n_kv || d != kHeadDim || num_splits < 0) return 0;
  long long grid = 0;
  if (num_splits > 0) {
    grid = (long long)num_splits * B * n_kv;
  } else {
    // the automatic grid of the current device (both block sizes), or the
    // largest automatic grid when no device is usable
    grid = kAutoMaxCtas;
    const int G = n_q / n_kv;
    int g[4] = {0, 0, 0, 0};
    if (supported_group(G) && auto_grid(G, 16, B, &g[0]) == PGD_OK &&
        auto_grid(G, 32, B, &g[1]) == PGD_OK && auto_grid(G, 16, B, &g[2], true) == PGD_OK &&
        auto_grid(G, 32, B, &g[3], true) == PGD_OK)
      grid = std::max(std::max(g[0], g[1]), std::max(g[2], g[3]));
    clear_error_detail();
  }
  return ws_layout(B, n_q, n_kv, grid).total;
}

int32_t pgd_attention_grid(int32_t B, int32_t n_q, int32_t n_kv, int32_t bs, int32_t num_splits) {
  if (B <= 0 || n_kv <= 0 || n_q <= 0 || n_q % n_kv || num_splits < 0) return 0;
  if (!supported_group(n_q / n_kv) || !supported_bs(bs)) return 0;
  if (num_splits > 0) return (int32_t)((long long)num_splits * B * n_kv);
  int grid = 0;
  if (auto_grid(n_q / n_kv, bs, B, &grid) != PGD_OK) return 0;
  return grid;
}

// Checks of a verify call (T new tokens per sequence) beyond those of a
// decode call.
static pgd_status check_verify(int32_t B, int32_t T, int32_t n_q, int32_t n_kv) {
  if (T < 1) return fail(PGD_ERR_INVALID_ARG, "T = %d", T);
  if (unit_rows(T, n_q / n_kv) == 0)
    return fail(PGD_ERR_UNSUPPORTED, "T * (n_q / n_kv) = %d > 16 query rows per KV head",
                T * (n_q / n_kv));
  if ((long long)B * T * n_q >= 0x7fffffffLL) return fail(PGD_ERR_INVALID_ARG, "B * T * n_q");
  return PGD_OK;
}

size_t pgd_verify_workspace_size(int32_t B, int32_t T, int32_t n_q, int32_t n_kv, int32_t d,
                                 int32_t num_splits) {
  if (B < 0 || n_kv <= 0 || n_q <= 0 || n_q % n_kv || d != kHeadDim || num_splits < 0) return 0;
  const int Gh = n_q / n_kv;
  if (!supported_group(Gh)) return 0;
  const int G = unit_rows(T, Gh);
  if (G == 0) return 0;
  long long grid = 0;
  if (num_splits > 0) {
    grid = (long long)num_splits * B * n_kv;
  } else {
    grid = kAutoMaxCtas;
    int g[2] = {0, 0};
    if (auto_grid(G, 16, B, &g[0]) == PGD_OK && auto_grid(G, 32, B, &g[1]) == PGD_OK)
      grid = std::max(g[0], g[1]);
    clear_error_detail();
  }
  return ws_layout(B, G * n_kv, n_kv, grid).total;
}

pgd_status pgd_paged_verify_attention(void *out, const void *q, const void *k_cache,
                                      const void *v_cache, const int32_t *block_tables,
                                      const int32_t *context_lens, int32_t B, int32_t T,
                                      int32_t n_q, int32_t n_kv, int32_t d, int32_t bs,
                                      int32_t MB, int32_t NB, float scale, int32_t num_splits,
                                      void *workspace, size_t workspace_bytes, void *stream) {
  pgd_status s = check_attention_args(out, q, k_cache, v_cache, block_tables, context_lens, B,
                                      n_q, n_kv, d, bs, MB, NB, scale, num_splits);
  if (s != PGD_OK) return s;
  if ((s = check_verify(B, T, n_q, n_kv)) != PGD_OK) return s;
  if (B == 0) return ok();
  PreparedAttention pa;
  s = prepare_attention(out, q, k_cache, v_cache, block_tables, context_lens, B, n_q, n_kv, bs, MB,
                        NB, scale, num_splits, workspace, workspace_bytes, &pa, false, T);
  if (s != PGD_OK) return s;
  s = launch_prepared(pa, static_cast<cudaStream_t>(stream));
  return s == PGD_OK ? ok() : s;
}

// kv_append of the T new tokens at context_lens[b] - T + j, then the verify
// attention over the updated caches, told (as in append_then_attend) that
// the kernel before it writes only the caches.  Every check runs before the
// first launch.
static pgd_status append_then_verify(void *out, const void *q, const void *k_new,
                                     const void *v_new, void *k_cache, void *v_cache,
                                     const int32_t *tables, const int32_t *ctx, int32_t B,
                                     int32_t T, int32_t n_q, int32_t n_kv, int32_t bs, int32_t MB,
                                     int32_t NB, float scale, int32_t num_splits, void *workspace,
                                     size_t workspace_bytes, cudaStream_t stream) {
  if (!k_new || !v_new) return fail(PGD_ERR_INVALID_ARG, "null pointer");
  if (!aligned(k_new, 16) || !aligned(v_new, 16))
    return fail(PGD_ERR_INVALID_ARG, "bf16 arrays must be 16-byte aligned");
  if ((long long)B * T * n_kv > 0x7ffffffcLL)
    return fail(PGD_ERR_INVALID_ARG, "B * T * n_kv too large");
  PreparedAttention pa;
  pgd_status s = prepare_attention(out, q, k_cache, v_cache, tables, ctx, B, n_q, n_kv, bs, MB,
                                   NB, scale, num_splits, workspace, workspace_bytes, &pa, false,
                                   T);
  if (s != PGD_OK) return s;
  cudaError_t e = kv_append_launch(k_new, v_new, k_cache, v_cache, tables, ctx, -T, B, T, n_kv,
                                   bs, MB, NB, pa.p.err, stream);
  if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
  pa.p.wait_late = 1;
  return launch_prepared(pa, stream);
}

pgd_status pgd_append_verify_attention(void *out, const void *q, const void *k_new,
                                       const void *v_new, void *k_cache, void *v_cache,
                                       const int32_t *block_tables, const int32_t *context_lens,
                                       int32_t B, int32_t T, int32_t n_q, int32_t n_kv, int32_t d,
                                       int32_t bs, int32_t MB, int32_t NB, float scale,
                                       int32_t num_splits, void *workspace,
                                       size_t workspace_bytes, void *stream) {
  pgd_status s = check_attention_args(out, q, k_cache, v_cache, block_tables, context_lens, B,
                                      n_q, n_kv, d, bs, MB, NB, scale, num_splits);
  if (s != PGD_OK) return s;
  if ((s = check_verify(B, T, n_q, n_kv)) != PGD_OK) return s;
  if (B == 0) return ok();
  s = append_then_verify(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, B, T,
                         n_q, n_kv, bs, MB, NB, scale, num_splits, workspace, workspace_bytes,
                         static_cast<cudaStream_t>(stream));
  return s == PGD_OK ? ok() : s;
}

pgd_status pgd_paged_decode_attention(void *out, const void *q, const void *k_cache,
                                      const void *v_cache, const int32_t *block_tables,
                                      const int32_t *context_lens, int32_t B, int32_t n_q,
                                      int32_t n_kv, int32_t d, int32_t bs, int32_t MB,
                                      int32_t NB, float scale, int32_t num_splits,
                                      void *workspace, size_t workspace_bytes, void *stream) {
  pgd_status s = check_attention_args(out, q, k_cache, v_cache, block_tables, context_lens, B,
                                      n_q, n_kv, d, bs, MB, NB, scale, num_splits);
  if (s != PGD_OK) return s;
  if (B == 0) return ok();
  s = launch_attention(out, q, k_cache, v_cache, block_tables, context_lens, B, n_q, n_kv, bs,
                       MB, NB, scale, num_splits, workspace, workspace_bytes,
                       static_cast<cudaStream_t>(stream));
  return s == PGD_OK ? ok() : s;
}

pgd_status pgd_append_decode_attention(void *out, const void *q, const void *k_new,
                                       const void *v_new, void *k_cache, void *v_cache,
                                       const int32_t *block_tables, const int32_t *context_lens,
                                       int32_t B, int32_t n_q, int32_t n_kv, int32_t d, int32_t bs,
                                       int32_t MB, int32_t NB, float scale, int32_t num_splits,
                                       void *workspace, size_t workspace_bytes, void *stream) {
  pgd_status s = check_attention_args(out, q, k_cache, v_cache, block_tables, context_lens, B,
                                      n_q, n_kv, d, bs, MB, NB, scale, num_splits);
  if (s != PGD_OK) return s;
  if (B == 0) return ok();
  s = append_then_attend(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, B,
                         n_q, n_kv, bs, MB, NB, scale, num_splits, workspace, workspace_bytes,
                         static_cast<cudaStream_t>(stream));
  return s == PGD_OK ? ok() : s;
}

// -------------------------------------------------- cascade (shared prefix)

size_t pgd_cascade_workspace_size(int32_t B, int32_t n_q, int32_t n_kv, int32_t d, int32_t bs,
                                  int32_t num_splits, int32_t max_group_size,
                                  int32_t max_group_blocks) {
  if (max_group_size < 0 || max_group_blocks < 0 || bs <= 0) return 0;
  const size_t dec = pgd_attention_workspace_size(B, n_q, n_kv, d, num_splits);
  if (dec == 0) return 0;
  // (sized for the largest split of the prefix: one group)
  return cascade_plan(B, n_q, n_kv, bs, 1, max_group_size, max_group_blocks, dec, 1 << 20).total;
}

pgd_status pgd_cascade_decode_attention(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, const int32_t *seq_prefix_blocks,
    const int32_t *group_first, const int32_t *group_size, const int32_t *group_blocks,
    int32_t n_groups, int32_t max_group_size, int32_t max_group_blocks, int32_t B, int32_t n_q,
    int32_t n_kv, int32_t d, int32_t bs, int32_t MB, int32_t NB, float scale, int32_t num_splits,
    void *workspace, size_t workspace_bytes, void *stream) {
  pgd_status s = check_attention_args(out, q, k_cache, v_cache, block_tables, context_lens, B,
                                      n_q, n_kv, d, bs, MB, NB, scale, num_splits);
  if (s != PGD_OK) return s;
  if (B == 0) return ok();
  if (n_groups < 0 || max_group_size < 0 || max_group_blocks < 0 || max_group_blocks > MB ||
      (n_groups > 0 && (max_group_size < 1 || max_group_size > B)))
    return fail(PGD_ERR_INVALID_ARG, "bad group bounds");
  if ((long long)n_groups * n_kv * 16 * ((max_group_size * (n_q / n_kv) + 127) / 128) > (1LL << 30))
    return fail(PGD_ERR_INVALID_ARG, "too many groups");
  if (n_groups > 0 && (!seq_prefix_blocks || !group_first || !group_size || !group_blocks))
    return fail(PGD_ERR_INVALID_ARG, "null group array");
  if (!workspace || !aligned(workspace, kWsAlign))
    return fail(PGD_ERR_WORKSPACE, "workspace is NULL or not 256-aligned");
  const size_t dec = pgd_attention_workspace_size(B, n_q, n_kv, d, num_splits);
  const CascadePlan plan =
      cascade_plan(B, n_q, n_kv, bs, n_groups, max_group_size, max_group_blocks, dec, sm_count());
  if (workspace_bytes < plan.total)
    return fail(PGD_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, plan.total);
  PreparedAttention pa;
  s = prepare_attention(out, q, k_cache, v_cache, block_tables, context_lens, B, n_q, n_kv, bs, MB,
                        NB, scale, num_splits, workspace, dec, &pa);
  if (s != PGD_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (n_groups == 0) {  // plain attention, through the same kernel choice
    s = short_path(pa, num_splits, MB, bs)
            ? launch_short(pa, nullptr, nullptr, const_cast<void *>(k_cache),
                           const_cast<void *>(v_cache), st)
            : launch_prepared(pa, st);
    return s == PGD_OK ? ok() : s;
  }
  // 1. shared-prefix pass, on a few SMs; it lets the suffix pass launch at
  //    once on the others
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  float *pre_ml = reinterpret_cast<float *>(ws + plan.pre_ml);
  float *pre_o = reinterpret_cast<float *>(ws + plan.pre_o);
  PrefixParams pp;
  pp.q = static_cast<const __nv_bfloat16 *>(q);
  pp.k_cache = static_cast<const unsigned char *>(k_cache);
  pp.v_cache = static_cast<const unsigned char *>(v_cache);
  pp.tables = block_tables;
  pp.group_first = group_first;
  pp.group_size = group_size;
  pp.group_blocks = group_blocks;
  pp.n_groups = n_groups;
  pp.B = B;
  pp.n_q = n_q;
  pp.n_kv = n_kv;
  pp.MB = MB;
  pp.NB = NB;
  pp.n_rchunk = plan.n_rchunk;
  pp.n_tsplit = plan.n_tsplit;
  pp.qk_scale_log2 = pa.p.qk_scale_log2;
  pp.pre_ml = pre_ml;
  pp.pre_o = pre_o;
  pp.err = pa.p.err;
  pp.wait_limit_ns = pa.p.wait_limit_ns;
  const int grid = n_groups * n_kv * plan.n_rchunk * plan.n_tsplit;
  cudaError_t e = prefix_attention_launch(pp, pa.G, bs, grid, st);
  if (e != cudaSuccess) return cuda_fail(e, "shared-prefix pass launch");
  // 2. suffix pass: each sequence's own blocks, partial states only, on the
  //    SMs the prefix pass leaves (an automatic grid shrinks by its CTAs); it
  //    waits for the prefix pass only before exiting
  pa.p.seq_prefix_blocks = seq_prefix_blocks;
  pa.p.pre_ml = pre_ml;
  pa.p.pre_o = pre_o;
  pa.p.n_tsplit = plan.n_tsplit;
  pa.p.part_info = reinterpret_cast<int2 *>(ws + plan.part_info);
  pa.p.wait_late = 2;
  if (num_splits == 0) {
    const int sms = sm_count();
    pa.grid = std::max(std::min(pa.grid, sms - grid), std::max(1, sms / 2));
  }
  pa.p.prefetch_units = (num_splits == 0 && (long long)B * n_kv <= pa.grid) ? 1 : 0;
  s = launch_prepared(pa, st);
  if (s != PGD_OK) return s;
  // 3. combine: suffix and prefix parts of every unit with a shared prefix
  CombineParams cp;
  cp.out = pa.p.out;
  cp.seq_prefix_blocks = seq_prefix_blocks;
  cp.part_ml = pa.p.part_ml;
  cp.part_o = pa.p.part_o;
  cp.part_info = pa.p.part_info;
  cp.pre_ml = pre_ml;
  cp.pre_o = pre_o;
  cp.B = B;
  cp.n_q = n_q;
  cp.n_kv = n_kv;
  cp.n_tsplit = plan.n_tsplit;
  cp.ctx = context_lens;
  cp.bs = bs;
  cp.MB = MB;
  cp.parts = pa.grid;
  e = cascade_combine_launch(cp, pa.G, st);
  if (e != cudaSuccess) return cuda_fail(e, "cascade combine launch");
  return ok();
}

// ------------------------------------------------------------- MLA latent cache

constexpr int kMlaD = 576, kMlaDv = 512;

// Parts of each sequence's context for an automatic MLA call: as many as
// fill the SMs with one CTA each (the kernel's shared memory allows one per
// SM), at least one.
int mla_auto_parts(int32_t B, int32_t H) {
  const long long units = (long long)B * ((H + mla_heads_per_cta() - 1) / mla_heads_per_cta());
  if (units <= 0) return 1;
  return (int)std::max(1LL, std::min(64LL, (long long)sm_count() / units));
}

size_t mla_ws_bytes(int32_t B, int32_t H, int parts) {
  if (parts <= 1) return 0;
  const size_t rows = (size_t)B * H * parts;
  return round_up(rows * 2 * 4, kWsAlign) + rows * kMlaDv * 4;
}

size_t pgd_mla_workspace_size(int32_t B, int32_t H, int32_t num_splits) {
  if (B < 0 || H <= 0 || num_splits < 0) return 0;
  const int parts = num_splits > 0 ? num_splits : mla_auto_parts(B, H);
  clear_error_detail();
  return std::max<size_t>(mla_ws_bytes(B, H, parts), 256);
}

pgd_status check_mla_append(const void *c_new, const void *cache, const int32_t *block_tables,
                            const int32_t *positions, int32_t B, int32_t d, int32_t bs,
                            int32_t MB, int32_t NB) {
  if (B < 0) return fail(PGD_ERR_INVALID_ARG, "B = %d", B);
  if (d != kMlaD) return fail(PGD_ERR_UNSUPPORTED, "d = %d (576 cached values per token)", d);
  if (bs != 16 && bs != 32 && bs != 64) return fail(PGD_ERR_UNSUPPORTED, "block size %d", bs);
  if (MB <= 0 || NB <= 0) return fail(PGD_ERR_INVALID_ARG, "MB, NB must be > 0");
  if ((long long)B * MB >= 0x7fffffffLL) return fail(PGD_ERR_INVALID_ARG, "B * MB >= 2^31");
  if (B == 0) return PGD_OK;
  if (!c_new || !cache || !block_tables || !positions)
    return fail(PGD_ERR_INVALID_ARG, "null pointer");
  if (!aligned(c_new, 16) || !aligned(cache, 16))
    return fail(PGD_ERR_INVALID_ARG, "bf16 arrays must be 16-byte aligned");
  return PGD_OK;
}

// Checks and the parameter block of an MLA attention call; nothing enqueued.
pgd_status mla_prepare(void *out, const void *q, const void *cache, const int32_t *block_tables,
                       const int32_t *context_lens, int32_t B, int32_t H, int32_t d, int32_t dv,
                       int32_t bs, int32_t MB, int32_t NB, float scale, int32_t num_splits,
                       void *workspace, size_t workspace_bytes, MlaParams *pp) {
  if (B < 0 || H <= 0) return fail(PGD_ERR_INVALID_ARG, "B = %d, H = %d", B, H);
  if (d != kMlaD || dv != kMlaDv)
    return fail(PGD_ERR_UNSUPPORTED, "d = %d, dv = %d (576 and 512)", d, dv);
  if (bs != 16 && bs != 32 && bs != 64) return fail(PGD_ERR_UNSUPPORTED, "block size %d", bs);
  if (MB <= 0 || NB <= 0) return fail(PGD_ERR_INVALID_ARG, "MB, NB must be > 0");
  if (!(scale > 0.f) || !isfinite(scale)) return fail(PGD_ERR_INVALID_ARG, "scale must be > 0");
  if (num_splits < 0 || num_splits > 1024) return fail(PGD_ERR_INVALID_ARG, "num_splits");
  if ((long long)B * MB >= 0x7fffffffLL || (long long)B * H * 1024 >= 0x7fffffffLL)
    return fail(PGD_ERR_INVALID_ARG, "sizes too large");
  if (B == 0) return PGD_OK;
  if (!out || !q || !cache || !block_tables || !context_lens)
    return fail(PGD_ERR_INVALID_ARG, "null pointer");
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(cache, 16))
    return fail(PGD_ERR_INVALID_ARG, "bf16 arrays must be 16-byte aligned");
  const int parts = num_splits > 0 ? num_splits : mla_auto_parts(B, H);
  const size_t need = mla_ws_bytes(B, H, parts);
  if (need > 0 && (!workspace || !aligned(workspace, kWsAlign) || workspace_bytes < need))
    return fail(PGD_ERR_WORKSPACE, "workspace: %zu bytes (256-aligned) needed", need);
  int32_t *err = nullptr;
  pgd_status s = error_word(&err);
  if (s != PGD_OK) return s;
  MlaParams p;
  p.out = static_cast<__nv_bfloat16 *>(out);
  p.q = static_cast<const __nv_bfloat16 *>(q);
  p.cache = static_cast<const unsigned char *>(cache);
  p.tables = block_tables;
  p.ctx = context_lens;
  p.B = B;
  p.H = H;
  p.MB = MB;
  p.NB = NB;
  p.bs = bs;
  p.n_parts = parts;
  p.wait_late = 0;
  p.qk_scale_log2 = (float)((double)scale * 1.4426950408889634);
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  const size_t rows = (size_t)B * H * parts;
  p.part_ml = need ? reinterpret_cast<float *>(ws) : nullptr;
  p.part_o = need ? reinterpret_cast<float *>(ws + round_up(rows * 2 * 4, kWsAlign)) : nullptr;
  p.err = err;
  p.wait_limit_ns = g_wait_limit_ns.load();
  *pp = p;
  return PGD_OK;
}

pgd_status pgd_mla_append(const void *c_new, void *cache, const int32_t *block_tables,
                          const int32_t *positions, int32_t B, int32_t d, int32_t bs, int32_t MB,
                          int32_t NB, void *stream) {
  pgd_status s = check_mla_append(c_new, cache, block_tables, positions, B, d, bs, MB, NB);
  if (s != PGD_OK) return s;
  if (B == 0) return ok();
  int32_t *err = nullptr;
  s = error_word(&err);
  if (s != PGD_OK) return s;
  cudaError_t e = mla_append_launch(c_new, cache, block_tables, positions, 0, B, bs, MB, NB, err,
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "MLA append launch");
  return ok();
}

pgd_status pgd_mla_decode_attention(void *out, const void *q, const void *cache,
                                    const int32_t *block_tables, const int32_t *context_lens,
                                    int32_t B, int32_t H, int32_t d, int32_t dv, int32_t bs,
                                    int32_t MB, int32_t NB, float scale, int32_t num_splits,
                                    void *workspace, size_t workspace_bytes, void *stream) {
  MlaParams p;
  pgd_status s = mla_prepare(out, q, cache, block_tables, context_lens, B, H, d, dv, bs, MB, NB,
                             scale, num_splits, workspace, workspace_bytes, &p);
  if (s != PGD_OK) return s;
  if (B == 0) return ok();
  cudaError_t e = mla_attention_launch(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "MLA attention launch");
  return ok();
}

pgd_status pgd_mla_append_decode_attention(void *out, const void *q, const void *c_new,
                                           void *cache, const int32_t *block_tables,
                                           const int32_t *context_lens, int32_t B, int32_t H,
                                           int32_t d, int32_t dv, int32_t bs, int32_t MB,
                                           int32_t NB, float scale, int32_t num_splits,
                                           void *workspace, size_t workspace_bytes,
                                           void *stream) {
  pgd_status s = check_mla_append(c_new, cache, block_tables, context_lens, B, d, bs, MB, NB);
  if (s != PGD_OK) return s;
  MlaParams p;
  s = mla_prepare(out, q, cache, block_tables, context_lens, B, H, d, dv, bs, MB, NB, scale,
                  num_splits, workspace, workspace_bytes, &p);
  if (s != PGD_OK) return s;
  if (B == 0) return ok();
  // the append at context_lens[b] - 1, then the attention, told that the
  // kernel before it writes only the cache
  cudaError_t e = mla_append_launch(c_new, cache, block_tables, context_lens, -1, B, bs, MB, NB,
                                    p.err, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "MLA append launch");
  p.wait_late = 1;
  e = mla_attention_launch(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "MLA attention launch");
  return ok();
}

// ------------------------------------------------------------- 8-bit cache

pgd_status pgd_kv_append_fp8(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                             const int32_t *block_tables, const int32_t *positions, int32_t B,
                             int32_t n_kv, int32_t d, int32_t bs, int32_t MB, int32_t NB,
                             void *stream) {
  if (B < 0) return fail(PGD_ERR_INVALID_ARG, "B = %d", B);
  pgd_status s = check_cache_shape(n_kv, d, bs, MB, NB);
  if (s != PGD_OK) return s;
  if ((long long)B * n_kv > 0x7fffffffLL) return fail(PGD_ERR_INVALID_ARG, "B * n_kv too large");
  if (B == 0) return ok();
  if (!k_new || !v_new || !k_cache || !v_cache || !block_tables || !positions)
    return fail(PGD_ERR_INVALID_ARG, "null pointer");
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return fail(PGD_ERR_INVALID_ARG, "arrays must be 16-byte aligned");
  int32_t *err = nullptr;
  s = error_word(&err);
  if (s != PGD_OK) return s;
  cudaError_t e = kv_append_fp8_launch(k_new, v_new, k_cache, v_cache, block_tables, positions, 0,
                                       B, n_kv, bs, MB, NB, err,
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_append_fp8 launch");
  return ok();
}

pgd_status pgd_paged_decode_attention_fp8(void *out, const void *q, const void *k_cache,
                                          const void *v_cache, const int32_t *block_tables,
                                          const int32_t *context_lens, int32_t B, int32_t n_q,
                                          int32_t n_kv, int32_t d, int32_t bs, int32_t MB,
                                          int32_t NB, float scale, int32_t num_splits,
                                          void *workspace, size_t workspace_bytes,
                                          void *stream) {
  pgd_status s = check_attention_args(out, q, k_cache, v_cache, block_tables, context_lens, B,
                                      n_q, n_kv, d, bs, MB, NB, scale, num_splits);
  if (s != PGD_OK) return s;
  if (B == 0) return ok();
  PreparedAttention pa;
  s = prepare_attention(out, q, k_cache, v_cache, block_tables, context_lens, B, n_q, n_kv, bs, MB,
                        NB, scale, num_splits, workspace, workspace_bytes, &pa, true);
  if (s != PGD_OK) return s;
  s = short_path(pa, num_splits, MB, bs)
          ? launch_short(pa, nullptr, nullptr, const_cast<void *>(k_cache),
                         const_cast<void *>(v_cache), static_cast<cudaStream_t>(stream))
          : launch_prepared(pa, static_cast<cudaStream_t>(stream));
  return s == PGD_OK ? ok() : s;
}

pgd_status pgd_append_decode_attention_fp8(void *out, const void *q, const void *k_new,
                                           const void *v_new, void *k_cache, void *v_cache,
                                           const int32_t *block_tables,
                                           const int32_t *context_lens, int32_t B, int32_t n_q,
                                           int32_t n_kv, int32_t d, int32_t bs, int32_t MB,
                                           int32_t NB, float scale, int32_t num_splits,
                                           void *workspace, size_t workspace_bytes,
                                           void *stream) {
  pgd_status s = check_attention_args(out, q, k_cache, v_cache, block_tables, context_lens, B,
                                      n_q, n_kv, d, bs, MB, NB, scale, num_splits);
  if (s != PGD_OK) return s;
  if (B == 0) return ok();
  s = append_then_attend(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, B,
                         n_q, n_kv, bs, MB, NB, scale, num_splits, workspace, workspace_bytes,
                         static_cast<cudaStream_t>(stream), true);
  return s == PGD_OK ? ok() : s;
}

// The device's address of a page-locked host buffer that it can reach (and
// that is 16-byte aligned, as the kernels' vector accesses need), else null.
static void *device_alias(const void *h) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer || !aligned(a.devicePointer, 16))
    return nullptr;
  return a.devicePointer;
}

}  // extern "C"

// The host half of a step with host buffers: page-locked host buffers that
// the device addresses (16-byte aligned) are read -- q, k_new, v_new, the
// context lengths -- and written -- out -- in place by the kernels over the
// host link, instead of through a copy each (a copy in the stream would also
// end the chain of kernels launched while their predecessor runs); any other
// buffer goes through its device buffer and a copy.  `launch` enqueues the
// step's kernels on the pointers it is given, told whether every input is
// read in place (then no kernel of the stream writes them, and the kernels
// may read them before the previous kernel has completed).  qb: bytes of q
// (and out), kvb: bytes of k_new (and v_new).
template <typename Launch>
static pgd_status host_step(void *out_h, const void *q_h, const void *k_new_h, const void *v_new_h,
                            const int32_t *context_lens_h, void *out_d, void *q_d, void *k_new_d,
                            void *v_new_d, int32_t *context_lens_d, int32_t B, size_t qb,
                            size_t kvb, cudaStream_t st, Launch launch) {
  const void *q_in = device_alias(q_h), *kn_in = device_alias(k_new_h),
             *vn_in = device_alias(v_new_h);
  void *out_to = device_alias(out_h);
  const int32_t *cl_in = static_cast<const int32_t *>(device_alias(context_lens_h));
  cudaError_t e = cudaSuccess;
  if ((!q_in && (e = cudaMemcpyAsync(q_d, q_h, qb, cudaMemcpyHostToDevice, st)) != cudaSuccess) ||
      (!kn_in &&
       (e = cudaMemcpyAsync(k_new_d, k_new_h, kvb, cudaMemcpyHostToDevice, st)) != cudaSuccess) ||
      (!vn_in &&
       (e = cudaMemcpyAsync(v_new_d, v_new_h, kvb, cudaMemcpyHostToDevice, st)) != cudaSuccess) ||
      (!cl_in && (e = cudaMemcpyAsync(context_lens_d, context_lens_h, (size_t)B * 4,
                                      cudaMemcpyHostToDevice, st)) != cudaSuccess))
    return cuda_fail(e, "host-buffer step: host-to-device copy");
  const bool in_place = q_in && kn_in && vn_in && cl_in;
  pgd_status s = launch(out_to ? out_to : out_d, q_in ? q_in : q_d, kn_in ? kn_in : k_new_d,
                        vn_in ? vn_in : v_new_d, cl_in ? cl_in : context_lens_d, st, in_place);
  if (s != PGD_OK) return s;
  if (!out_to && (e = cudaMemcpyAsync(out_h, out_d, qb, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
    return cuda_fail(e, "host-buffer step: device-to-host copy");
  return ok();
}

extern "C" {

static pgd_status decode_step_impl(bool fp8, void *out_h, const void *q_h, const void *k_new_h, const void *v_new_h,
                           const int32_t *context_lens_h, void *out_d, void *q_d, void *k_new_d,
                           void *v_new_d, int32_t *context_lens_d, void *k_cache, void *v_cache,
                           const int32_t *block_tables, int32_t B, int32_t n_q, int32_t n_kv,
                           int32_t d, int32_t bs, int32_t MB, int32_t NB, float scale,
                           int32_t num_splits, void *workspace, size_t workspace_bytes,
                           void *stream) {
  pgd_status s = check_attention_args(out_d, q_d, k_cache, v_cache, block_tables, context_lens_d,
                                      B, n_q, n_kv, d, bs, MB, NB, scale, num_splits);
  if (s != PGD_OK) return s;
  if (B == 0) return ok();
  if (!out_h || !q_h || !k_new_h || !v_new_h || !context_lens_h || !k_new_d || !v_new_d)
    return fail(PGD_ERR_INVALID_ARG, "null pointer");
  if (!aligned(k_new_d, 16) || !aligned(v_new_d, 16))
    return fail(PGD_ERR_INVALID_ARG, "bf16 arrays must be 16-byte aligned");
  {
    // every check of the device half runs before the first copy is enqueued
    PreparedAttention pa;
    s = prepare_attention(out_d, q_d, k_cache, v_cache, block_tables, context_lens_d, B, n_q,
                          n_kv, bs, MB, NB, scale, num_splits, workspace, workspace_bytes, &pa,
                          fp8);
    if (s != PGD_OK) return s;
  }
  const size_t qb = (size_t)B * n_q * kHeadDim * 2, kvb = (size_t)B * n_kv * kHeadDim * 2;
  return host_step(out_h, q_h, k_new_h, v_new_h, context_lens_h, out_d, q_d, k_new_d, v_new_d,
                   context_lens_d, B, qb, kvb, static_cast<cudaStream_t>(stream),
                   [&](void *o, const void *q, const void *kn, const void *vn, const int32_t *cl,
                       cudaStream_t st, bool in_place) {
                     return append_then_attend(o, q, kn, vn, k_cache, v_cache, block_tables, cl,
                                               B, n_q, n_kv, bs, MB, NB, scale, num_splits,
                                               workspace, workspace_bytes, st, fp8, in_place);
                   });
}

pgd_status pgd_decode_step(void *out_h, const void *q_h, const void *k_new_h, const void *v_new_h,
                           const int32_t *context_lens_h, void *out_d, void *q_d, void *k_new_d,
                           void *v_new_d, int32_t *context_lens_d, void *k_cache, void *v_cache,
                           const int32_t *block_tables, int32_t B, int32_t n_q, int32_t n_kv,
                           int32_t d, int32_t bs, int32_t MB, int32_t NB, float scale,
                           int32_t num_splits, void *workspace, size_t workspace_bytes,
                           void *stream) {
  return decode_step_impl(false, out_h, q_h, k_new_h, v_new_h, context_lens_h, out_d, q_d, k_new_d,
                          v_new_d, context_lens_d, k_cache, v_cache, block_tables, B, n_q, n_kv, d,
                          bs, MB, NB, scale, num_splits, workspace, workspace_bytes, stream);
}

pgd_status pgd_decode_step_fp8(void *out_h, const void *q_h, const void *k_new_h,
                               const void *v_new_h, const int32_t *context_lens_h, void *out_d,
                               void *q_d, void *k_new_d, void *v_new_d, int32_t *context_lens_d,
                               void *k_cache, void *v_cache, const int32_t *block_tables,
                               int32_t B, int32_t n_q, int32_t n_kv, int32_t d, int32_t bs,
                               int32_t MB, int32_t NB, float scale, int32_t num_splits,
                               void *workspace, size_t workspace_bytes, void *stream) {
  return decode_step_impl(true, out_h, q_h, k_new_h, v_new_h, context_lens_h, out_d, q_d, k_new_d,
                          v_new_d, context_lens_d, k_cache, v_cache, block_tables, B, n_q, n_kv, d,
                          bs, MB, NB, scale, num_splits, workspace, workspace_bytes, stream);
}

pgd_status pgd_verify_step(void *out_h, const void *q_h, const void *k_new_h, const void *v_new_h,
                           const int32_t *context_lens_h, void *out_d, void *q_d, void *k_new_d,
                           void *v_new_d, int32_t *context_lens_d, void *k_cache, void *v_cache,
                           const int32_t *block_tables, int32_t B, int32_t T, int32_t n_q,
                           int32_t n_kv, int32_t d, int32_t bs, int32_t MB, int32_t NB,
                           float scale, int32_t num_splits, void *workspace,
                           size_t workspace_bytes, void *stream) {
  pgd_status s = check_attention_args(out_d, q_d, k_cache, v_cache, block_tables, context_lens_d,
                                      B, n_q, n_kv, d, bs, MB, NB, scale, num_splits);
  if (s != PGD_OK) return s;
  if ((s = check_verify(B, T, n_q, n_kv)) != PGD_OK) return s;
  if (B == 0) return ok();
  if (!out_h || !q_h || !k_new_h || !v_new_h || !context_lens_h || !k_new_d || !v_new_d)
    return fail(PGD_ERR_INVALID_ARG, "null pointer");
  if (!aligned(k_new_d, 16) || !aligned(v_new_d, 16))
    return fail(PGD_ERR_INVALID_ARG, "bf16 arrays must be 16-byte aligned");
  if ((long long)B * T * n_kv > 0x7ffffffcLL)
    return fail(PGD_ERR_INVALID_ARG, "B * T * n_kv too large");
  {
    // every check of the device half runs before the first copy is enqueued
    PreparedAttention pa;
    s = prepare_attention(out_d, q_d, k_cache, v_cache, block_tables, context_lens_d, B, n_q,
                          n_kv, bs, MB, NB, scale, num_splits, workspace, workspace_bytes, &pa,
                          false, T);
    if (s != PGD_OK) return s;
  }
  const size_t qb = (size_t)B * T * n_q * kHeadDim * 2, kvb = (size_t)B * T * n_kv * kHeadDim * 2;
  return host_step(out_h, q_h, k_new_h, v_new_h, context_lens_h, out_d, q_d, k_new_d, v_new_d,
                   context_lens_d, B, qb, kvb, static_cast<cudaStream_t>(stream),
                   [&](void *o, const void *q, const void *kn, const void *vn, const int32_t *cl,
                       cudaStream_t st, bool in_place) {
                     (void)in_place;  // (the verify kernels read their inputs after the wait)
                     return append_then_verify(o, q, kn, vn, k_cache, v_cache, block_tables, cl,
                                               B, T, n_q, n_kv, bs, MB, NB, scale, num_splits,
                                               workspace, workspace_bytes, st);
                   });
}

// The MLA step with host buffers.  q is always copied: every context part
// of a (sequence, head group) loads it, so reading it in place would move it
// over the host link several times; c_new, the context lengths and the output
// are read and written in place when page-locked, like pgd_decode_step's.
pgd_status pgd_mla_step(void *out_h, const void *q_h, const void *c_new_h,
                        const int32_t *context_lens_h, void *out_d, void *q_d, void *c_new_d,
                        int32_t *context_lens_d, void *cache, const int32_t *block_tables,
                        int32_t B, int32_t H, int32_t d, int32_t dv, int32_t bs, int32_t MB,
                        int32_t NB, float scale, int32_t num_splits, void *workspace,
                        size_t workspace_bytes, void *stream) {
  pgd_status s = check_mla_append(c_new_d, cache, block_tables, context_lens_d, B, d, bs, MB, NB);
  if (s != PGD_OK) return s;
  MlaParams p;
  s = mla_prepare(out_d, q_d, cache, block_tables, context_lens_d, B, H, d, dv, bs, MB, NB, scale,
                  num_splits, workspace, workspace_bytes, &p);
  if (s != PGD_OK) return s;
  if (B == 0) return ok();
  if (!out_h || !q_h || !c_new_h || !context_lens_h)
    return fail(PGD_ERR_INVALID_ARG, "null pointer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t qb = (size_t)B * H * kMlaD * 2, cb = (size_t)B * kMlaD * 2,
               ob = (size_t)B * H * kMlaDv * 2;
  const void *cn_in = device_alias(c_new_h);
  const int32_t *cl_in = static_cast<const int32_t *>(device_alias(context_lens_h));
  void *out_to = device_alias(out_h);
  cudaError_t e = cudaSuccess;
  if ((e = cudaMemcpyAsync(q_d, q_h, qb, cudaMemcpyHostToDevice, st)) != cudaSuccess ||
      (!cn_in && (e = cudaMemcpyAsync(c_new_d, c_new_h, cb, cudaMemcpyHostToDevice, st)) !=
                     cudaSuccess) ||
      (!cl_in && (e = cudaMemcpyAsync(context_lens_d, context_lens_h, (size_t)B * 4,
                                      cudaMemcpyHostToDevice, st)) != cudaSuccess))
    return cuda_fail(e, "MLA step: host-to-device copy");
  if (cl_in) p.ctx = cl_in;
  if (out_to) p.out = static_cast<__nv_bfloat16 *>(out_to);
  e = mla_append_launch(cn_in ? cn_in : c_new_d, cache, block_tables, p.ctx, -1, B, bs, MB, NB,
                        p.err, st);
  if (e != cudaSuccess) return cuda_fail(e, "MLA append launch");
  p.wait_late = 1;
  e = mla_attention_launch(p, st);
  if (e != cudaSuccess) return cuda_fail(e, "MLA attention launch");
  if (!out_to && (e = cudaMemcpyAsync(out_h, out_d, ob, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
    return cuda_fail(e, "MLA step: device-to-host copy");
  return ok();
}


pgd_status pgd_copy_blocks(void *k_cache, void *v_cache, const int32_t *src_ids,
                           const int32_t *dst_ids, int32_t n, int32_t n_kv, int32_t d,
                           int32_t bs, int32_t NB, void *stream) {
  if (n < 0) return fail(PGD_ERR_INVALID_ARG, "n = %d", n);
  pgd_status s = check_cache_shape(n_kv, d, bs, 1, NB);
  if (s != PGD_OK) return s;
  if (n == 0) return ok();
  if (!k_cache || !v_cache || !src_ids || !dst_ids) return fail(PGD_ERR_INVALID_ARG, "null pointer");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16))
    return fail(PGD_ERR_INVALID_ARG, "caches must be 16-byte aligned");
  int32_t *err = nullptr;
  s = error_word(&err);
  if (s != PGD_OK) return s;
  cudaError_t e = copy_blocks_launch(k_cache, v_cache, src_ids, dst_ids, n, n_kv, bs, NB, err,
                                     static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "copy_blocks launch");
  return ok();
}

pgd_status pgd_read_stream(const void *src, size_t bytes, int32_t mode, void *stream) {
  if (mode != 0 && mode != 1) return fail(PGD_ERR_INVALID_ARG, "mode %d (0 or 1)", mode);
  if (bytes == 0) return ok();
  if (!src) return fail(PGD_ERR_INVALID_ARG, "null pointer");
  if (!aligned(src, 16)) return fail(PGD_ERR_INVALID_ARG, "src must be 16-byte aligned");
  const size_t unit = mode == 1 ? 4096 : 16;
  if (bytes % unit) return fail(PGD_ERR_INVALID_ARG, "bytes must be a multiple of %zu", unit);
  int32_t *err = nullptr;
  pgd_status s = error_word(&err);
  if (s != PGD_OK) return s;
  cudaError_t e = read_stream_launch(src, bytes, mode, err, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "read stream launch");
  return ok();
}

void pgd_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store((unsigned long long)ns); }

int32_t pgd_set_short_context_tokens(int32_t max_tokens) {
  return g_short_tokens.exchange(max_tokens < 0 ? 1024 : max_tokens);
}

int32_t pgd_short_path(int32_t B, int32_t n_kv, int32_t bs, int32_t MB, int32_t num_splits) {
  return short_rule(B, n_kv, MB, bs, num_splits, 1) ? 1 : 0;
}

uint64_t pgd_wait_limit_ns(void) {
  const unsigned long long v = g_wait_limit_ns.load();
  return v ? (uint64_t)v : (uint64_t)kWaitLimitNs;
}

pgd_status pgd_device_errors(int32_t *flags, int32_t clear, void *stream) {
  if (!flags) return fail(PGD_ERR_INVALID_ARG, "flags is NULL");
  int32_t *err = nullptr;
  pgd_status s = error_word(&err);
  if (s != PGD_OK) return s;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  e = cudaMemcpy(flags, err, sizeof(int32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  if (clear) {
    e = cudaMemset(err, 0, sizeof(int32_t));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "clear error word");
  }
  return ok();
}

}  // extern "C"
