// pgd_device.cuh -- device-side helpers shared by the libpgd kernels:
// mbarrier and bulk-copy (TMA engine) wrappers in inline PTX, bounded waits,
// bf16 unpacking and the kernel parameter blocks.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pgd.h"

namespace pgd {

constexpr int kHeadDim = 128;
constexpr unsigned kFullMask = 0xffffffffu;
// A bounded wait gives up after this long (ns of %globaltimer) and reports
// PGD_DEVERR_TIMEOUT instead of hanging the GPU.  Launches carry their own
// limit for the waits on other roles of the CTA (0 = this default; a test of
// the timeout exit sets a short one); the drains that make sure no copy is
// still landing when a CTA exits always use this one.
constexpr uint64_t kWaitLimitNs = 4000000000ull;

// Per-CTA wait control in shared memory: the abort flag that every bounded
// wait of the CTA checks (first member, so a pointer to it is a pointer to
// the whole), then the launch's wait limit.
struct WaitCtl {
  int abort;
  int pad;
  unsigned long long limit_ns;
};
__device__ __forceinline__ volatile int *init_wait_ctl(void *slot, unsigned long long limit_ns) {
  volatile WaitCtl *c = reinterpret_cast<volatile WaitCtl *>(slot);
  c->abort = 0;
  c->limit_ns = limit_ns ? limit_ns : kWaitLimitNs;
  return &c->abort;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- mbarrier (shared::cta) ------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// The same with a bound on how long the thread may be suspended inside the
// poll (hint_ns), instead of the system's own bound.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t *bar, uint32_t parity,
                                                   uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// Wait until the phase with the given parity has completed, or give up after
// kWaitLimitNs.  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ---- bulk copy global -> shared through the TMA engine ---------------------
// L2 policy for data read exactly once per call (the KV stream).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// dst (shared) and src (global) 16-byte aligned, bytes a multiple of 16.
// Completion is signalled as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Bulk prefetch of global memory into L2 (src 16-byte aligned, bytes a
// multiple of 16); a hint, with no completion to wait for.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Programmatic dependent launch.  launch_dependents lets the next kernel of
// the stream (launched with programmatic stream serialization) start its
// prologue; wait blocks until every kernel this one depends on has completed
// and its writes are visible.  Both are no-ops without such a neighbour.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Atomic add at GPU scope with acquire-release semantics: the calling
// thread's earlier writes (and those ordered before them by a CTA barrier)
// become visible with it, and the writes released by earlier additions are
// visible after it.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int *addr, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
  return old;
}

// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---- bf16 helpers ----------------------------------------------------------
// Two bf16 packed in one 32-bit word (element 2i in the low half).  bf16 is
// the upper half of a binary32, so widening is a shift or a mask.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void unpack8(const uint4 &r, float (&f)[8]) {
  f[0] = bf16lo(r.x); f[1] = bf16hi(r.x);
  f[2] = bf16lo(r.y); f[3] = bf16hi(r.y);
  f[4] = bf16lo(r.z); f[5] = bf16hi(r.z);
  f[6] = bf16lo(r.w); f[7] = bf16hi(r.w);
}

__device__ __forceinline__ void unpack4(const uint2 &r, float (&f)[4]) {
  f[0] = bf16lo(r.x); f[1] = bf16hi(r.x);
  f[2] = bf16lo(r.y); f[3] = bf16hi(r.y);
}

// ---- kernel parameter blocks ----------------------------------------------
struct AttnParams {
  __nv_bfloat16 *out;            // [B][n_q][D]
  const __nv_bfloat16 *q;        // [B][n_q][D]
  const unsigned char *k_cache;  // pool bytes: bf16 tiles, or 8-bit groups (codes + scales)
  const unsigned char *v_cache;
  const int32_t *tables;         // [B][MB]
  const int32_t *ctx;            // [B]
  int B, n_q, n_kv, MB, NB;
  int T;                         // query tokens per sequence: 1 (decode) or the new tokens of
                                 // a multi-query call, which attend causally among themselves
  int lg_gh;                     // log2 of the query heads per KV head
  int rows;                      // query rows per unit, T << lg_gh (<= the kernel's G)
  float qk_scale_log2;           // scale * log2(e): scores live in the log2 domain
  float *part_o;                 // [slots][G][D]  unnormalised partial outputs
  float *part_ml;                // [slots][G][2]  partial (max, sum), log2 domain
  int32_t *counters;             // [B * n_kv]     arrivals per split unit
  int auto_split;                // 1: whole units or balanced cuts, chosen per call
  int prefetch_units;            // 1: no more units than CTAs (automatic split): CTA c most
                                 //    likely streams unit c from its first block, whose first
                                 //    stages it asks L2 for during the prologue
  int wait_late;                 // 1: the previous kernel wrote only the caches (kv_append):
                                 //    wait for it just before the first cache read;
                                 // 2: it is a cascade's shared-prefix pass, independent of
                                 //    this one, which waited for the inputs before letting
                                 //    this grid launch: wait for it only before exiting, so
                                 //    that this grid completes after it
  // cascade (all null / 0 otherwise): sequence b's first seq_prefix_blocks[b]
  // blocks were attended by the shared-prefix pass, whose partial states for
  // (b, h) are pre_ml / pre_o[(b * n_q + h) * n_tsplit + part]
  const int32_t *seq_prefix_blocks;
  const float *pre_ml;
  const float *pre_o;
  int n_tsplit;
  int2 *part_info;               // cascade: per unit (first part, parts); such units are
                                 // merged with their prefix parts by the combine kernel
  int32_t *err;                  // device error word
  unsigned long long wait_limit_ns;  // bounded waits give up after this (0: kWaitLimitNs)
};

// Final merge of cascade attention (prefix_attention.cu): decode parts of
// each unit with a shared prefix, then the prefix parts, into the output.
struct CombineParams {
  __nv_bfloat16 *out;
  const int32_t *seq_prefix_blocks;
  const float *part_ml, *part_o;   // decode parts [slots][G][2] / [slots][G][D]
  const int2 *part_info;           // [units] (first part, parts)
  const float *pre_ml, *pre_o;     // prefix parts [B][n_q][n_tsplit][2] / [..][D]
  const int32_t *ctx;              // context lengths [B]
  int B, n_q, n_kv, n_tsplit;
  int bs, MB;                      // block size, blocks per table row
  int parts;                       // parts of the suffix pass (its grid)
};

// Shared-prefix pass of cascade attention (prefix_attention.cu).
struct PrefixParams {
  const __nv_bfloat16 *q;        // [B][n_q][D]
  const unsigned char *k_cache;  // bf16 tiled pools
  const unsigned char *v_cache;
  const int32_t *tables;         // [B][MB]
  const int32_t *group_first;    // [n_groups] first sequence of each group
  const int32_t *group_size;     // [n_groups] sequences in the group (consecutive)
  const int32_t *group_blocks;   // [n_groups] leading table blocks shared by the group
  int n_groups, B, n_q, n_kv, MB, NB;
  int n_rchunk;                  // chunks of 128 / G sequences per group
  int n_tsplit;                  // parts of each prefix
  float qk_scale_log2;
  float *pre_ml;                 // [B][n_q][n_tsplit][2]   partial (max, sum), log2 domain
  float *pre_o;                  // [B][n_q][n_tsplit][D]   unnormalised partial outputs
  int32_t *err;
  unsigned long long wait_limit_ns;  // bounded waits give up after this (0: kWaitLimitNs)
};

// Decode attention over an MLA latent cache (mla_attention.cu).
struct MlaParams {
  __nv_bfloat16 *out;            // [B][H][512] latent outputs
  const __nv_bfloat16 *q;        // [B][H][576] absorbed queries
  const unsigned char *cache;    // latent pool, bf16 [NB][bs/8][72][8][8]
  const int32_t *tables;         // [B][MB]
  const int32_t *ctx;            // [B]
  int B, H, MB, NB, bs;
  int n_parts;                   // parts of each sequence's context (1: no merge)
  int wait_late;                 // 1: the previous kernel is this library's latent append,
                                 //    which writes only the cache: wait for it just before
                                 //    the first cache read
  float qk_scale_log2;           // scale * log2(e)
  float *part_ml;                // [B][H][n_parts][2] partial (max, sum), log2 domain
  float *part_o;                 // [B][H][n_parts][512] unnormalised partial outputs
  int32_t *err;
  unsigned long long wait_limit_ns;  // bounded waits give up after this (0: kWaitLimitNs)
};

}  // namespace pgd
