// attention_kernel.cuh -- paged GQA decode attention for sm_103a on the
// fifth-generation tensor cores (tcgen05, accumulators in tensor memory),
// for a bf16 cache and for an 8-bit (FP8 E4M3 + per-token scale) cache.
// attention.cu and attention_fp8.cu instantiate it.
//
// What it computes ("Module 10: inference and serving", section "Attention
// reads a different cache per sequence"; "The math of Transformer inference",
// section 4): for every sequence b and query head h,
//   out[b][h] = sum_t softmax_t(scale * q[b][h] . k_t) v_t over the
//   context_lens[b] cached positions, K/V head h / G, read through the block
//   table ("Module 10", section "Mapping logical positions to physical
//   blocks").  The template's G is the number of query rows a unit serves:
//   the heads of a KV head, times the T new tokens of a multi-query
//   (speculative verify) call, whose token i sees positions up to
//   context_lens[b] - T + i ("Module 10", Lab 2's mask) -- up to 16 rows.
//
// Work split.  A unit is one (sequence, KV head); its K/V tiles are read once
// and serve all G query rows.  The units are laid end to end (sequence-major,
// then KV head) in a cost space -- each unit costs its blocks plus a fixed
// charge for a segment's start and end -- cut into one contiguous part per
// CTA in one of two ways, chosen by every CTA alike from the context lengths:
//   units     CTA c takes unit c whole (when there are no more units than
//             CTAs and the longest unit still streams no longer than the
//             whole job takes at the HBM rate): no partial states at all;
//   balanced  CTA c of P takes cost positions [X*c/P, X*(c+1)/P): every CTA
//             carries the same cost whatever the length mix.
// (Cascade calls start each sequence past its shared prefix and leave every
// such unit's partial states to a combine kernel.)
// A CTA walks its part unit by unit ("segments").  A segment that covers a
// whole unit writes the output; otherwise it writes its (max, sum, weighted
// sum) state and the last CTA of the unit to arrive merges the states by
// log-sum-exp ("The math of Transformer inference", section 8: split the
// sequence, attend locally, merge by log-sum-exp; the running-state update is
// the one in "LLM inference systems engineering", 2.8.3).  Arrival is an
// atomic counter per unit; no CTA waits for another.
//
// The two contractions of a 128-token stage run on the tensor cores with
// tokens on the M side (decode attention is HBM bound; on CUDA cores the
// 2 * G * 128 multiply-adds per token and KV head took most issue slots):
//   S^T[128 tok][16]  = K[128 tok][128 d]   . Q^T[128 d][16 heads]
//   O^T[128 d][16]   += V^T[128 d][128 tok] . P^T[128 tok][16 heads]
// N = 16 is the smallest N for M = 128; the G <= 8 real heads use the first
// columns, the rest are zeros.
//
// Operands.  The pool stores every (block, KV head) tile as 8 x 8 core
// matrices (row group of 8 tokens x 16 column chunks of 8 dims; element
// (slot s, dim i) at ((s/8)*16 + i/8)*64 + (s%8)*8 + i%8).  One bulk copy per
// tile therefore lands exactly in the tensor cores' no-swizzle layout, and
// the tiles of a stage placed back to back form one operand with uniform
// strides: K as the K-major A operand of q.k^T (8-row groups 2048 B apart,
// 16-byte column chunks 128 B apart) and V as the MN-major A operand of p.v
// (the same core matrices read the other way).  Q is written by threads as a
// K-major, 128-byte-swizzled B operand and P as an MN-major B operand.
//
// Roles (384 threads, one CTA per SM):
//   warps 0-3  softmax; thread t owns TMEM lane t (token row t of S)
//   warp 4     K producer, warp 5 V producer: bulk copies on the TMA engine,
//              one tile per lane, table entries prefetched 32 ahead; the K
//              producer also writes each segment's Q
//   warp 6     allocates tensor memory and issues q.k^T (one lane)
//   warp 7     issues p.v (one lane); with two issuers the q.k^T of the next
//              stages never queues behind the p.v of the current one
//   warps 8-11 epilogue: per segment, read O from tensor memory and write the
//              output or a partial state (and merge a unit's partials when
//              they are complete), off the softmax warps' critical path
//   warps 12-15 (8-bit cache only) V dequantisation into f16 operands
// Rings: 3 K stages and 3 V stages of 32 KiB; a K stage is free as soon as
// its q.k^T has completed, a V stage after its p.v.  S and P are double
// buffered by stage parity, O and Q by segment parity.  Every wait is bounded.
//
// 8-bit cache ("Module 10", section "Quantize the cache, evaluate the final
// artifact"; "The math of Transformer inference", section 11: KV in 8 bits
// halves the bytes a step reads, scales per head and token, dequantisation
// fused into the kernel).  A pool tile is (bs / 8) groups of 8 tokens, each
// group the tokens' E4M3 codes as 8-row x 16-byte core matrices (1024 B)
// followed by their 8 fp32 scales (32 B): one bulk copy per tile still lands
// codes and scales, and the groups sit 1056 B apart -- a uniform stride the
// MMA descriptors can step over.  q.k^T runs on the tensor cores in E4M3
// (kind::f8f6f4): each query head h is split into a high and a low E4M3 part
// (q / s_q = hi + lo, s_q a power of two that puts max |q| in [128, 256)),
// hi in column h and lo in column 8 + h of the same N = 16 MMA.  A bf16
// element has 8 significant bits, hi takes 4 and lo the other 4, so the
// split is the bf16 query itself (up to 2^-10 s_q for elements more than
// 2^9 below the head's largest) at no extra MMA; the softmax adds the two
// columns and applies s_q and the key's scale.  Four more warps dequantise V
// to f16 (code * scale, each thread its own token row) for an f16 p.v with
// f16 probabilities.
//
// Softmax keeps one reference maximum per head.  A stage moves the reference
// (and rescales O in tensor memory, after the previous p.v has completed)
// only when its maximum exceeds the reference by more than 8 in log2 units,
// so P <= 256 in bf16 and rescaling is rare; O and l share the reference, so
// the final division is exact up to rounding.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <math.h>

#include "pgd_device.cuh"

namespace pgd {
namespace tc {

constexpr int TOK = 128;                    // tokens per stage (MMA M of q.k^T)
constexpr int NPAD = 16;                    // MMA N: query rows padded to 16
constexpr int RMAX = 16;                    // query rows per unit at most (= NPAD)
constexpr int P_BYTES = TOK * NPAD * 2;     // [16 token groups][2 head groups][8][16 B]
constexpr int WARP_KP = 4, WARP_VP = 5, WARP_QK = 6, WARP_PV = 7, WARP_EPI = 8, WARP_CVT = 12;
// 12 warps; the 8-bit kernel adds NCVT warps that dequantise V (warps 12..)
constexpr int NCVT = 4;
template <bool FP8> constexpr int kThreads = FP8 ? 384 + 32 * NCVT : 384;
constexpr int NSB = 4;                      // S buffers (q.k^T may run 4 stages ahead)
constexpr uint32_t TMEM_COLS = 128;
constexpr float kRescaleLog2 = 8.f;         // move the reference when exceeded by 2^8
// Split choice.  One CTA streams at most about 1/kCtaShare of the HBM rate
// (its three 64 KiB K+V stages in flight over the load latency); merging a
// unit's partial states costs the CTA that merges them about
// kMergeFixedBytes of streaming time plus kMergePartBytes per part (a store,
// a fence and an atomic per part, then the reloads, in series).
// (per kind of cache: three 64 KiB bf16 stages, or four 33 KiB 8-bit ones)
template <bool FP8> constexpr long long kCtaShare = FP8 ? 140 : 96;
// (measured on 8 units of 32 blocks: one part per unit 12.8 us a step, two
// 16.5, nineteen 19.0)
constexpr long long kMergeFixedBytes = 24ll << 20;
constexpr long long kMergePartBytes = 1ll << 20;
// Fixed cost of a segment in blocks of streaming time: about three stages.
// (A per-CTA timeline of the cascade suffix pass, whose parts are made of
// many short segments, shows a one-stage segment taking 2-3 us against about
// 0.7 us per stage inside a long one; charging 2, 3, 4 and 6 stages gave
// 39.9, 39.3, 39.3 and 40.3 us a step there and left the ragged and
// single-sequence batches unchanged.)
template <int BS> constexpr int kSegCost = 3 * TOK / BS;
// Blocks of a CTA's likely first unit asked of L2 during the prologue: three
// stages (about the data HBM can deliver to each CTA while the prologue runs).
template <int BS> constexpr int kPrefetchBlocks = 3 * TOK / BS;
constexpr int MERGE_PAIRS = 128;
constexpr int SMEM_SLACK = 1024;

// Shared memory of one CTA (offsets from a 1024-byte aligned base).
template <bool FP8>
struct Lay {
  static constexpr int GROUP = FP8 ? 8 * 128 + 32 : 8 * 256;  // bytes per 8-token group
  static constexpr int STAGE = (TOK / 8) * GROUP;              // K (or V) bytes of a stage
  static constexpr int NSK = FP8 ? 4 : 3, NSV = FP8 ? 4 : 3;   // ring depths
  // Q operand per buffer: bf16 [half][16 rows][128 B] with 128-byte swizzle,
  // or E4M3 [16 rows][128 B] as 8 x 16-byte core matrices
  static constexpr int Q_BYTES = FP8 ? NPAD * 128 : 2 * NPAD * 128;
  static constexpr int VB_BYTES = FP8 ? 2 * TOK * 256 : 0;     // converted V, by stage parity
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NSK * STAGE;
  static constexpr int OFF_VB = OFF_V + NSV * STAGE;
  static constexpr int OFF_Q = OFF_VB + VB_BYTES;  // Q double buffered by segment parity
  static constexpr int OFF_P = OFF_Q + 2 * Q_BYTES;
  // 8-bit cache: the key scales of the last NKS stages, f32 [NKS][TOK], copied
  // out of each K stage by the q.k^T warp so that the stage frees with its MMA
  static constexpr int NKS = 8;
  static constexpr int OFF_KS = OFF_P + 2 * P_BYTES;
  static constexpr int OFF_BAR = OFF_KS + (FP8 ? NKS * TOK * 4 : 0);
  static constexpr int OFF_RED = OFF_BAR + 512;    // f32 [2][4][RMAX] warp maxima
  static constexpr int OFF_LRED = OFF_RED + 2 * 4 * RMAX * 4;  // f32 [2][4][RMAX] warp sums
  static constexpr int OFF_MREF = OFF_LRED + 2 * 4 * RMAX * 4;  // f32 [2][RMAX] reference maxima
  static constexpr int OFF_QS = OFF_MREF + 2 * RMAX * 4;  // f32 [2][8] Q scales per Q buffer (8-bit)
  static constexpr int OFF_MERGE = OFF_QS + 64;    // float2 [MERGE_PAIRS] partial (max, sum)
  static constexpr int OFF_MISC = OFF_MERGE + MERGE_PAIRS * 8;  // tmem base, flags, masks
  static constexpr int OFF_PRE = OFF_MISC + 128;   // int [B + 1]
};

template <bool FP8>
__host__ __device__ constexpr size_t smem_bytes(int B) {
  return (size_t)SMEM_SLACK + Lay<FP8>::OFF_PRE + (size_t)(B + 1) * 4;
}
static_assert(smem_bytes<false>(PGD_MAX_BATCH) <= 232448, "bf16 layout exceeds 227 KB");
static_assert((Lay<false>::OFF_MISC + 24) % 8 == 0 && (Lay<true>::OFF_MISC + 24) % 8 == 0,
              "WaitCtl alignment");
static_assert(smem_bytes<true>(PGD_MAX_BATCH) <= 232448, "8-bit layout exceeds 227 KB");

__device__ __forceinline__ uint32_t col_s(int sb) { return (uint32_t)sb * 16u; }  // sb < NSB

// 2^x by the hardware approximation, results below 2^-126 flushed to zero: a
// probability is rounded to f16 (bf16) next, whose step near 1 is 2^-11
// (2^-8), far above the approximation's error, and whose smallest value
// (2^-24) lies far above the flush.
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t col_o(int ob) { return 64u + (uint32_t)ob * 16u; }

// ---------------------------------------------------------------- PTX helpers
// Shared-memory matrix descriptor (tcgen05): start address, leading and
// stride byte offsets (16-byte units), descriptor version 1, layout
// (0 = no swizzle, 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)layout << 61);
}

// Instruction descriptor, kind::f16: D f32, A and B bf16 (or both f16),
// M = 128, N = 16; a_mn / b_mn select MN-major operands.
__host__ __device__ constexpr uint32_t instr_desc(bool a_mn, bool b_mn, bool bf16 = true) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(NPAD >> 3) << 17) |
         ((uint32_t)(TOK >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor, kind::f8f6f4: D f32, A and B E4M3 (format 0),
// both K-major, M = 128, N = 16.
__host__ __device__ constexpr uint32_t instr_desc_e4m3() {
  return (1u << 4) | ((uint32_t)(NPAD >> 3) << 17) | ((uint32_t)(TOK >> 4) << 24);
}

__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Generic-proxy shared-memory writes become visible to the tensor cores.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 8 consecutive fp32 columns of this warp's 32 TMEM lanes (wait included).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r0, r1, r2, r3, r4, r5, r6, r7;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3), "=r"(r4), "=r"(r5), "=r"(r6), "=r"(r7)
      : "r"(taddr)
      : "memory");
  v[0] = __uint_as_float(r0); v[1] = __uint_as_float(r1);
  v[2] = __uint_as_float(r2); v[3] = __uint_as_float(r3);
  v[4] = __uint_as_float(r4); v[5] = __uint_as_float(r5);
  v[6] = __uint_as_float(r6); v[7] = __uint_as_float(r7);
}

// 8 columns of this warp's 32 lanes, without the wait: the registers are
// valid only after tmem_wait8 on them (which names them, so the compiler
// cannot use them earlier).
__device__ __forceinline__ void tmem_ld8_async(uint32_t taddr, uint32_t *r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait8(uint32_t *r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7])
               :
               : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
      : "memory");
}

template <int G> constexpr int kLog2 = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : G == 8 ? 3 : 4;

// Max (or sum) over the warp of G per-lane values, one per head, with the
// values halved at each of the first log2(G) exchange steps (a lane keeps one
// half and sends the other), so G - 1 + 5 - log2(G) shuffles instead of 5 G.
// Lane l returns the result of head l >> (5 - log2(G)).
template <int G, bool MAX>
__device__ __forceinline__ float warp_reduce_heads(const float (&v)[G], int lane) {
  float a[G];
#pragma unroll
  for (int i = 0; i < G; ++i) a[i] = v[i];
#pragma unroll
  for (int n = G, off = 16; n > 1; n >>= 1, off >>= 1) {
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float keep = up ? a[i + n / 2] : a[i];
      const float send = up ? a[i] : a[i + n / 2];
      const float r = __shfl_xor_sync(kFullMask, send, off);
      a[i] = MAX ? fmaxf(keep, r) : keep + r;
    }
  }
#pragma unroll
  for (int off = 16 >> kLog2<G>; off > 0; off >>= 1) {
    const float r = __shfl_xor_sync(kFullMask, a[0], off);
    a[0] = MAX ? fmaxf(a[0], r) : a[0] + r;
  }
  return a[0];
}

// Bounded wait that gives up at once after any earlier timeout in the CTA, so
// that the control flow (and every named barrier) is the same for all threads
// whatever happens.  abort_flag is the first member of the CTA's WaitCtl,
// which also holds the launch's wait limit.
// (The spin is a function of its own: one copy of it instead of one per
// wait keeps the kernel's code small enough for the instruction caches.)
static __device__ __noinline__ void wait_spin(uint64_t *bar, uint32_t parity,
                                              volatile int *abort_flag, int32_t *err) {
  if (*abort_flag) return;
  const uint64_t limit = reinterpret_cast<const volatile WaitCtl *>(abort_flag)->limit_ns;
  const uint64_t t0 = global_timer_ns();
  // Every 32 failed polls: an earlier timeout in the CTA, or this wait's own.
  auto gave_up = [&]() {
    if (*abort_flag) return true;
    if (global_timer_ns() - t0 > limit) {
      *abort_flag = 1;
      atomicOr(err, PGD_DEVERR_TIMEOUT);
      return true;
    }
    return false;
  };
  if (limit < 1000000ull) {
    // A short limit (set only to exercise this exit) also bounds each poll's
    // suspension, and the clock is read after the first failed poll too, so
    // that an unmet wait gives up whatever the system's own suspension bound.
    for (uint32_t i = 1;; ++i) {
      if (mbar_try_wait_hint(bar, parity, (uint32_t)limit)) return;
      if ((i & 31u) == 1 && gave_up()) return;
    }
  }
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return;
    if ((i & 31u) == 0 && gave_up()) return;
  }
}
__device__ __forceinline__ void wait_or_abort(uint64_t *bar, uint32_t parity,
                                              volatile int *abort_flag, int32_t *err) {
  if (!mbar_try_wait(bar, parity)) wait_spin(bar, parity, abort_flag, err);
}

// The piece of a CTA's part inside one unit (sequence b, KV head g): blocks
// j0 .. j0 + n - 1 of the nblk blocks the kernel attends for sequence b; the
// unit spans [ucs, uce) of the cost space.
struct Segment {
  int b, g, j0, nblk, n;
  long long ucs, uce;
};

// Parts of one call: part c (taken by CTA c) is a contiguous range of the
// flattened cost space, in index order; a closed form of c, so every thread
// can map a part to its range and a cost position to its part.  Each unit
// costs its blocks plus ov: the ov positions in front of its first block
// stand for the fixed time of starting a segment (latency the softmax and
// epilogue pay per unit), so balanced cuts also balance the units per CTA.
struct Schedule {
  long long X;     // cost of all units
  long long P;     // parts
  bool units;      // part c = unit c (else X * c / P balanced cuts)
  const int *pre;  // cost of one head of the sequences before b
  int ov;          // cost of a unit beyond its blocks (0 for sequences without blocks)
  int n_kv;
  __device__ __forceinline__ void range(long long i, long long &a, long long &b) const {
    if (units) {
      const int sb = (int)(i / n_kv), g = (int)(i % n_kv);
      const long long nb = pre[sb + 1] - pre[sb];
      a = (long long)n_kv * pre[sb] + g * nb;
      b = a + nb;
    } else {
      a = X * i / P;
      b = X * (i + 1) / P;
    }
  }
  // Part holding cost position x (only needed for units that are cut,
  // which happens in balanced mode alone).
  __device__ __forceinline__ long long part_of(long long x) const {
    return (P * (x + 1) - 1) / X;
  }
};

// Query row r of unit (b, g) -- query token r >> lg_gh of the sequence's T,
// query head g * 2^lg_gh + (r & (2^lg_gh - 1)) -- as a row index of q and of
// out ([B][T][n_q] rows of d values; T = 1 for decode).
__device__ __forceinline__ size_t q_index(const AttnParams &p, int b, int g, int r) {
  return ((size_t)b * p.T + (size_t)(r >> p.lg_gh)) * p.n_q + ((size_t)g << p.lg_gh) +
         (size_t)(r & ((1 << p.lg_gh) - 1));
}

// First block of sequence b that this kernel attends (the blocks before it
// were attended by the shared-prefix pass of a cascade call).
__device__ __forceinline__ int start_block(const AttnParams &p, int b) {
  return p.seq_prefix_blocks ? __ldg(p.seq_prefix_blocks + b) : 0;
}

// A role's walk over the CTA's part, one segment (the piece of the part
// inside one unit that holds blocks) at a time.  Every role walks the same
// segments.  Only the first unit is found by search; the cursor then steps
// to the next unit (next head, or the next sequence with blocks).
struct SegCursor {
  long long x, end;  // rest of the part
  int b, g;          // unit of the last segment (b = -1 before the first)
  __device__ __forceinline__ SegCursor(const Schedule &sc) {
    x = end = 0;
    b = -1;
    g = 0;
    if ((long long)blockIdx.x < sc.P) sc.range(blockIdx.x, x, end);
  }
  __device__ __forceinline__ bool next(const Schedule &sc, int B, Segment &sg) {
    const int *pre = sc.pre;
    while (x < end) {
      if (b < 0) {
        int lo = 0, hi = B - 1;  // largest b with n_kv * pre[b] <= x
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if ((long long)sc.n_kv * pre[mid] <= x) lo = mid; else hi = mid - 1;
        }
        b = lo;
        const int cost = pre[b + 1] - pre[b];
        g = (int)((x - (long long)sc.n_kv * pre[b]) / cost);
      } else if (++g == sc.n_kv) {  // x is the start of the unit after (b, g)
        g = 0;
        do { ++b; } while (b < B - 1 && pre[b + 1] == pre[b]);
      }
      const int cost = pre[b + 1] - pre[b];
      const long long ucs = (long long)sc.n_kv * pre[b] + (long long)g * cost;
      const long long uce = ucs + cost;
      const long long e = end < uce ? end : uce;
      const int j0 = (int)max(0ll, x - ucs - sc.ov);
      const int j1 = (int)max(0ll, e - ucs - sc.ov);
      x = e;
      if (j1 > j0) {
        sg.b = b;
        sg.g = g;
        sg.j0 = j0;
        sg.nblk = cost - sc.ov;
        sg.n = j1 - j0;
        sg.ucs = ucs;
        sg.uce = uce;
        return true;
      }
    }
    return false;
  }
};

// E4M3 pair from two binary32 values (round to nearest even, saturating to
// +-448; x.x in the low byte) and back to binary32.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t v) {
  const __half2 h = __half2(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3));
  return __half22float2(h);
}

// 16 E4M3 codes of one token -> 16 dequantised f16 values code * scale (two
// 16-byte rows of 8): the code widens to f16 exactly, the product rounds to
// nearest.
__device__ __forceinline__ void e4m3x16_dequant_f16(const uint4 &c, __half2 scale, uint4 &lo,
                                                    uint4 &hi) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint16_t pair = (uint16_t)(w[i >> 1] >> ((i & 1) * 16));
    const __half2 h = __hmul2(
        __half2(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)pair, __NV_E4M3)), scale);
    o[i] = *reinterpret_cast<const uint32_t *>(&h);
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// One query head's 8 dims (one 16-byte piece of q) as E4M3 high and low
// parts of x = q / s_q: hi = E4M3(x), lo = E4M3(x - hi).  With s_q a power
// of two, x has a bf16 element's 8 significant bits; hi holds the top 4 and
// x - hi the rest (at most 4 bits), so hi + lo = x exactly whenever lo is
// not below E4M3's subnormal step 2^-9 -- for every element within a factor
// 2^9 of the head's largest -- and within 2^-10 of x otherwise.
__device__ __forceinline__ void q_hi_lo(const uint4 &piece, float inv_sq, uint2 &hi, uint2 &lo) {
  float f[8];
  unpack8(piece, f);
  uint16_t h[4], l[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float x0 = f[2 * j] * inv_sq, x1 = f[2 * j + 1] * inv_sq;
    h[j] = e4m3x2(x0, x1);
    const float2 hv = e4m3x2_to_float2(h[j]);
    l[j] = e4m3x2(x0 - hv.x, x1 - hv.y);
  }
  hi = make_uint2(h[0] | ((uint32_t)h[1] << 16), h[2] | ((uint32_t)h[3] << 16));
  lo = make_uint2(l[0] | ((uint32_t)l[1] << 16), l[2] | ((uint32_t)l[3] << 16));
}

// One producer warp (K or V): walks the CTA's stages and copies one tile per
// lane with the TMA engine.  The K producer also records which blocks of a
// stage had an invalid id and writes each segment's Q (the B operand of
// q.k^T) into buffer k & 1 as segment k starts: bf16 K-major with 128-byte
// swizzle (row = head, two 64-column halves), or for the 8-bit cache E4M3
// high parts in rows 0-7 and low parts in rows 8-15 (8 x 16-byte core
// matrices) plus one scale per head.  Loads run one step ahead: the next
// segment's Q and first 64 block ids while the current segment streams, and
// within a segment the block ids 32 entries ahead.
template <int G, int BS, bool FP8, bool IS_K>
__device__ __forceinline__ void produce(const AttnParams &p, const Schedule &sc,
                                        const unsigned char *cache, unsigned char *ring,
                                        uint64_t *full, uint64_t *empty,
                                        volatile int *stage_mask, unsigned char *qbuf,
                                        float *qscale, uint64_t *q_ready, uint64_t *q_free,
                                        volatile int *abort_flag, int lane) {
  using L = Lay<FP8>;
  constexpr int SB = TOK / BS;                         // blocks per stage
  constexpr uint32_t TILE_BYTES = (BS / 8) * L::GROUP;  // one (block, head) tile
  constexpr int NS = IS_K ? L::NSK : L::NSV;
  constexpr int QPL = (16 * G + 31) / 32;  // Q 16-byte pieces per lane
  const uint64_t policy = l2_policy_evict_first();

  struct Ahead {
    uint4 q[QPL];
    int tab, tab_next;
  };
  auto load_ahead = [&](const Segment &g, Ahead &a) {
    if (IS_K) {
#pragma unroll
      for (int i = 0; i < QPL; ++i) {
        const int j = lane + 32 * i, r = j >> 4, c = j & 15;
        a.q[i] = (j < 16 * G && r < p.rows)
                     ? __ldg(reinterpret_cast<const uint4 *>(p.q + q_index(p, g.b, g.g, r) *
                                                                       kHeadDim + c * 8))
                     : make_uint4(0, 0, 0, 0);
      }
    }
    const int32_t *trow = p.tables + (size_t)g.b * p.MB + start_block(p, g.b) + g.j0;
    a.tab = (lane < g.n) ? __ldg(trow + lane) : 0;
    a.tab_next = (32 + lane < g.n) ? __ldg(trow + 32 + lane) : 0;
  };

  SegCursor cur(sc);
  Segment sg, nsg;
  Ahead cur_a{}, next_a{};
  bool have = cur.next(sc, p.B, sg);
  if (have) load_ahead(sg, cur_a);
  if (p.wait_late == 1) pdl_wait();  // kv_append has written the caches
  int s = 0, k = 0;  // s: stages armed so far
  bool stop = false;  // after a timeout in the CTA: arm nothing more
  while (have && !stop) {
    const bool have_next = cur.next(sc, p.B, nsg);
    if (have_next) load_ahead(nsg, next_a);
    if (IS_K) {
      const int qb = k & 1;
      if (lane == 0)
        wait_or_abort(&q_free[qb], ((uint32_t)(k >> 1) & 1u) ^ 1u, abort_flag, p.err);
      __syncwarp();
      unsigned char *qdst = qbuf + qb * L::Q_BYTES;
      if constexpr (FP8) {
        // Lanes 16h'..16h'+15 of piece i hold head r = 2i + h': the head's
        // max |q| is a reduction over those 16 lanes.
#pragma unroll
        for (int i = 0; i < QPL; ++i) {
          const int j = lane + 32 * i, r = j >> 4, c = j & 15;
          float f[8];
          unpack8(cur_a.q[i], f);
          float a = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) a = fmaxf(a, fabsf(f[e]));
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(kFullMask, a, o));
          // s_q = 2^(e - 7), e = the exponent of max |q| (at least -119, so
          // that both s_q and 1 / s_q are normal binary32): q / s_q is q with
          // its exponent shifted, every element keeps its 8 significant bits,
          // and the largest lands in [128, 256), inside E4M3's range.
          const int e = max((int)((__float_as_uint(a) >> 23) & 0xffu) - 127, -119);
          const float sq = __uint_as_float((uint32_t)(e + 120) << 23);
          const float inv_sq = __uint_as_float((uint32_t)(134 - e) << 23);
          if (j < 16 * G) {
            uint2 hi, lo;
            q_hi_lo(cur_a.q[i], inv_sq, hi, lo);
            // row n, dims 8c..8c+7: core matrix (n / 8, c / 2), row n % 8
            const int off = (c >> 1) * 128 + (c & 1) * 8;
            *reinterpret_cast<uint2 *>(qdst + r * 16 + off) = hi;
            *reinterpret_cast<uint2 *>(qdst + 8 * 128 + r * 16 + off) = lo;
            if (c == 0) qscale[qb * 8 + r] = sq;
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < QPL; ++i) {
          const int j = lane + 32 * i, r = j >> 4, c = j & 15, half = c >> 3, cc = c & 7;
          if (j < 16 * G)
            *reinterpret_cast<uint4 *>(qdst + half * (NPAD * 128) + r * 128 +
                                       ((cc ^ (r & 7)) << 4)) = cur_a.q[i];
        }
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_ready[qb]);
    }
    ++k;
    const int32_t *trow = p.tables + (size_t)sg.b * p.MB + start_block(p, sg.b) + sg.j0;
    int tab = cur_a.tab, tab_next = cur_a.tab_next;
    int tchunk = 0;
    const int nstages = (sg.n + SB - 1) / SB;
    for (int st = 0; st < nstages; ++st, ++s) {
      const int first = st * SB;
      if ((first >> 5) != tchunk) {  // next 32 table entries; prefetch the ones after
        tchunk = first >> 5;
        tab = tab_next;
        const int j = (tchunk + 1) * 32 + lane;
        tab_next = (j < sg.n) ? __ldg(trow + j) : 0;
      }
      const int nb = min(SB, sg.n - first);
      const int blk = __shfl_sync(kFullMask, tab, (first & 31) + (lane & (SB - 1)));
      const bool ok = lane < nb && (unsigned)blk < (unsigned)p.NB;
      const unsigned okmask = __ballot_sync(kFullMask, ok);
      const unsigned want = (1u << nb) - 1u;
      const int slot = s % NS;
      // One decision for the whole warp: after a timeout the slot's earlier
      // copies may still be landing, so it is neither armed again (an
      // arrival there could meet a phase whose bytes are still pending) nor
      // written; the drain below waits for what was armed.
      int go = 1;
      if (lane == 0) {
        wait_or_abort(&empty[slot], ((uint32_t)(s / NS) & 1u) ^ 1u, abort_flag, p.err);
        go = *abort_flag ? 0 : 1;
      }
      if (!__shfl_sync(kFullMask, go, 0)) {
        stop = true;
        break;
      }
      if (lane == 0) {
        if (IS_K) {
          stage_mask[s & 7] = (int)(want & ~okmask);
          if (want & ~okmask) atomicOr(p.err, PGD_DEVERR_BAD_BLOCK_ID);
        } else if (FP8) {
          stage_mask[slot] = (int)(want & ~okmask);  // per V slot, for the V converters
        }
        const uint32_t bytes = (uint32_t)__popc(okmask) * TILE_BYTES;
        if (bytes == 0)
          mbar_arrive(&full[slot]);
        else
          mbar_arrive_expect_tx(&full[slot], bytes);
      }
      __syncwarp();
      if (ok) {
        const unsigned char *src = cache + ((size_t)blk * p.n_kv + sg.g) * (size_t)TILE_BYTES;
        bulk_copy_g2s(ring + (size_t)slot * L::STAGE + (size_t)lane * TILE_BYTES, src,
                      TILE_BYTES, &full[slot], policy);
      }
    }
    sg = nsg;
    cur_a = next_a;
    have = have_next;
  }
  // no copy may still be landing when the CTA exits: wait for the last NS
  // armed stages (every earlier one was consumed before its slot was armed
  // again), with the fixed limit whatever the launch's
  if (lane == 0) {
    for (int k = 1; k <= NS && k <= s; ++k) {
      const int last = s - k;
      if (!mbar_wait_bounded(&full[last % NS], (uint32_t)(last / NS) & 1u))
        atomicOr(p.err, PGD_DEVERR_TIMEOUT);
    }
  }
}

// Last-arriver merge of a unit's n_parts partial states (parts c0 ..), by
// log-sum-exp, into the bf16 output rows of query rows h < rows (row h at
// obase + (h >> lg_gh) * n_q + h mod 2^lg_gh); run by the 128 epilogue threads,
// thread e owning dim e.  The (max, sum) pairs are staged in shared memory
// PPB parts at a time; the partial outputs are read U parts at a time, every
// load of a group issued before any is used, the first group's while the
// maxima are formed.  Cold (once per cut unit), so out of line.
template <int G, bool FP8>
__device__ __noinline__ void merge_parts(const float *__restrict__ part_o,
                                         const float *__restrict__ part_ml,
                                         __nv_bfloat16 *__restrict__ out, int unit, int c0,
                                         int n_parts, size_t obase, int lg_gh, int n_q,
                                         int rows, int e, float2 *mlb) {
  constexpr int NET = 128;
  constexpr int PPB = MERGE_PAIRS / G;
  // (at most 24 parts; fewer where the running state takes more registers,
  // and under the 8-bit kernel's register budget)
  constexpr int U0 = (FP8 ? 16 : G >= 8 ? 48 : 96) / G;
  constexpr int U = U0 < 24 ? U0 : 24;
  const size_t row0 = ((size_t)unit + (size_t)c0) * G;
  float Mx[G], Lm[G], O[G];
#pragma unroll
  for (int h = 0; h < G; ++h) { Mx[h] = -INFINITY; Lm[h] = 0.f; O[h] = 0.f; }
#pragma unroll 1
  for (int base = 0; base < n_parts; base += PPB) {
    const int nb = min(PPB, n_parts - base);
    const size_t rb = row0 + (size_t)base * G;
    float ov[U][G];
    auto load_group = [&](int i0) {
#pragma unroll
      for (int i = 0; i < U; ++i) {
        if (i0 + i >= nb) break;
#pragma unroll
        for (int h = 0; h < G; ++h)
          ov[i][h] = __ldcg(part_o + (rb + (size_t)(i0 + i) * G + h) * kHeadDim + e);
      }
    };
    load_group(0);  // (independent of the maxima: in flight while they are formed)
#pragma unroll 1
    for (int j = e; j < nb * G; j += NET)
      mlb[j] = __ldcg(reinterpret_cast<const float2 *>(part_ml) + rb + j);
    named_barrier_sync(2, NET);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float bm = Mx[h];
#pragma unroll 8
      for (int i = 0; i < nb; ++i) bm = fmaxf(bm, mlb[i * G + h].x);
      if (bm != Mx[h] && Mx[h] != -INFINITY) {
        const float cf = exp2f(Mx[h] - bm);
        Lm[h] *= cf;
        O[h] *= cf;
      }
      Mx[h] = bm;
    }
#pragma unroll 1
    for (int i0 = 0; i0 < nb; i0 += U) {
      if (i0 > 0) load_group(i0);
#pragma unroll
      for (int i = 0; i < U; ++i) {
        if (i0 + i >= nb) break;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float2 ml = mlb[(i0 + i) * G + h];
          const float cf = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - Mx[h]);
          Lm[h] = fmaf(cf, ml.y, Lm[h]);
          O[h] = fmaf(cf, ov[i][h], O[h]);
        }
      }
    }
    named_barrier_sync(2, NET);  // mlb is reused by the next batch
  }
#pragma unroll
  for (int h = 0; h < G; ++h)
    if (h < rows)
      out[(obase + (size_t)(h >> lg_gh) * n_q + (h & ((1 << lg_gh) - 1))) * kHeadDim + e] =
          __float2bfloat16_rn(O[h] / Lm[h]);
}

template <int G, int BS, bool FP8>
__global__ void __launch_bounds__(kThreads<FP8>, 1) paged_attention_kernel(const AttnParams p) {
  using L = Lay<FP8>;
  constexpr int SB = TOK / BS;
  constexpr uint32_t IDESC_QK = instr_desc(false, false);
  constexpr uint32_t IDESC_QK8 = instr_desc_e4m3();
  constexpr uint32_t IDESC_PV = instr_desc(true, true);
  constexpr uint32_t IDESC_PV16 = instr_desc(true, true, false);  // f16 V and P
  // G: query rows per unit (heads per KV head x query tokens), padded to a
  // power of two; the 8-bit kernel keeps its query split in rows h and 8 + h.
  static_assert(G >= 1 && G <= (FP8 ? 8 : RMAX) && TOK % BS == 0 && BS % 8 == 0 && SB <= 32,
                "shape");

  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
  uint64_t *full_k = bars;                 // [NSK]
  uint64_t *empty_k = full_k + L::NSK;     // [NSK]
  uint64_t *full_v = empty_k + L::NSK;     // [NSV]
  uint64_t *empty_v = full_v + L::NSV;     // [NSV]
  uint64_t *s_full = empty_v + L::NSV;     // [NSB]
  uint64_t *s_free = s_full + NSB;         // [NSB]
  uint64_t *p_full = s_free + NSB;         // [2]
  uint64_t *p_free = p_full + 2;        // [2]
  uint64_t *o_full = p_free + 2;        // [2]
  uint64_t *o_free = o_full + 2;        // [2]
  uint64_t *m_ready = o_free + 2;       // [NSB]
  uint64_t *q_ready = m_ready + NSB;    // [2] per Q buffer
  uint64_t *q_free = q_ready + 2;       // [2] per Q buffer
  uint64_t *done = q_free + 2;          // [2] one per MMA issuer
  uint64_t *seg_done = done + 2;        // [2] softmax -> epilogue, per segment parity
  uint64_t *vb_full = seg_done + 2;     // [2] 8-bit: V converters -> p.v, by stage parity
  float *red = reinterpret_cast<float *>(smem + L::OFF_RED);
  float *lred = reinterpret_cast<float *>(smem + L::OFF_LRED);
  float *mref = reinterpret_cast<float *>(smem + L::OFF_MREF);
  float *qscale = reinterpret_cast<float *>(smem + L::OFF_QS);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 24);  // WaitCtl
  volatile int *flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 8);         // [3]
  int *nmax_slot = reinterpret_cast<int *>(smem + L::OFF_MISC + 20);
  volatile int *stage_mask = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 40);  // [8]
  volatile int *vmask = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 72);       // [NSV]
  int *over_flag = reinterpret_cast<int *>(smem + L::OFF_MISC + 96);  // [2][4] softmax votes
  int *pre = reinterpret_cast<int *>(smem + L::OFF_PRE);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Launched with programmatic stream serialization: the previous kernel of
  // the stream may still run.  Unless it is known to write only the caches,
  // wait for it before reading anything.
  if (!p.wait_late) pdl_wait();
  // Whole-unit guess: with no more units than CTAs, CTA c most likely
  // streams unit c from its first block.  The K producer warp reads that
  // unit's first table entries now and, after the prologue's first barrier,
  // asks L2 for its first stages, so that HBM works while the prologue runs
  // -- for units at least four times longer than that (batch 16 x 8192: a
  // step 1.8 us shorter; on units of 32 blocks it cost 0.6 us).  A hint: a
  // wrong guess only costs the prefetched bytes.
  const bool pf_unit = p.prefetch_units && warp == WARP_KP && (int)blockIdx.x < p.B * p.n_kv;
  int pf_ctx = 0, pf_blk = -1;
  if (pf_unit) {
    const int b = (int)blockIdx.x / p.n_kv, j = start_block(p, b) + lane;
    pf_ctx = __ldg(p.ctx + b);
    if (lane < kPrefetchBlocks<BS> && j >= 0 && j < p.MB)
      pf_blk = __ldg(p.tables + (size_t)b * p.MB + j);
  }

  if (tid == 0) {
    // 8-bit cache: the whole q.k^T warp hands each stage's key scales to
    // the softmax through m_ready; the softmax warps release a Q buffer once
    // they hold its scales, and the V converter warps release the V slots.
    for (int i = 0; i < L::NSK; ++i) {
      mbar_init(&full_k[i], 1);
      mbar_init(&empty_k[i], 1);
    }
    for (int i = 0; i < L::NSV; ++i) {
      mbar_init(&full_v[i], 1);
      mbar_init(&empty_v[i], FP8 ? NCVT : 1);
    }
    for (int i = 0; i < NSB; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 4);
      mbar_init(&m_ready[i], FP8 ? 32 : 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], 4);
      mbar_init(&p_free[i], 1);
      mbar_init(&o_full[i], 1);
      mbar_init(&o_free[i], 4);
      mbar_init(&done[i], 1);
      mbar_init(&seg_done[i], 4);
      mbar_init(&vb_full[i], NCVT);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_ready[i], 1);
      mbar_init(&q_free[i], FP8 ? 1 + 4 : 1);
    }
    mbar_init_fence();
    init_wait_ctl(smem + L::OFF_MISC + 24, p.wait_limit_ns);
  }
  // Q pad rows and P pad columns stay zero for the whole kernel.
  {
    uint4 *z = reinterpret_cast<uint4 *>(smem + L::OFF_Q);
    for (int i = tid; i < (2 * L::Q_BYTES + 2 * P_BYTES) / 16; i += kThreads<FP8>)
      z[i] = make_uint4(0, 0, 0, 0);
  }
  // Blocks per sequence, then an exclusive prefix over the batch.
  const int max_tokens = p.MB * BS;
  bool bad_ctx = false;
  for (int b = tid; b < p.B; b += kThreads<FP8>) {
    const int c = p.ctx[b];
    int nb = 0;
    // (a multi-query call's T new tokens are the last T of the context)
    if (c >= max(1, p.T) && c <= max_tokens) nb = (c + BS - 1) / BS; else bad_ctx = true;
    const int s0 = start_block(p, b);
    if (s0 < 0 || (nb > 0 && s0 >= nb)) bad_ctx = true;  // the suffix must keep >= 1 block
    pre[b + 1] = (s0 >= 0 && s0 < nb) ? nb - s0 + kSegCost<BS> : 0;
  }
  if (bad_ctx && blockIdx.x == 0) atomicOr(p.err, PGD_DEVERR_BAD_CONTEXT);
  if (warp == WARP_QK) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_proxy_async();
  __syncthreads();
  if (pf_unit) {
    const int b = (int)blockIdx.x / p.n_kv, g = (int)blockIdx.x % p.n_kv;
    const int nb = (pf_ctx >= 1 && pf_ctx <= max_tokens)
                       ? (pf_ctx + BS - 1) / BS - start_block(p, b) : 0;
    if (nb >= 4 * kPrefetchBlocks<BS> && lane < kPrefetchBlocks<BS> &&
        (unsigned)pf_blk < (unsigned)p.NB) {
      constexpr uint32_t TILE = (BS / 8) * L::GROUP;
      const size_t off = ((size_t)pf_blk * p.n_kv + g) * TILE;
      bulk_prefetch_l2(p.k_cache + off, TILE);
      bulk_prefetch_l2(p.v_cache + off, TILE);
    }
  }
  if (warp == 0) {
    int carry = 0, longest = 0;
    for (int base = 0; base < p.B; base += 32) {
      const int i = base + lane;
      int v = (i < p.B) ? pre[i + 1] : 0;
      longest = max(longest, v);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFullMask, v, o);
        if (lane >= o) v += n;
      }
      if (i < p.B) pre[i + 1] = v + carry;
      carry += __shfl_sync(kFullMask, v, 31);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) longest = max(longest, __shfl_xor_sync(kFullMask, longest, o));
    if (lane == 0) {
      pre[0] = 0;
      *nmax_slot = longest;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  Schedule sc;
  sc.X = (long long)p.n_kv * pre[p.B];
  sc.pre = pre;
  sc.n_kv = p.n_kv;
  sc.ov = kSegCost<BS>;
  sc.P = sc.X < (long long)gridDim.x ? sc.X : (long long)gridDim.x;
  sc.units = false;
  if (p.auto_split && sc.X > 0) {
    // The job's time in blocks of HBM streaming time: for P balanced cuts,
    // the longest part at one CTA's share of HBM (or the whole job at the
    // HBM rate), then the merge of a unit's parts -- a fixed cost and one per
    // part, so a small job takes fewer, longer parts: X share / P + m1 P / U
    // is least near P = sqrt(share X U / m1), within the grid.  Whole units
    // (the longest at one CTA's share) when they fit in the grid and cost no
    // more.
    const long long U = (long long)p.B * p.n_kv, nmax = *nmax_slot;
    constexpr long long kBlockBytes = 2ll * (BS / 8) * L::GROUP;  // K and V of one block
    constexpr long long m0 = kMergeFixedBytes / kBlockBytes, m1 = kMergePartBytes / kBlockBytes;
    const long long grid = (long long)gridDim.x;
    long long P = (long long)sqrtf((float)kCtaShare<FP8> * (float)sc.X * (float)U / (float)m1);
    P = max(1ll, min(P, sc.P));
    const long long cost_cut =
        max((sc.X + P - 1) / P * kCtaShare<FP8>, sc.X) + m0 + m1 * ((P + U - 1) / U);
    sc.P = P;
    if (U <= grid) {
      const long long cost_units = max(nmax * kCtaShare<FP8>, sc.X);
      if (cost_units <= cost_cut) {
        sc.units = true;
        sc.P = U;
      }
    }
  }

  if (warp == WARP_KP) {
    produce<G, BS, FP8, true>(p, sc, p.k_cache, smem + L::OFF_K, full_k, empty_k, stage_mask,
                              smem + L::OFF_Q, qscale, q_ready, q_free, abort_flag, lane);
  } else if (warp == WARP_VP) {
    produce<G, BS, FP8, false>(p, sc, p.v_cache, smem + L::OFF_V, full_v, empty_v, vmask,
                               nullptr, nullptr, nullptr, nullptr, abort_flag, lane);
  } else if (warp == WARP_QK) {
    // ---------------------------------------------------- q.k^T issuer
    // (one lane issues; under the 8-bit cache the whole warp first copies the
    // stage's key scales into their ring, so that the K slot frees as soon
    // as its q.k^T has completed)
    if (FP8 || lane == 0) {
      const uint32_t q_base = smem_addr(smem + L::OFF_Q);
      SegCursor cur(sc);
      Segment sg;
      int s = 0, k = 0;
      while (cur.next(sc, p.B, sg)) {
        const int nstages = (sg.n + SB - 1) / SB;
        // Q of segment k is in buffer k & 1 (written by the K producer); it is
        // rewritten for segment k + 2 only after q_free signals that every
        // q.k^T of segment k has completed.
        if (lane == 0)
          wait_or_abort(&q_ready[k & 1], (uint32_t)(k >> 1) & 1u, abort_flag, p.err);
        const uint32_t q_seg = q_base + (uint32_t)((k & 1) * L::Q_BYTES);
        for (int st = 0; st < nstages; ++st, ++s) {
          const int slot = s % L::NSK, sb = s % NSB;
          // (the key-scale slot s % NKS was last read for stage s - NKS, in
          // an earlier softmax iteration than the one that freed S of s - NSB)
          if (FP8 || lane == 0) {
            wait_or_abort(&full_k[slot], (uint32_t)(s / L::NSK) & 1u, abort_flag, p.err);
            wait_or_abort(&s_free[sb], ((uint32_t)(s / NSB) & 1u) ^ 1u, abort_flag, p.err);
          }
          if constexpr (FP8) {
            // 16 token groups x 32 B of scales: lane l takes half l & 1 of group l >> 1
            const int g = lane >> 1, hf = lane & 1;
            const uint4 v = *reinterpret_cast<const uint4 *>(
                smem + L::OFF_K + slot * L::STAGE + g * L::GROUP + 1024 + hf * 16);
            *reinterpret_cast<uint4 *>(smem + L::OFF_KS + (s % L::NKS) * (TOK * 4) + g * 32 +
                                       hf * 16) = v;
            __syncwarp();
          }
          tc_fence_after();
          if (lane == 0 && !*abort_flag) {
            const uint32_t dS = tmem + col_s(sb);
            const uint32_t k_st = smem_addr(smem + L::OFF_K + slot * L::STAGE);
            if constexpr (FP8) {
              // E4M3, K = 32 per MMA: K core matrices 128 B apart along d,
              // token groups 1056 B apart; Q rows 8 apart at 1024 B.  A k-step
              // moves both by two core matrices (256 B).
              const uint64_t kd = smem_desc(k_st, 128, L::GROUP, 0);
              const uint64_t qd = smem_desc(q_seg, 128, 1024, 0);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_e4m3(dS, kd + (uint64_t)(kk * 16), qd + (uint64_t)(kk * 16), IDESC_QK8,
                          kk > 0 ? 1u : 0u);
            } else {
              // Descriptors are built once; a k-step only moves the start
              // address (the low field, in 16-byte units): K by 256 B, Q by
              // 32 B within a 128-byte swizzle row and by 2048 B to the second
              // half.
              const uint64_t kd = smem_desc(k_st, 128, 2048, 0);
              const uint64_t qd = smem_desc(q_seg, 16, 1024, 2);
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                umma_bf16(dS, kd + (uint64_t)(kk * 16),
                          qd + (uint64_t)((kk >> 2) * 128 + (kk & 3) * 2), IDESC_QK,
                          kk > 0 ? 1u : 0u);
            }
          }
          if (lane == 0) {
            umma_commit(&s_full[sb]);
            umma_commit(&empty_k[slot]);
          }
          // Hand the stage's invalid-block mask (written by the K producer
          // before it armed full_k, which lane 0 acquired) and, under the
          // 8-bit cache, its key scales (each lane its own) to the softmax.
          if (FP8 || lane == 0) mbar_arrive(&m_ready[sb]);
        }
        if (lane == 0) umma_commit(&q_free[k & 1]);  // Q buffer reusable once these complete
        ++k;
      }
      // every MMA has completed before tensor memory is released
      if (lane == 0 && s > 0) {
        umma_commit(&done[0]);
        mbar_wait_bounded(&done[0], 0);
      }
    }
  } else if (warp == WARP_PV) {
    // ------------------------------------------------------- p.v issuer
    if (lane == 0) {
      SegCursor cur(sc);
      Segment sg;
      int s = 0, k = 0;
      while (cur.next(sc, p.B, sg)) {
        const int ctx_b = __ldg(p.ctx + sg.b);
        const int sb0 = start_block(p, sg.b);
        const int nstages = (sg.n + SB - 1) / SB;
        const int ob = k & 1;
        for (int st = 0; st < nstages; ++st, ++s) {
          const int slot = s % L::NSV, sb = s & 1;
          // k-steps past the sequence's last token are not issued (their
          // rows hold no valid token and were never zeroed)
          const int nb = min(SB, sg.n - st * SB);
          int nvalid = nb * BS;
          if (sg.j0 + st * SB + nb == sg.nblk) nvalid -= (sg.nblk + sb0) * BS - ctx_b;
          const int nkt = min(8, max(1, (nvalid + 15) >> 4));
          wait_or_abort(&p_full[sb], (uint32_t)(s >> 1) & 1u, abort_flag, p.err);
          if (FP8)  // V dequantised into the f16 buffer of parity sb
            wait_or_abort(&vb_full[sb], (uint32_t)(s >> 1) & 1u, abort_flag, p.err);
          else
            wait_or_abort(&full_v[slot], (uint32_t)(s / L::NSV) & 1u, abort_flag, p.err);
          if (st == 0)
            wait_or_abort(&o_free[ob], ((uint32_t)(k >> 1) & 1u) ^ 1u, abort_flag, p.err);
          tc_fence_after();
          if (!*abort_flag) {
            // 16 tokens per k-step: V moves by 4096 B, P by 512 B.
            const uint64_t vd = smem_desc(
                smem_addr(smem + (FP8 ? L::OFF_VB + sb * (TOK * 256) : L::OFF_V + slot * L::STAGE)),
                2048, 128, 0);
            const uint64_t pd = smem_desc(smem_addr(smem + L::OFF_P + sb * P_BYTES), 256, 128, 0);
            const uint32_t dO = tmem + col_o(ob);
            const uint32_t acc0 = st > 0 ? 1u : 0u;
#pragma unroll
            for (int kt = 0; kt < 8; ++kt)
              if (kt < nkt)
                umma_bf16(dO, vd + (uint64_t)(kt * 256), pd + (uint64_t)(kt * 32),
                          FP8 ? IDESC_PV16 : IDESC_PV, kt > 0 ? 1u : acc0);
          }
          if (!FP8) umma_commit(&empty_v[slot]);
          umma_commit(&p_free[sb]);  // P (and converted V) of parity sb reusable
          if (st + 1 == nstages) umma_commit(&o_full[ob]);
        }
        ++k;
      }
      if (s > 0) {
        umma_commit(&done[1]);
        mbar_wait_bounded(&done[1], 0);
      }
    }
  } else if (warp < 4) {
    // ----------------------------------------------------------- softmax
    // Two MMA stages (256 tokens) per iteration: one tile maximum, one named
    // barrier and one rescale decision serve both, so the fixed latency of a
    // step (waits, tensor-memory loads, barrier, fences) is paid once per 256
    // tokens.  Thread t owns token row t of each of the two stages.  (One
    // stage per iteration for 16 query rows.)
    const int t = tid;  // 0..127: token row of S
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    constexpr int NCT = 128;
    constexpr int NSC = (FP8 || G > 8) ? 16 : 8;  // S columns per stage (8-bit: high and low parts)
    // MMA stages per iteration: two, or one for 16 query rows (whose per-row
    // arrays would not fit the register budget twice over)
    constexpr int SPI = G > 8 ? 1 : 2;
    auto stage_max = [](const float (&x)[SPI][G], int h) {
      float m = x[0][h];
#pragma unroll
      for (int u = 1; u < SPI; ++u) m = fmaxf(m, x[u][h]);
      return m;
    };
    // Query token of each column, for the causal mask among a multi-query
    // call's T new tokens (token a of the context is seen by column h iff
    // a - (ctx - T) <= tok[h]); padding columns see nothing.
    int tok[G];
#pragma unroll
    for (int h = 0; h < G; ++h) tok[h] = h < p.rows ? (h >> p.lg_gh) : -(1 << 30);
    SegCursor cur(sc);
    Segment sg, nsg;
    int s = 0, k = 0, it = 0;
    // each segment's context length and first block, loaded a segment ahead
    bool have = cur.next(sc, p.B, sg);
    int ctx_b = have ? __ldg(p.ctx + sg.b) : 0, sb0 = have ? start_block(p, sg.b) : 0;
    while (have) {
      const bool have_next = cur.next(sc, p.B, nsg);
      const int ctx_n = have_next ? __ldg(p.ctx + nsg.b) : 0;
      const int sb0_n = have_next ? start_block(p, nsg.b) : 0;
      const int nstages = (sg.n + SB - 1) / SB;
      const int ob = k & 1;
      float m_ref[G], l_part[G];
      float qsc[G];  // 8-bit cache: Q scale of each head times scale * log2(e)
#pragma unroll
      for (int h = 0; h < G; ++h) { m_ref[h] = -INFINITY; l_part[h] = 0.f; qsc[h] = 0.f; }

      for (int st = 0; st < nstages; st += SPI, ++it) {
        const int n2 = min(SPI, nstages - st);  // stages in this iteration
        bool valid[SPI] = {};
        int msk[SPI] = {};
        int lim[SPI] = {};  // rows p.v reads: the valid length rounded up to 16
        int epos[SPI] = {};  // this row's token minus the first new token (T > 1)
        // Invalid-block mask of each stage: the K producer wrote it before
        // arming full_k; the q.k^T issuer acquired full_k and then released
        // m_ready.  (Waiting on full_k here could alias: a K stage is freed
        // after its q.k^T alone, so full_k may run two phases ahead.)  The
        // 8-entry mask ring cannot move on before these stages free their S
        // buffers.
#pragma unroll
        for (int u = 0; u < SPI; ++u) {
          if (u < n2) {
            const int su = s + u, sbu = su % NSB;
            wait_or_abort(&s_full[sbu], (uint32_t)(su / NSB) & 1u, abort_flag, p.err);
            wait_or_abort(&m_ready[sbu], (uint32_t)(su / NSB) & 1u, abort_flag, p.err);
            msk[u] = stage_mask[su & 7];
            const int nb = min(SB, sg.n - (st + u) * SB);
            int nvalid = nb * BS;
            if (sg.j0 + (st + u) * SB + nb == sg.nblk)  // the sequence's last block
              nvalid -= (sg.nblk + sb0) * BS - ctx_b;
            valid[u] = (t < nvalid) && !((msk[u] >> (t / BS)) & 1);
            lim[u] = (nvalid + 15) & ~15;
            epos[u] = (sb0 + sg.j0 + (st + u) * SB) * BS + t - (ctx_b - p.T);
          }
        }
        tc_fence_after();
        uint32_t sv[SPI][NSC];
#pragma unroll
        for (int u = 0; u < SPI; ++u) {
          if (u < n2) {
            const uint32_t a0 = tmem + lane_base + col_s((s + u) % NSB);
            tmem_ld8_async(a0, sv[u]);
            if (NSC > 8) tmem_ld8_async(a0 + 8, sv[u] + 8);
          }
        }
#pragma unroll
        for (int u = 0; u < SPI; ++u) {
          if (u < n2) {
            tmem_wait8(sv[u]);
            if (NSC > 8) tmem_wait8(sv[u] + 8);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&s_free[s % NSB]);
          if (n2 > 1) mbar_arrive(&s_free[(s + 1) % NSB]);
        }

        float sc_[SPI][G];
        if constexpr (FP8) {
          // Key scale of each token (from the ring the q.k^T warp filled
          // before m_ready), and at a segment's first stage the Q scales (the
          // K producer wrote them before q_ready, which the q.k^T issuer
          // acquired before m_ready).
          float ks[SPI] = {};
#pragma unroll
          for (int u = 0; u < SPI; ++u)
            if (u < n2)
              ks[u] = reinterpret_cast<const float *>(
                  smem + L::OFF_KS)[((s + u) % L::NKS) * TOK + t];
          if (st == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) qsc[h] = qscale[(k & 1) * 8 + h] * p.qk_scale_log2;
          }
          __syncwarp();
          if (lane == 0 && st == 0) mbar_arrive(&q_free[k & 1]);
#pragma unroll
          for (int u = 0; u < SPI; ++u)
#pragma unroll
            for (int h = 0; h < G; ++h)
              sc_[u][h] = valid[u] ? (__uint_as_float(sv[u][h]) + __uint_as_float(sv[u][8 + h])) *
                                         (qsc[h] * ks[u])
                                   : -INFINITY;
        } else {
#pragma unroll
          for (int u = 0; u < SPI; ++u)
#pragma unroll
            for (int h = 0; h < G; ++h)
              sc_[u][h] = (valid[u] && tok[h] >= epos[u])
                              ? __uint_as_float(sv[u][h]) * p.qk_scale_log2
                              : -INFINITY;
        }

        // Does any score of the SPI x 128 rows exceed its head's reference by
        // more than 2^8?  One vote per warp (rarely yes); only then are the
        // exact tile maxima reduced and the reference moved.  A segment's
        // first iteration, where the reference is -inf, moves it unasked.
        const int rb = it & 1;
        bool move = true;  // (a segment's first iteration always moves it)
        if (st > 0) {
          bool over = false;
#pragma unroll
          for (int h = 0; h < G; ++h)
            over |= stage_max(sc_, h) > m_ref[h] + kRescaleLog2;
          const bool wover = __any_sync(kFullMask, over);
          if (lane == 0) over_flag[rb * 4 + warp] = wover ? 1 : 0;
          named_barrier_sync(1, NCT);
          const int4 votes = *reinterpret_cast<const int4 *>(over_flag + rb * 4);
          move = (votes.x | votes.y | votes.z | votes.w) != 0;
        }
        if (move) {
          float v2[G];
#pragma unroll
          for (int h = 0; h < G; ++h) v2[h] = stage_max(sc_, h);
          const float wm = warp_reduce_heads<G, true>(v2, lane);
          constexpr int SH = 5 - kLog2<G>;  // lanes per head after the reduction
          if ((lane & ((1 << SH) - 1)) == 0) red[(rb * 4 + warp) * RMAX + (lane >> SH)] = wm;
          named_barrier_sync(1, NCT);
          constexpr int G4 = (G + 3) / 4;  // float4s of maxima per warp
          float tmax[4 * G4];
#pragma unroll
          for (int h = 0; h < 4 * G4; ++h) tmax[h] = -INFINITY;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const float4 *src = reinterpret_cast<const float4 *>(red + (rb * 4 + w) * RMAX);
#pragma unroll
            for (int j = 0; j < G4; ++j) {
              const float4 a = src[j];
              tmax[4 * j + 0] = fmaxf(tmax[4 * j + 0], a.x);
              tmax[4 * j + 1] = fmaxf(tmax[4 * j + 1], a.y);
              tmax[4 * j + 2] = fmaxf(tmax[4 * j + 2], a.z);
              tmax[4 * j + 3] = fmaxf(tmax[4 * j + 3], a.w);
            }
          }
          constexpr int GO = G > 8 ? 16 : 8;  // O columns held per TMEM lane
          float alpha[GO];
#pragma unroll
          for (int h = 0; h < GO; ++h) alpha[h] = 1.f;
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float mn = fmaxf(m_ref[h], tmax[h]);
            alpha[h] = (m_ref[h] == -INFINITY) ? 0.f : exp2f(m_ref[h] - mn);
            m_ref[h] = mn;
            l_part[h] *= alpha[h];
          }
          if (st > 0) {
            // rescale O in tensor memory once the previous p.v has completed
            wait_or_abort(&p_free[(s - 1) & 1], (uint32_t)((s - 1) >> 1) & 1u, abort_flag, p.err);
            tc_fence_after();
#pragma unroll
            for (int c8 = 0; c8 < GO / 8; ++c8) {
              float ov[8];
              tmem_ld8(tmem + lane_base + col_o(ob) + 8 * c8, ov);
#pragma unroll
              for (int h = 0; h < 8; ++h) ov[h] *= alpha[8 * c8 + h];
              tmem_st8(tmem + lane_base + col_o(ob) + 8 * c8, ov);
            }
            tc_fence_before();
          }
        }
        // probabilities, rounded as the tensor cores will see them (bf16, or
        // f16 beside the 8-bit cache's f16 V; p <= 2^8 either way)
#pragma unroll
        for (int u = 0; u < SPI; ++u) {
          if (u < n2) {
            const int su = s + u, pbuf = su & 1;
            uint32_t packed[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if constexpr (!FP8 && G >= 2) {
#pragma unroll
              for (int h = 0; h < G; h += 2) {
                const float p0 =
                    (valid[u] && tok[h] >= epos[u]) ? exp2_approx(sc_[u][h] - m_ref[h]) : 0.f;
                const float p1 = (valid[u] && tok[h + 1] >= epos[u])
                                     ? exp2_approx(sc_[u][h + 1] - m_ref[h + 1])
                                     : 0.f;
                const __nv_bfloat162 pb2 = __floats2bfloat162_rn(p0, p1);
                const float2 back = __bfloat1622float2(pb2);
                l_part[h] += back.x;
                l_part[h + 1] += back.y;
                packed[h >> 1] = *reinterpret_cast<const uint32_t *>(&pb2);
              }
            } else if constexpr (FP8 && G >= 2) {
              // (two heads per conversion either way: under the 8-bit cache
              // these warps share the SM's sub-partitions with the V
              // converters, whose conversions dominate the issue slots)
#pragma unroll
              for (int h = 0; h < G; h += 2) {
                const float p0 =
                    (valid[u] && tok[h] >= epos[u]) ? exp2_approx(sc_[u][h] - m_ref[h]) : 0.f;
                const float p1 = (valid[u] && tok[h + 1] >= epos[u])
                                     ? exp2_approx(sc_[u][h + 1] - m_ref[h + 1])
                                     : 0.f;
                const __half2 ph = __floats2half2_rn(p0, p1);
                const float2 back = __half22float2(ph);
                l_part[h] += back.x;
                l_part[h + 1] += back.y;
                packed[h >> 1] = *reinterpret_cast<const uint32_t *>(&ph);
              }
            } else
#pragma unroll
            for (int h = 0; h < G; ++h) {
              const float pv = !(valid[u] && tok[h] >= epos[u]) ? 0.f
                               : FP8 ? exp2_approx(sc_[u][h] - m_ref[h])
                                     : exp2f(sc_[u][h] - m_ref[h]);
              uint16_t bits;
              if constexpr (FP8) {
                const __half ph = __float2half_rn(pv);
                l_part[h] += __half2float(ph);
                bits = __half_as_ushort(ph);
              } else {
                const __nv_bfloat16 pb = __float2bfloat16_rn(pv);
                l_part[h] += __bfloat162float(pb);
                bits = __bfloat16_as_ushort(pb);
              }
              packed[h >> 1] |= (uint32_t)bits << ((h & 1) * 16);
            }
            wait_or_abort(&p_free[pbuf], ((uint32_t)(su >> 1) & 1u) ^ 1u, abort_flag, p.err);
            *reinterpret_cast<uint4 *>(smem + L::OFF_P + pbuf * P_BYTES + (t >> 3) * 256 +
                                       (t & 7) * 16) =
                make_uint4(packed[0], packed[1], packed[2], packed[3]);
            if (G > 8)  // rows 8..15: the second 8-column group of the MN-major P
              *reinterpret_cast<uint4 *>(smem + L::OFF_P + pbuf * P_BYTES + (t >> 3) * 256 +
                                         128 + (t & 7) * 16) =
                  make_uint4(packed[4], packed[5], packed[6], packed[7]);
            if (!FP8 && !valid[u] && t < lim[u]) {
              // rows that p.v reads but that are not valid tokens (the tail
              // of the last block, a block whose id was bad) must not feed
              // NaN/Inf into it: zero them once their copy has landed
              const int vslot = su % L::NSV;
              wait_or_abort(&full_v[vslot], (uint32_t)(su / L::NSV) & 1u, abort_flag, p.err);
              uint4 *vrow = reinterpret_cast<uint4 *>(smem + L::OFF_V + vslot * L::STAGE +
                                                      (t >> 3) * 2048 + (t & 7) * 16);
#pragma unroll
              for (int c = 0; c < 16; ++c) vrow[c * 8] = make_uint4(0, 0, 0, 0);
            }
          }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&p_full[s & 1]);
          if (n2 > 1) mbar_arrive(&p_full[(s + 1) & 1]);
        }
        s += n2;
      }

      // ---- end of segment: hand the segment's reference maxima and per-warp
      // sums to the epilogue warps.
      // lred/mref[ob] were last read by the epilogue of segment k - 2, which
      // then released O buffer ob
      wait_or_abort(&o_free[ob], ((uint32_t)(k >> 1) & 1u) ^ 1u, abort_flag, p.err);
      {
        const float ws = warp_reduce_heads<G, false>(l_part, lane);
        constexpr int SH = 5 - kLog2<G>;
        if ((lane & ((1 << SH) - 1)) == 0) lred[(ob * 4 + warp) * RMAX + (lane >> SH)] = ws;
      }
      if (t == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) mref[ob * RMAX + h] = m_ref[h];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&seg_done[ob]);
      ++k;
      sg = nsg;
      ctx_b = ctx_n;
      sb0 = sb0_n;
      have = have_next;
    }
  } else if (warp < WARP_CVT) {
    // ---------------------------------------------------------- epilogue
    const int e = tid - 32 * WARP_EPI;  // 0..127: head-dim row of O
    const int ew = warp - WARP_EPI;     // TMEM lane quadrant
    const uint32_t lane_base = (uint32_t)(ew * 32) << 16;
    constexpr int NET = 128;
    SegCursor cur(sc);
    Segment sg;
    const int part = (int)blockIdx.x;
    int k = 0;
    while (cur.next(sc, p.B, sg)) {
      const int ob = k & 1;
      const int unit = sg.b * p.n_kv + sg.g;
      wait_or_abort(&seg_done[ob], (uint32_t)(k >> 1) & 1u, abort_flag, p.err);
      float Lsum[G], M[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        Lsum[h] = (lred[(ob * 4 + 0) * RMAX + h] + lred[(ob * 4 + 1) * RMAX + h]) +
               (lred[(ob * 4 + 2) * RMAX + h] + lred[(ob * 4 + 3) * RMAX + h]);
        M[h] = mref[ob * RMAX + h];
      }
      wait_or_abort(&o_full[ob], (uint32_t)(k >> 1) & 1u, abort_flag, p.err);
      tc_fence_after();
      constexpr int GO = G > 8 ? 16 : 8;
      float ov[GO];
#pragma unroll
      for (int c8 = 0; c8 < GO / 8; ++c8)
        tmem_ld8(tmem + lane_base + col_o(ob) + 8 * c8, *reinterpret_cast<float(*)[8]>(ov + 8 * c8));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free[ob]);

      // a cascade unit with a shared prefix always merges: its prefix
      // partial states come from the shared-prefix pass
      const bool has_prefix = p.pre_ml != nullptr && start_block(p, sg.b) > 0;
      const bool whole = sg.j0 == 0 && sg.n == sg.nblk && !has_prefix;
      // parts holding the unit's first and last blocks
      const long long c_first = sc.units ? (long long)part : sc.part_of(sg.ucs + sc.ov);
      const long long c_last = sc.units ? (long long)part : sc.part_of(sg.uce - 1);
      const size_t obase = q_index(p, sg.b, sg.g, 0);  // output row of query row 0
      if (whole) {
#pragma unroll
        for (int h = 0; h < G; ++h)
          if (h < p.rows)
            p.out[(obase + (size_t)(h >> p.lg_gh) * p.n_q + (h & ((1 << p.lg_gh) - 1))) *
                      kHeadDim + e] = __float2bfloat16_rn(ov[h] / Lsum[h]);
      } else if (has_prefix) {
        // cascade unit: the combine kernel merges all its parts; record
        // where they are (every part writes the same pair)
        const size_t srow = ((size_t)unit + (size_t)part) * G;
#pragma unroll
        for (int h = 0; h < G; ++h) p.part_o[(srow + h) * kHeadDim + e] = ov[h];
#pragma unroll
        for (int h = 0; h < G; ++h)
          if (e == h)
            *reinterpret_cast<float2 *>(p.part_ml + (srow + h) * 2) = make_float2(M[h], Lsum[h]);
        if (e == 0) p.part_info[unit] = make_int2((int)c_first, (int)(c_last - c_first + 1));
      } else {
        const size_t srow = ((size_t)unit + (size_t)part) * G;
#pragma unroll
        for (int h = 0; h < G; ++h) p.part_o[(srow + h) * kHeadDim + e] = ov[h];
#pragma unroll
        for (int h = 0; h < G; ++h)
          if (e == h)
            *reinterpret_cast<float2 *>(p.part_ml + (srow + h) * 2) = make_float2(M[h], Lsum[h]);
        // publish this part; the last part of the unit to arrive merges all.
        // The barrier orders the 128 threads' stores before thread 0's
        // atomic, whose release makes them visible with it and whose acquire
        // (in the last arriver) the other parts' stores; the second barrier
        // passes that on to the threads that read them.
        named_barrier_sync(2, NET);
        if (e == 0) {
          // (whole-unit parts: the unit's only part is this CTA's)
          const int n_parts = (int)(c_last - c_first + 1);
          const int before = atomic_add_acq_rel_gpu(p.counters + unit, 1);
          const int last = (before == n_parts - 1);
          if (last) atomicExch(p.counters + unit, 0);  // ready for the next call
          flag[0] = last;
          flag[1] = (int)c_first;
          flag[2] = n_parts;
        }
        named_barrier_sync(2, NET);
        if (flag[0]) {
          merge_parts<G, FP8>(p.part_o, p.part_ml, p.out, unit, flag[1], flag[2], obase, p.lg_gh,
                              p.n_q, p.rows, e, reinterpret_cast<float2 *>(smem + L::OFF_MERGE));
        }
        named_barrier_sync(2, NET);  // flags are reused by the next segment
      }
      ++k;
    }
  } else if constexpr (FP8) {
    // ------------------------------------------------ V converters (8-bit)
    // NPART threads per token row t of each stage, each a part of the row:
    // they dequantise the codes (code * scale, f16) into the p.v operand of
    // parity s & 1 once the p.v that last read that buffer has completed,
    // and zero rows that are not valid tokens (past the context, or in a
    // block whose id was bad).
    constexpr int NPART = NCVT * 32 / TOK, NCH = 8 / NPART;  // 16-dim chunks per thread
    const int ct = tid - 32 * WARP_CVT;
    const int t = ct & (TOK - 1), part = ct / TOK;
    SegCursor cur(sc);
    Segment sg;
    int s = 0;
    while (cur.next(sc, p.B, sg)) {
      const int ctx_b = __ldg(p.ctx + sg.b);
      const int sb0 = start_block(p, sg.b);
      const int nstages = (sg.n + SB - 1) / SB;
      for (int st = 0; st < nstages; ++st, ++s) {
        const int vslot = s % L::NSV, sb = s & 1;
        const int nb = min(SB, sg.n - st * SB);
        int nvalid = nb * BS;
        if (sg.j0 + st * SB + nb == sg.nblk)  // the sequence's last block
          nvalid -= (sg.nblk + sb0) * BS - ctx_b;
        wait_or_abort(&full_v[vslot], (uint32_t)(s / L::NSV) & 1u, abort_flag, p.err);
        const bool valid = (t < nvalid) && !((vmask[vslot] >> (t / BS)) & 1);
        const unsigned char *grp = smem + L::OFF_V + vslot * L::STAGE + (t >> 3) * L::GROUP;
        const __half2 vs2 =
            __float2half2_rn(*reinterpret_cast<const float *>(grp + 1024 + (t & 7) * 4));
        uint4 codes[NCH];
#pragma unroll
        for (int i = 0; i < NCH; ++i)
          codes[i] = *reinterpret_cast<const uint4 *>(grp + (NCH * part + i) * 128 + (t & 7) * 16);
        wait_or_abort(&p_free[sb], ((uint32_t)(s >> 1) & 1u) ^ 1u, abort_flag, p.err);
        unsigned char *dst = smem + L::OFF_VB + sb * (TOK * 256) + (t >> 3) * 2048 + (t & 7) * 16;
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
          const int c = NCH * part + i;  // 16-dim chunk
          uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
          if (valid) e4m3x16_dequant_f16(codes[i], vs2, lo, hi);
          *reinterpret_cast<uint4 *>(dst + (2 * c) * 128) = lo;
          *reinterpret_cast<uint4 *>(dst + (2 * c + 1) * 128) = hi;
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&empty_v[vslot]);
          mbar_arrive(&vb_full[sb]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // (cascade: this grid completes only after the shared-prefix pass, so the
  // combine kernel that waits for it sees both passes' partial states.  The
  // wait comes after the barrier: a lane blocked in it would hold up the
  // lanes of its warp that still have work, like the issuing lane 0 of the
  // MMA warps.)
  if (p.wait_late == 2) pdl_wait();
  tc_fence_after();
  if (warp == WARP_QK) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// The dynamic shared-memory limit is raised once per device, to the size the
// largest accepted batch needs.
template <int G, int BS, bool FP8>
static cudaError_t ensure_smem_limit() {
  static volatile int done[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(paged_attention_kernel<G, BS, FP8>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem_bytes<FP8>(PGD_MAX_BATCH));
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = 1;
  return e;
}

template <int G, int BS, bool FP8>
static cudaError_t launch_cfg(const AttnParams &p, int grid, cudaStream_t stream) {
  cudaError_t e = ensure_smem_limit<G, BS, FP8>();
  if (e != cudaSuccess) return e;
  // Programmatic stream serialization: the CTAs may launch and run their
  // prologue while the previous kernel finishes (see pdl_wait above).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads<FP8>);
  cfg.dynamicSmemBytes = smem_bytes<FP8>(p.B);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, paged_attention_kernel<G, BS, FP8>, p);
}

template <int G, int BS, bool FP8>
static int occupancy_cfg(int B) {
  if (ensure_smem_limit<G, BS, FP8>() != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, paged_attention_kernel<G, BS, FP8>,
                                                    kThreads<FP8>, smem_bytes<FP8>(B)) !=
      cudaSuccess)
    return 0;
  return n;
}

}  // namespace tc

// Dispatch over the supported (G, block size) pairs for one kind of cache.
template <bool FP8>
int attention_ctas_per_sm_t(int G, int bs, int B) {
#define PGD_CASE(G_, BS_) \
  if (G == G_ && bs == BS_) return tc::occupancy_cfg<G_, BS_, FP8>(B);
  PGD_CASE(1, 16) PGD_CASE(2, 16) PGD_CASE(4, 16) PGD_CASE(8, 16)
  PGD_CASE(1, 32) PGD_CASE(2, 32) PGD_CASE(4, 32) PGD_CASE(8, 32)
  if constexpr (!FP8) {
    PGD_CASE(16, 16) PGD_CASE(16, 32)
  }
#undef PGD_CASE
  return 0;
}

template <bool FP8>
cudaError_t attention_launch_t(const AttnParams &p, int G, int bs, int grid,
                               cudaStream_t stream) {
#define PGD_CASE(G_, BS_) \
  if (G == G_ && bs == BS_) return tc::launch_cfg<G_, BS_, FP8>(p, grid, stream);
  PGD_CASE(1, 16) PGD_CASE(2, 16) PGD_CASE(4, 16) PGD_CASE(8, 16)
  PGD_CASE(1, 32) PGD_CASE(2, 32) PGD_CASE(4, 32) PGD_CASE(8, 32)
  if constexpr (!FP8) {
    PGD_CASE(16, 16) PGD_CASE(16, 32)
  }
#undef PGD_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pgd
