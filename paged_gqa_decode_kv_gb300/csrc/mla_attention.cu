// mla_attention.cu -- decode attention over an MLA latent cache (multi-head
// latent attention in its absorbed form), and the append of latent rows.
//
// "The math of Transformer inference", MLA section: per layer and token the
// cache holds the latent c_t (d_c = 512) and a decoupled RoPE key k_t^R
// (d_r = 64), 576 values shared by every head; with W^UK absorbed into the
// query and W^UV into the output projection, head h scores
//     s_t = scale * q_h . c_t          (q_h = [W_h^{UK T} q_h^C ; q_h^R], 576)
// and returns the 512-d latent  o_h = sum_t softmax(s)_t c_t[0 .. 512)
// ("LLM inference systems engineering", 2.8.2: the identities behind the
// absorption).  Decode is then MQA with G = n_h: one cache, all heads.
//
// On the tensor cores a CTA takes 64 heads of one sequence and all 512 output
// dims; q.c^T has the head rows on the MMA's M side, p.c is computed
// transposed, with the latent dims on M:
//   S[64 rows][64 tok]  = Q[64 rows][576] . C^T          (M = 64: A = Q, B = C, K-major)
//   O^T[128 d][64 rows] += V^T[128 d][16 tok] . P^T       (M = 128, one MMA per 128-dim
//                                                          block: A = the stage, MN-major;
//                                                          B = P, K-major)
// An MMA instruction costs about the larger of its math time (N / 2 cycles at
// M = 128 and at M = 64), its operand bytes at 128 B per cycle and a floor of
// about 44 cycles, so p.c at M = 128 runs at the full tensor rate and q.c^T
// is not repeated for different output dims: per token the two 64-head CTAs
// of a sequence spend ~25 cycles each (36 q.c^T steps at the floor over a
// 64-token stage, 16 p.c MMAs of 48 cycles).  Tensor memory holds O^T in 256
// columns (lanes = dims, a column per head) and the S buffers beside it; an
// M = 64 accumulator keeps row r in lane 32 (r / 16) + r % 16 (16 rows in each
// warp quadrant).  A 576-d latent row is 1152 B, so a 64-token stage is
// 72 KiB; two stages, Q (64 heads) and P fill the 227 KB.  (Sharing the
// q.c^T work of 128 heads between a CTA pair over distributed shared memory
// would move a 32 KB fp32 score tile each way per stage at about 20 B per
// cycle, more than the stage's own time.)  The latent pool is tiled as
// 8 x 8 core matrices per 8 tokens, so one bulk copy per block lands an
// MMA-ready operand for both contractions: element (slot s, dim i) of a block
// at ((s / 8) * 72 + i / 8) * 64 + (s % 8) * 8 + i % 8.
//
// Roles (352 threads): warps 0-7 softmax and epilogue (two threads per head
// row, each with half of the stage's tokens; the row maximum and sum combine
// the pair's through shared memory; a moved reference rescales the O^T
// columns of its head, 32 dims of two blocks per thread), warp 8 producer,
// warp 9 q.c^T issuer and tensor-memory owner, warp 10 p.c issuer (a separate
// thread, so that a p.c -- which frees its stage for the next load -- is not
// queued behind the issue of the next stage's 36 q.c^T steps).  Every wait is
// bounded.  A context longer than one part is split over CTAs; the parts'
// (max, sum, output) states are merged by mla_combine_kernel.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attention_kernel.cuh"

namespace pgd {
namespace mla {

using tc::fence_proxy_async;
using tc::smem_desc;
using tc::tc_fence_after;
using tc::tc_fence_before;
using tc::umma_bf16;
using tc::umma_commit;
using tc::wait_or_abort;

constexpr int D = 576;          // cached values per token (latent + RoPE key)
constexpr int DV = 512;         // latent dims (the value)
constexpr int TOKS = 64;        // tokens per stage
constexpr int NSTG = 2;         // stage buffers (and S buffers)
constexpr int NH = 64;          // head rows per CTA
constexpr int NDB = DV / 128;   // 128-dim blocks of O^T (the M of one p.c MMA)
constexpr int THREADS = 352;
// Softmax warps 0-7: warp w reaches TMEM lane quadrant w % 4, whose lanes
// 0..15 hold head rows 16 (w % 4) .. of S; warps 0-3 take token columns
// 0..31, warps 4-7 columns 32..63 of the same rows (and, for O^T, dims
// 32 (w % 4) .. of blocks 0-1 and 2-3).  Warp 8 produces, warp 9 issues
// q.c^T (and owns tensor memory), warp 10 issues p.c.
constexpr int WARP_PROD = 8, WARP_QK = 9, WARP_PV = 10;
constexpr int GRP = (D / 8) * 128;   // bytes per 8 rows of 576 values: 9216
constexpr int STAGE = (TOKS / 8) * GRP;  // 73,728
constexpr int Q_BYTES = (NH / 8) * GRP;  // 73,728
// A stage lands in NR ranges of latent dims, each on its own barrier, so
// that q.c^T starts on the first range while the second is still landing:
// one bulk copy per (8-token group, range) of RCH 16-byte chunks.  (One
// 72 KiB copy per stage lands in about 1 us; 32 copies of 2304 B took about
// 2 us for the last range, so finer ranges lose what the overlap gains:
// measured 86.8 us a step with one copy per block, 85.8 / 85.7 / 86.4 /
// 87.8 us with 1 / 2 / 3 / 4 ranges per token group.)
constexpr int NR = 2;
constexpr int RCH = (D / 8) / NR;         // 36 chunks (288 dims) per range
constexpr int RBYTES = RCH * 128;         // 4608 bytes of a token group per range
constexpr int KPR = (D / 16) / NR;        // 18 q.c^T k-steps per range
static_assert((D / 8) % NR == 0 && (D / 16) % NR == 0 && RBYTES % 16 == 0, "dim ranges");
constexpr int P_RG = (TOKS / 8) * 128;   // bytes per 8 rows of P: 1024
constexpr int P_BYTES = (NH / 8) * P_RG; // [8 row groups][8 token groups][8][16 B] = 8192
// P, then Q, then the stage ring.
constexpr int OFF_P = 0;
constexpr int OFF_Q = OFF_P + P_BYTES;
constexpr int OFF_C = OFF_Q + Q_BYTES;
constexpr int OFF_BAR = OFF_C + NSTG * STAGE;
constexpr int OFF_MISC = OFF_BAR + 128;
static_assert((NSTG * NR + 3 * NSTG + 3) * 8 <= OFF_MISC - OFF_BAR, "barrier area");
constexpr int OFF_X = OFF_MISC + 64;  // f32 [2 parities][2 halves][64 rows] row maxima,
                                      // [2 halves][64 rows] row sums, [64 rows] rescale factors
constexpr int SMEM_BYTES = 1024 + OFF_X + 7 * NH * 4;
static_assert(SMEM_BYTES <= 232448, "MLA kernel exceeds 227 KB of shared memory");

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_O = 0;          // O^T block k at columns 64 k .. 64 k + 63
constexpr uint32_t COL_S = NDB * NH;   // S buffers at 256 and 320

// kind::f16, D f32, A and B bf16, M = m, N = n; a_mn / b_mn: MN-major operands.
__host__ __device__ constexpr uint32_t idesc(int m, int n, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// Bulk prefetch of global memory into L2 (src 16-byte aligned, bytes a
// multiple of 16); a hint, with no completion to wait for.
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// 2^x by the hardware approximation (relative error about 2^-22, far below
// the bf16 rounding of the probabilities; -inf gives +0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Named barrier over `count` threads that also returns whether `pred` held
// for any of them.
__device__ __forceinline__ bool named_barrier_any(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes (wait included).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
      "%10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, "
      "%27, %28, %29, %30, %31, %32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// Rows 0..15 of this warp's lane quadrant (an M = 64 accumulator's rows),
// 32 consecutive columns: lanes t and t + 16 get row t's columns [0, 16) and
// [16, 32) (wait included).
__device__ __forceinline__ void tmem_ld_rows16(uint32_t taddr, float *v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16], 16;\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Stages [first, last) of a sequence's ceil(ctx / 64) for part `part` of n.
__device__ __forceinline__ void part_stages(int nst_seq, int part, int n_parts, int &first,
                                            int &last) {
  first = (int)((long long)nst_seq * part / n_parts);
  last = (int)((long long)nst_seq * (part + 1) / n_parts);
}

template <int BS>
__global__ void __launch_bounds__(THREADS, 1) mla_attention_kernel(const MlaParams p) {
  // A stage is copied in pieces of PB tokens: whole blocks, or a slice of
  // one block when blocks are longer than a stage.
  constexpr int PB = BS < TOKS ? BS : TOKS;
  constexpr uint32_t TILE = BS * D * 2;    // one block's latent rows
  constexpr uint32_t PIECE = PB * D * 2;
  constexpr uint32_t IDESC_QK = idesc(NH, TOKS, false, false);
  constexpr uint32_t IDESC_PV = idesc(128, NH, true, false);
  static_assert((TOKS % BS == 0 || BS % TOKS == 0) && BS % 8 == 0, "block size");

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Launched with programmatic stream serialization.  Unless the previous
  // kernel is this library's latent append, which writes only the cache (the
  // producer then waits for it before its first copy), wait for it now: q,
  // the cache and the tables may come from it.
  if (!p.wait_late) pdl_wait();

  int w = (int)blockIdx.x;
  const int part = w % p.n_parts;
  w /= p.n_parts;
  const int n_hg = (p.H + NH - 1) / NH;
  const int hg = w % n_hg, b = w / n_hg;
  if (b >= p.B) return;
  const int rows = min(NH, p.H - hg * NH);  // real head rows of this CTA
  const int ctx = __ldg(p.ctx + b);
  const bool ctx_ok = ctx >= 1 && ctx <= p.MB * BS;
  const int nst_seq = ctx_ok ? (ctx + TOKS - 1) / TOKS : 0;
  int st0, st1;
  part_stages(nst_seq, part, p.n_parts, st0, st1);
  const int nst = st1 - st0;
  if (!ctx_ok && tid == 0 && hg == 0 && part == 0)
    atomicOr(p.err, PGD_DEVERR_BAD_CONTEXT);

  const int r = tid;  // head row of warps 0-1 (empty parts)
  const bool row_ok = r < rows;
  const int h = hg * NH + r;
  // partial state slot of (b, h, part)
  const size_t slot = ((size_t)b * p.H + h) * p.n_parts + part;

  if (nst <= 0) {  // an empty part (or a rejected sequence): a -inf maximum
    if (warp < 2 && row_ok && p.n_parts > 1) {
      *reinterpret_cast<float2 *>(p.part_ml + slot * 2) = make_float2(-INFINITY, 0.f);
      float4 *o = reinterpret_cast<float4 *>(p.part_o + slot * DV);
      for (int i = 0; i < DV / 4; ++i) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return;
  }

  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
  // c_full[buf * NR + r]: range r of stage buffer buf has landed
  uint64_t *c_full = bars, *c_empty = bars + NSTG * NR, *s_full = c_empty + NSTG;
  uint64_t *s_free = s_full + NSTG;
  uint64_t *p_full = s_free + NSTG, *p_free = p_full + 1, *o_done = p_full + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 16);  // WaitCtl
  volatile int *bad_mask = reinterpret_cast<volatile int *>(smem + OFF_MISC + 8);  // [NSTG]

  if (tid == 0) {
    for (int i = 0; i < NSTG; ++i) {
      for (int r = 0; r < NR; ++r) mbar_init(&c_full[i * NR + r], 1);
      mbar_init(&c_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 8);  // one arrival per softmax warp
    }
    mbar_init(p_full, 1);
    mbar_init(p_free, 1);
    mbar_init(o_done, 1);
    mbar_init_fence();
    init_wait_ctl(smem + OFF_MISC + 16, p.wait_limit_ns);
  }
  // Q rows as the K-major A operand: head row r, dims 8c..8c+7 in core
  // matrix (r / 8, c), row r % 8; rows past the real heads are zeros.
  {
    const uint4 *qsrc = reinterpret_cast<const uint4 *>(p.q);
    for (int i = tid; i < NH * (D / 8); i += THREADS) {
      const int qr = i / (D / 8), c = i % (D / 8);
      const uint4 v = (qr < rows) ? __ldg(qsrc + ((size_t)b * p.H + hg * NH + qr) * (D / 8) + c)
                                  : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4 *>(smem + OFF_Q + (qr >> 3) * GRP + c * 128 + (qr & 7) * 16) = v;
    }
  }
  if (warp == WARP_QK) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int32_t *trow = p.tables + (size_t)b * p.MB;

  // valid tokens of local stage i (the sequence's last stage may be partial)
  auto stage_tokens = [&](int i) { return min(TOKS, ctx - (st0 + i) * TOKS); };

  if (warp == WARP_PROD) {
    // ------------------------------------------------------------ producer
    if (p.wait_late == 1) pdl_wait();  // the latent append has written the cache
    const uint64_t policy = l2_policy_evict_first();
    int armed = 0;  // stages armed; after a timeout in the CTA nothing more is
    for (int i = 0; i < nst; ++i) {
      const int buf = i % NSTG;
      const uint32_t par = (uint32_t)(i / NSTG) & 1u;
      const int nb = (stage_tokens(i) + PB - 1) / PB;  // pieces with a valid token
      const int ng = (stage_tokens(i) + 7) / 8;        // token groups with a valid token
      // lane = r * 8 + tg: range r of token group tg (ranges in order, so
      // that the first lands first; lanes past 8 NR idle)
      const int tg = lane & 7, rr = lane >> 3;
      const int t0 = (st0 + i) * TOKS + tg * 8;        // first token of this lane's group
      const int blk = (tg < ng && rr < NR) ? __ldg(trow + t0 / BS) : -1;
      const bool ok = rr < NR && tg < ng && (unsigned)blk < (unsigned)p.NB;
      const unsigned okmask = __ballot_sync(kFullMask, ok);
      // bad-block mask by piece (bit j: tokens [j PB, (j + 1) PB) of the stage)
      unsigned bad = 0;
      for (int j = 0; j < nb; ++j) {
        const int l0 = (j * PB) / 8;  // a group of piece j, range 0
        if (!((okmask >> l0) & 1u)) bad |= 1u << j;
      }
      // one decision for the warp: after a timeout the buffer's earlier copy
      // may still be landing, so it is neither armed again nor written
      int go = 1;
      if (lane == 0) {
        wait_or_abort(&c_empty[buf], par ^ 1u, abort_flag, p.err);
        go = *abort_flag ? 0 : 1;
      }
      if (!__shfl_sync(kFullMask, go, 0)) break;
      armed = i + 1;
      if (lane == 0) {
        bad_mask[buf] = (int)bad;
        if (bad) atomicOr(p.err, PGD_DEVERR_BAD_BLOCK_ID);
        const uint32_t bytes = (uint32_t)__popc(okmask & 0xffu) * RBYTES;  // per range
        for (int r = 0; r < NR; ++r) {
          if (bytes == 0)
            mbar_arrive(&c_full[buf * NR + r]);
          else
            mbar_arrive_expect_tx(&c_full[buf * NR + r], bytes);
        }
      }
      __syncwarp();
      if (ok)
        bulk_copy_g2s(smem + OFF_C + buf * STAGE + tg * GRP + rr * RBYTES,
                      p.cache + (size_t)blk * TILE + (size_t)((t0 % BS) / 8) * GRP + rr * RBYTES,
                      RBYTES, &c_full[buf * NR + rr], policy);
      // The stage after next goes to L2 now: its buffer frees only after this
      // stage's p.c, and its copy then finds the data on chip.
      const int ip = i + NSTG;
      if (ip < nst) {
        const int nbp = (stage_tokens(ip) + PB - 1) / PB;
        const int tp = (st0 + ip) * TOKS + lane * PB;
        const int blkp = (lane < nbp) ? __ldg(trow + tp / BS) : -1;
        if ((unsigned)blkp < (unsigned)p.NB)
          prefetch_l2(p.cache + (size_t)blkp * TILE + (size_t)((tp % BS) / 8) * GRP, PIECE);
      }
    }
    if (lane == 0) {  // no copy may still be landing when the CTA exits
      for (int k = 1; k <= NSTG && k <= armed; ++k) {
        const int last = armed - k;
        for (int r = 0; r < NR; ++r)
          if (!mbar_wait_bounded(&c_full[(last % NSTG) * NR + r], (uint32_t)(last / NSTG) & 1u))
            atomicOr(p.err, PGD_DEVERR_TIMEOUT);
      }
    }
  } else if (warp == WARP_QK) {
    // ---------------------------------------------------- q.c^T issuer
    if (lane == 0) {
      const uint64_t qd = smem_desc(smem_addr(smem + OFF_Q), 128, GRP, 0);
      for (int i = 0; i < nst; ++i) {
        const int buf = i % NSTG;
        const uint32_t par = (uint32_t)(i / NSTG) & 1u;
        wait_or_abort(&s_free[buf], par ^ 1u, abort_flag, p.err);
        // A = Q, B = C, both K-major: a k-step of 16 dims moves both by two
        // core matrices (256 B); range r's k-steps are issued once it landed
        const uint64_t cd = smem_desc(smem_addr(smem + OFF_C + buf * STAGE), 128, GRP, 0);
        for (int r = 0; r < NR; ++r) {
          wait_or_abort(&c_full[buf * NR + r], par, abort_flag, p.err);
          tc_fence_after();
          if (!*abort_flag) {
#pragma unroll
            for (int k = 0; k < KPR; ++k) {
              const int kk = r * KPR + k;
              umma_bf16(tmem + COL_S + (uint32_t)(buf * TOKS), qd + (uint64_t)(kk * 16),
                        cd + (uint64_t)(kk * 16), IDESC_QK, kk > 0 ? 1u : 0u);
            }
          }
        }
        umma_commit(&s_full[buf]);
      }
    }
  } else if (warp == WARP_PV) {
    // ------------------------------------------------------ p.c issuer
    if (lane == 0) {
      // B = P^T: heads on N, K-major (8 tokens per 16-byte row, 128 B per
      // token group, P_RG per 8 heads)
      const uint64_t pd = smem_desc(smem_addr(smem + OFF_P), 128, P_RG, 0);
      for (int j = 0; j < nst; ++j) {
        const int buf = j % NSTG;
        const int nkt = (stage_tokens(j) + 15) >> 4;  // 16-token steps with a valid token
        wait_or_abort(p_full, (uint32_t)(j & 1), abort_flag, p.err);
        tc_fence_after();
        if (!*abort_flag) {
          // A = V^T: 128 dims on M, MN-major (8 dims per 16-byte row, 128 B
          // per 8 dims; 8 tokens per core matrix, GRP per token group)
          const uint64_t vd = smem_desc(smem_addr(smem + OFF_C + buf * STAGE), GRP, 128, 0);
          for (int kt = 0; kt < nkt; ++kt)
#pragma unroll
            for (int db = 0; db < NDB; ++db)
              umma_bf16(tmem + COL_O + (uint32_t)(db * NH),
                        vd + (uint64_t)((db * 16 * 128 + kt * 2 * GRP) >> 4),
                        pd + (uint64_t)(kt * 16), IDESC_PV, (j > 0 || kt > 0) ? 1u : 0u);
        }
        umma_commit(&c_empty[buf]);  // the stage buffer may be refilled
        umma_commit(p_free);         // P may be rewritten
      }
      // (every q.c^T completed before its stage's softmax released p.c)
      umma_commit(o_done);
      mbar_wait_bounded(o_done, 0);
    }
  } else if (warp < 8) {
    // ------------------------------ softmax, four threads per head row
    const int sh = warp >> 2;              // token half of this warp (and O^T blocks 2 sh ..)
    const int tq = lane >> 4;              // 16-token quarter of the half (lanes t, t + 16)
    const int r = (warp & 3) * 16 + (lane & 15);  // head row (lanes 0..15 of the quadrant)
    const int st = tid;                    // 0..255 over the eight warps
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const bool rok = lane < 16 && r < rows;
    const int hr = hg * NH + r;
    const size_t slot_r = ((size_t)b * p.H + hr) * p.n_parts + part;
    float *xmax = reinterpret_cast<float *>(smem + OFF_X);  // [parity][half][row]
    float *lx = xmax + 4 * NH;                               // [half][row]
    float *alpha_s = lx + 2 * NH;                            // [row]
    constexpr int TT = TOKS / 4;           // token columns per thread
    float m_ref = -INFINITY, l = 0.f;
    for (int i = 0; i < nst; ++i) {
      const int buf = i % NSTG;
      const uint32_t par = (uint32_t)(i / NSTG) & 1u;
      const int nv = stage_tokens(i);
      wait_or_abort(&s_full[buf], par, abort_flag, p.err);
      // (the producer wrote the stage's bad-block mask before arming c_full;
      // that phase has completed and cannot move on before this stage's p.c)
      for (int rg = 0; rg < NR; ++rg) wait_or_abort(&c_full[buf * NR + rg], par, abort_flag, p.err);
      const int bad = bad_mask[buf];
      tc_fence_after();
      float sv[TT];  // row r, tokens sh * 32 + tq * 16 + [0, 16)
      tmem_ld_rows16(tmem + lane_base + COL_S + (uint32_t)(buf * TOKS + sh * 2 * TT), sv);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[buf]);
      // Scores stay unscaled (the scale is > 0, so the maximum commutes with
      // it); masked tokens become -inf.  A full stage needs no mask.
      if (nv < TOKS || bad) {
#pragma unroll
        for (int c = 0; c < TT; ++c) {
          const int t = (2 * sh + tq) * TT + c;
          if (t >= nv || ((bad >> (t / PB)) & 1)) sv[c] = -INFINITY;
        }
      }
      float hm[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
      for (int c = 4; c < TT; ++c) hm[c & 3] = fmaxf(hm[c & 3], sv[c]);
      float hmax = fmaxf(fmaxf(hm[0], hm[1]), fmaxf(hm[2], hm[3]));
      hmax = fmaxf(hmax, __shfl_xor_sync(kFullMask, hmax, 16)) * p.qk_scale_log2;
      // the row maximum: this half's and the pair's (one exchange a stage,
      // by stage parity so that no second barrier is needed)
      if (lane < 16) xmax[((i & 1) * 2 + sh) * NH + r] = hmax;
      named_barrier_sync(1, 256);
      const float rmax = fmaxf(hmax, xmax[((i & 1) * 2 + (sh ^ 1)) * NH + r]);
      // lazy rescale: move the row's reference when exceeded by 2^8.  O^T
      // keeps a head per column, so a move rescales that column of every
      // block; the pass runs when any row moved, with factor 1 elsewhere.
      const bool need = rmax > m_ref + tc::kRescaleLog2;  // (alike in the row's four threads)
      float alpha = 1.f;
      if (need) {
        alpha = (m_ref == -INFINITY) ? 0.f : exp2f(m_ref - rmax);
        m_ref = rmax;
        l *= alpha;
      }
      if (sh == 0 && lane < 16) alpha_s[r] = alpha;
      const bool any = named_barrier_any(1, 256, need);
      // P and the O^T rescale both wait for the previous p.c
      wait_or_abort(p_free, ((uint32_t)(i & 1)) ^ 1u, abort_flag, p.err);
      if (i > 0 && any) {
        tc_fence_after();
#pragma unroll 1
        for (int k = 0; k < 2 * (NH / 32); ++k) {  // blocks 2 sh, 2 sh + 1; 32 heads at a time
          float ov[32];
          const uint32_t col = COL_O + (uint32_t)((2 * sh + (k >> 1)) * NH + (k & 1) * 32);
          tmem_ld32(tmem + lane_base + col, ov);
#pragma unroll
          for (int c = 0; c < 32; ++c) ov[c] *= alpha_s[(k & 1) * 32 + c];
          tmem_st32(tmem + lane_base + col, ov);
        }
        tc_fence_before();
      }
      // probabilities 2^(s * scale - m) in bf16 (one fma and one ex2 each; a
      // masked -inf score gives 0), summed as the tensor cores see them; row
      // r's 8-token pieces at core matrix (r / 8, token group), row r % 8
      {
        unsigned char *prow =
            smem + OFF_P + (r >> 3) * P_RG + ((2 * sh + tq) * (TT / 8)) * 128 + (r & 7) * 16;
        const float mb = (m_ref == -INFINITY) ? 0.f : m_ref;  // (every score masked so far)
        float ls[2] = {0.f, 0.f};
#pragma unroll
        for (int g = 0; g < TT / 8; ++g) {
          uint32_t pk[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int c = g * 8 + 2 * k;
            const __nv_bfloat162 pr = __floats2bfloat162_rn(
                ex2_approx(fmaf(sv[c], p.qk_scale_log2, -mb)),
                ex2_approx(fmaf(sv[c + 1], p.qk_scale_log2, -mb)));
            pk[k] = *reinterpret_cast<const uint32_t *>(&pr);
            ls[k & 1] += bf16lo(pk[k]) + bf16hi(pk[k]);
          }
          *reinterpret_cast<uint4 *>(prow + g * 128) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        l += ls[0] + ls[1];
      }
      // Latent rows p.c reads that hold no valid token (the tail of the last
      // block, blocks with a bad id) must not feed NaN into it: zero them
      // (their copies have landed -- q.c^T waited for them -- and p.c of
      // this stage has not been issued).
      const int lim = ((nv + 15) & ~15);
      if (nv < lim || bad) {
        unsigned char *cs = smem + OFF_C + buf * STAGE;
        for (int k = st; k < lim * (D / 8); k += 256) {
          const int t = k / (D / 8), c = k % (D / 8);
          if (t >= nv || ((bad >> (t / PB)) & 1))
            *reinterpret_cast<uint4 *>(cs + (t >> 3) * GRP + c * 128 + (t & 7) * 16) =
                make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      named_barrier_sync(1, 256);  // all eight softmax warps have written P and zeroed
      if (st == 0) mbar_arrive(p_full);
    }
    // ---- epilogue: the row's sum over both halves; then O^T by dims, 32
    // dims of two blocks per thread, every head of the CTA
    l += __shfl_xor_sync(kFullMask, l, 16);  // the row's two quarters of this half
    if (lane < 16) lx[sh * NH + r] = l;
    named_barrier_sync(1, 256);
    const float l_row = l + lx[(sh ^ 1) * NH + r];
    float *linv = xmax;  // [row] 1 / sum (the maxima are no longer read)
    if (sh == 0 && lane < 16) linv[r] = 1.f / l_row;
    if (rok && p.n_parts > 1 && sh == 0)
      *reinterpret_cast<float2 *>(p.part_ml + slot_r * 2) = make_float2(m_ref, l_row);
    named_barrier_sync(1, 256);
    wait_or_abort(o_done, 0, abort_flag, p.err);
    tc_fence_after();
    const size_t row0 = (size_t)b * p.H + (size_t)hg * NH;  // first head row of the CTA
#pragma unroll 1
    for (int k = 0; k < 2 * (NH / 32); ++k) {
      float ov[32];
      const int db = 2 * sh + (k >> 1), h0 = (k & 1) * 32;
      const int dim = db * 128 + (warp & 3) * 32 + lane;  // this lane's latent dim
      tmem_ld32(tmem + lane_base + COL_O + (uint32_t)(db * NH + h0), ov);
      if (p.n_parts == 1) {
#pragma unroll 4
        for (int c = 0; c < 32; ++c)
          if (h0 + c < rows)
            p.out[(row0 + h0 + c) * DV + dim] = __float2bfloat16_rn(ov[c] * linv[h0 + c]);
      } else {
#pragma unroll 4
        for (int c = 0; c < 32; ++c)
          if (h0 + c < rows)
            p.part_o[((row0 + h0 + c) * p.n_parts + part) * DV + dim] = ov[c];
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == WARP_QK)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(TMEM_COLS)
                 : "memory");
}

// Merge of the parts of each (sequence, head) by log-sum-exp: a warp per
// row, lane e owning dims 4 (32 j + e) .. + 3 for j < 4 (coalesced float4s).
// The first four parts' outputs are loaded together with the maxima, ahead
// of the reduction that needs the maxima: one memory round trip per row for
// up to four parts.
__global__ void __launch_bounds__(128) mla_combine_kernel(const MlaParams p) {
  constexpr int KP = 4;  // parts whose outputs are loaded up front
  pdl_wait();
  const int row = (int)blockIdx.x * 4 + (threadIdx.x >> 5);  // b * H + h
  const int lane = threadIdx.x & 31;
  if (row >= p.B * p.H) return;
  const int c = __ldg(p.ctx + row / p.H);
  if (c < 1 || c > p.MB * p.bs) return;  // rejected (flagged by the attention kernel)
  const float2 *ml = reinterpret_cast<const float2 *>(p.part_ml) + (size_t)row * p.n_parts;
  const float4 *po = reinterpret_cast<const float4 *>(p.part_o) + (size_t)row * p.n_parts * (DV / 4);
  float4 x0[KP][4];
#pragma unroll
  for (int k = 0; k < KP; ++k)
#pragma unroll
    for (int j = 0; j < 4; ++j)
      x0[k][j] = (k < p.n_parts) ? __ldcg(po + (size_t)k * (DV / 4) + j * 32 + lane)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
  float M = -INFINITY;
  for (int k = lane; k < p.n_parts; k += 32) M = fmaxf(M, __ldcg(&ml[k].x));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, o));
  float L = 0.f;
  float4 acc[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  auto fold = [&](const float2 v, const float4 (&x)[4]) {
    if (v.x == -INFINITY) return;  // an empty part
    const float w = exp2f(v.x - M);
    L = fmaf(w, v.y, L);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[j].x = fmaf(w, x[j].x, acc[j].x);
      acc[j].y = fmaf(w, x[j].y, acc[j].y);
      acc[j].z = fmaf(w, x[j].z, acc[j].z);
      acc[j].w = fmaf(w, x[j].w, acc[j].w);
    }
  };
#pragma unroll
  for (int k = 0; k < KP; ++k)
    if (k < p.n_parts) fold(__ldcg(&ml[k]), x0[k]);
#pragma unroll 2
  for (int k = KP; k < p.n_parts; ++k) {
    float4 x[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] = __ldcg(po + (size_t)k * (DV / 4) + j * 32 + lane);
    fold(__ldcg(&ml[k]), x);
  }
  const float inv = 1.f / L;
  uint2 *o = reinterpret_cast<uint2 *>(p.out + (size_t)row * DV);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[j].x * inv, acc[j].y * inv);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[j].z * inv, acc[j].w * inv);
    o[j * 32 + lane] = make_uint2(*reinterpret_cast<const uint32_t *>(&lo),
                                  *reinterpret_cast<const uint32_t *>(&hi));
  }
}

// One warp per sequence: the new token's 576 values into its slot (72
// 16-byte pieces, piece c of slot s at ((s / 8) * 72 + c) * 8 + s % 8 uint4s
// into the block's tile).  A bit copy.
__global__ void __launch_bounds__(128)
mla_append_kernel(const uint4 *__restrict__ c_new, uint4 *__restrict__ cache,
                  const int32_t *__restrict__ tables, const int32_t *__restrict__ pos,
                  int pos_offset, int B, int bs, int MB, int NB, int32_t *err) {
  pdl_wait();  // the previous kernel (which may read this slot) has completed
  pdl_launch_dependents();
  const int b = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (b >= B) return;
  const int pp = __ldg(pos + b) + pos_offset;  // (pos_offset -1: pos are context lengths)
  if (pp < 0 || pp >= MB * bs) {
    if (lane == 0) atomicOr(err, PGD_DEVERR_BAD_POSITION);
    return;
  }
  const int blk = __ldg(tables + (size_t)b * MB + pp / bs);
  if ((unsigned)blk >= (unsigned)NB) {
    if (lane == 0) atomicOr(err, PGD_DEVERR_BAD_BLOCK_ID);
    return;
  }
  const int s = pp % bs;
  uint4 *tile = cache + (size_t)blk * bs * (D / 8);
  for (int c = lane; c < D / 8; c += 32)
    tile[((size_t)(s >> 3) * (D / 8) + c) * 8 + (s & 7)] = __ldg(c_new + (size_t)b * (D / 8) + c);
}

template <int BS>
static cudaError_t launch_bs(const MlaParams &p, int grid, cudaStream_t stream) {
  static volatile int done[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!(dev >= 0 && dev < 64 && done[dev])) {
    e = cudaFuncSetAttribute(mla_attention_kernel<BS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) done[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_attention_kernel<BS>, p);
}

}  // namespace mla

int mla_heads_per_cta() { return mla::NH; }

cudaError_t mla_attention_launch(const MlaParams &p, cudaStream_t stream) {
  const int n_hg = (p.H + mla::NH - 1) / mla::NH;
  const long long grid = (long long)p.B * n_hg * p.n_parts;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaError_t e = cudaErrorInvalidValue;
  switch (p.bs) {
    case 16: e = mla::launch_bs<16>(p, (int)grid, stream); break;
    case 32: e = mla::launch_bs<32>(p, (int)grid, stream); break;
    case 64: e = mla::launch_bs<64>(p, (int)grid, stream); break;
  }
  if (e != cudaSuccess || p.n_parts == 1) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((p.B * p.H + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla::mla_combine_kernel, p);
}

cudaError_t mla_append_launch(const void *c_new, void *cache, const int32_t *tables,
                              const int32_t *pos, int pos_offset, int B, int bs, int MB, int NB,
                              int32_t *err, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  // (launched with programmatic stream serialization: it may be scheduled
  // while the previous kernel finishes, and waits for it before any access)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((B + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla::mla_append_kernel, static_cast<const uint4 *>(c_new),
                            static_cast<uint4 *>(cache), tables, pos, pos_offset, B, bs, MB, NB,
                            err);
}

}  // namespace pgd
