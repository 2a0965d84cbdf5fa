// prefix_attention.cu -- the shared-prefix pass of cascade decode attention.
//
// Several sequences whose block tables start with the same physical blocks
// ("Module 10: inference and serving", section "Share only identical state":
// sequences may point at the same read-only prefix blocks) store that prefix
// once; reading it once per sequence wastes the traffic the sharing saved
// (same page, on storage sharing versus traffic reuse).  This pass reads each
// shared prefix tile once per group and KV head and multiplies it against
// every query row of the group at once: up to 128 rows (sequences x G query
// heads) on the tensor cores' M side, 128 tokens on N:
//   S[128 rows][128 tok] = Q[128 rows][128 d] . K^T   (A = Q, B = K, K-major)
//   O[128 rows][128 d]  += P[128 rows][128 tok] . V    (A = P K-major, B = V MN-major)
// with the same tiled pool as the decode kernel (one bulk copy per (block,
// head) tile lands an MMA-ready operand).  The lazy rescale moves a row's
// reference when exceeded by 2^8.  The result is a partial state (max, sum,
// unnormalised output) per (sequence, query head) and prefix part; the decode
// pass over each sequence's own suffix merges these into its output by
// log-sum-exp ("The math of Transformer inference", section 8; "LLM inference
// systems engineering", 2.8.3).
//
// Work item (one CTA): (group, KV head, chunk of 128 / G sequences, part of
// the prefix's blocks).  Roles (352 threads): warps 0-7 softmax and epilogue
// (two threads per row: warps w and w + 4 take tokens 0..63 and 64..127 of
// lane quadrant w's rows, and half of the output dims; the row maximum and
// sum combine through shared memory), warp 8 K producer, warp 9 V producer,
// warp 10 MMA issuer and tensor-memory owner.  Every wait is bounded.
#include "attention_kernel.cuh"

namespace pgd {
namespace pf {

using tc::smem_desc;
using tc::umma_bf16;
using tc::umma_commit;
using tc::tc_fence_after;
using tc::tc_fence_before;
using tc::fence_proxy_async;
using tc::wait_or_abort;

constexpr int TOKP = 128;     // tokens per stage (MMA N of q.k^T)
constexpr int ROWS = 128;     // query rows per CTA (MMA M)
constexpr int THREADS = 352;
constexpr int WARP_KP = 8, WARP_VP = 9, WARP_MMA = 10;
constexpr int STAGE = TOKP * 256;  // bytes of one K (or V) stage
constexpr int OFF_Q = 0;                       // [128 rows][128 d] bf16, K-major
constexpr int OFF_K = OFF_Q + ROWS * 256;      // 2 stages
constexpr int OFF_V = OFF_K + 2 * STAGE;       // 2 stages
constexpr int OFF_P = OFF_V + 2 * STAGE;       // 2 x [128 rows][128 tok] bf16, K-major
constexpr int OFF_BAR = OFF_P + 2 * ROWS * 256;
constexpr int OFF_MISC = OFF_BAR + 256;        // tmem base, abort flag, stage masks [4]
constexpr int OFF_X = OFF_MISC + 64;            // f32 [2 parities][2 halves][128 rows] maxima
                                                // (finally one parity's: row sums)
// (no swizzled operand: 128-byte alignment of the base suffices)
constexpr int SMEM_BYTES = 128 + OFF_X + 4 * ROWS * 4;
static_assert(SMEM_BYTES <= 232448, "prefix pass exceeds 227 KB of shared memory");
constexpr uint32_t TMEM_COLS = 512;            // S 2 x 128 columns, O 128 columns

__device__ __forceinline__ uint32_t col_s(int sb) { return (uint32_t)sb * 128u; }

// 2^x by the hardware approximation (relative error about 2^-22, far below
// the bf16 rounding of the probabilities; -inf gives +0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr uint32_t COL_O = 256;

// kind::f16 instruction descriptor for M = 128, N = 128, bf16 inputs, f32
// accumulation; b_mn selects an MN-major B operand.
__host__ __device__ constexpr uint32_t idesc128(bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(128 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// 32 consecutive fp32 columns of this warp's 32 lanes (wait included).
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

// One producer warp: the part's stages, one tile per lane, with the
// invalid-block mask of each stage recorded (K producer) before it is armed.
template <int BS>
__device__ __forceinline__ void produce(const PrefixParams &p, const int32_t *trow, int blk0,
                                        int nblk, const unsigned char *cache, int g,
                                        unsigned char *ring, uint64_t *full, uint64_t *empty,
                                        volatile int *mask, volatile int *abort_flag, int lane) {
  constexpr int SB = TOKP / BS;
  constexpr uint32_t TILE = BS * 256;
  const uint64_t policy = l2_policy_evict_first();
  const int nst = (nblk + SB - 1) / SB;
  int armed = 0;  // stages armed; after a timeout in the CTA nothing more is
  for (int st = 0; st < nst; ++st) {
    const int first = st * SB, nb = min(SB, nblk - first), slot = st & 1;
    const int blk = (lane < nb) ? __ldg(trow + blk0 + first + lane) : -1;
    const bool ok = lane < nb && (unsigned)blk < (unsigned)p.NB;
    const unsigned okmask = __ballot_sync(kFullMask, ok);
    const unsigned want = (1u << nb) - 1u;
    // one decision for the warp: after a timeout the slot's earlier copies
    // may still be landing, so it is neither armed again nor written
    int go = 1;
    if (lane == 0) {
      wait_or_abort(&empty[slot], ((uint32_t)(st >> 1) & 1u) ^ 1u, abort_flag, p.err);
      go = *abort_flag ? 0 : 1;
    }
    if (!__shfl_sync(kFullMask, go, 0)) break;
    armed = st + 1;
    if (lane == 0) {
      if (mask) {
        mask[st & 3] = (int)(want & ~okmask);
        if (want & ~okmask) atomicOr(p.err, PGD_DEVERR_BAD_BLOCK_ID);
      }
      const uint32_t bytes = (uint32_t)__popc(okmask) * TILE;
      if (bytes == 0)
        mbar_arrive(&full[slot]);
      else
        mbar_arrive_expect_tx(&full[slot], bytes);
    }
    __syncwarp();
    if (ok)
      bulk_copy_g2s(ring + (size_t)slot * STAGE + (size_t)lane * TILE,
                    cache + ((size_t)blk * p.n_kv + g) * (size_t)TILE, TILE, &full[slot], policy);
    // Later stages go to L2 now (stage st + 2 at the first stage, then
    // st + 3 at each): a slot frees only after its stage's MMA, and the copy
    // issued then finds its tiles on chip instead of paying the HBM latency
    // that the concurrent suffix pass's traffic lengthens.
    for (int ahead = (st == 0 ? 2 : 3); ahead <= 3; ++ahead) {
      const int sp = st + ahead;
      if (sp >= nst) break;
      const int fp = sp * SB, nbp = min(SB, nblk - fp);
      const int blkp = (lane < nbp) ? __ldg(trow + blk0 + fp + lane) : -1;
      if ((unsigned)blkp < (unsigned)p.NB)
        bulk_prefetch_l2(cache + ((size_t)blkp * p.n_kv + g) * (size_t)TILE, TILE);
    }
  }
  // no copy may still be landing when the CTA exits (fixed limit)
  if (lane == 0) {
    for (int k = 1; k <= 2 && k <= armed; ++k) {
      const int last = armed - k;
      if (!mbar_wait_bounded(&full[last & 1], (uint32_t)(last >> 1) & 1u))
        atomicOr(p.err, PGD_DEVERR_TIMEOUT);
    }
  }
}

template <int G, int BS>
__global__ void __launch_bounds__(THREADS, 1) prefix_attention_kernel(const PrefixParams p) {
  constexpr int SB = TOKP / BS;
  constexpr int SPC = ROWS / G;  // sequences per row chunk
  constexpr uint32_t IDESC_QK = idesc128(false);
  constexpr uint32_t IDESC_PV = idesc128(true);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Inputs (q, tables, the prefix blocks) may come from the previous kernel:
  // wait for it, then let the suffix pass that follows launch on the SMs this
  // grid leaves free (it waits for this grid only before it exits).
  pdl_wait();
  pdl_launch_dependents();

  int w = (int)blockIdx.x;
  const int ts = w % p.n_tsplit;
  w /= p.n_tsplit;
  const int rc = w % p.n_rchunk;
  w /= p.n_rchunk;
  const int g = w % p.n_kv, grp = w / p.n_kv;
  if (grp >= p.n_groups) return;
  const int first = __ldg(p.group_first + grp), size = __ldg(p.group_size + grp);
  int nbp = __ldg(p.group_blocks + grp);
  if (nbp < 0 || nbp > p.MB) {
    if (threadIdx.x == 0) atomicOr(p.err, PGD_DEVERR_BAD_CONTEXT);
    nbp = max(0, min(nbp, p.MB));
  }
  const int s0 = rc * SPC;
  const int nseq = max(0, min(SPC, size - s0));
  const int rows = nseq * G;
  if (rows == 0) return;  // uniform for the CTA
  const int blk0 = (int)((long long)nbp * ts / p.n_tsplit);
  const int nblk = (int)((long long)nbp * (ts + 1) / p.n_tsplit) - blk0;
  const int32_t *trow = p.tables + (size_t)first * p.MB;

  // this thread's row (warps 0-3)
  const int r = tid;
  const bool row_ok = r < ROWS && r < rows;
  const int rb = first + s0 + r / G, rh = g * G + r % G;
  const size_t slot_row = ((size_t)rb * p.n_q + rh) * p.n_tsplit + ts;

  if (nblk <= 0) {  // an empty part: the merge skips a -inf maximum
    if (row_ok) {
      *reinterpret_cast<float2 *>(p.pre_ml + slot_row * 2) = make_float2(-INFINITY, 0.f);
      float4 *o = reinterpret_cast<float4 *>(p.pre_o + slot_row * kHeadDim);
      for (int i = 0; i < kHeadDim / 4; ++i) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return;
  }

  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~(uintptr_t)127);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
  uint64_t *full_k = bars, *empty_k = bars + 2, *full_v = bars + 4, *empty_v = bars + 6;
  uint64_t *s_full = bars + 8, *s_free = bars + 10, *p_full = bars + 12, *p_free = bars + 14;
  uint64_t *m_ready = bars + 16, *o_done = bars + 18;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 32);  // WaitCtl
  volatile int *stage_mask = reinterpret_cast<volatile int *>(smem + OFF_MISC + 16);  // [4]

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full_k[i], 1);
      mbar_init(&empty_k[i], 1);
      mbar_init(&full_v[i], 1);
      mbar_init(&empty_v[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 8);  // one arrival per softmax warp
      mbar_init(&p_full[i], 8);
      mbar_init(&p_free[i], 1);
      mbar_init(&m_ready[i], 1);
    }
    mbar_init(o_done, 1);
    mbar_init_fence();
    init_wait_ctl(smem + OFF_MISC + 32, p.wait_limit_ns);
  }
  // Q rows as the K-major A operand: row r, dims 8c..8c+7 in core matrix
  // (r / 8, c), row r % 8; rows past the chunk are zeros.
  if (r < ROWS) {
    // (all 16 loads of the row in flight before the first store)
    const uint4 *src = reinterpret_cast<const uint4 *>(p.q + ((size_t)rb * p.n_q + rh) * kHeadDim);
    uint4 v[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) v[c] = row_ok ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int c = 0; c < 16; ++c)
      *reinterpret_cast<uint4 *>(smem + OFF_Q + ((r >> 3) * 16 + c) * 128 + (r & 7) * 16) = v[c];
  }
  if (warp == WARP_MMA) {
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
  const int nst = (nblk + SB - 1) / SB;

  if (warp == WARP_KP) {
    produce<BS>(p, trow, blk0, nblk, p.k_cache, g, smem + OFF_K, full_k, empty_k, stage_mask,
                abort_flag, lane);
  } else if (warp == WARP_VP) {
    produce<BS>(p, trow, blk0, nblk, p.v_cache, g, smem + OFF_V, full_v, empty_v, nullptr,
                abort_flag, lane);
  } else if (warp == WARP_MMA) {
    // ----------------------------------------------------- MMA issuer
    // q.k^T of stage i is issued before p.v of stage i - 1, so it overlaps
    // the softmax of stage i - 1.
    if (lane == 0) {
      const uint32_t qa = smem_addr(smem + OFF_Q);
      for (int i = 0; i <= nst; ++i) {
        if (i < nst) {
          const int slot = i & 1;
          wait_or_abort(&full_k[slot], (uint32_t)(i >> 1) & 1u, abort_flag, p.err);
          wait_or_abort(&s_free[slot], ((uint32_t)(i >> 1) & 1u) ^ 1u, abort_flag, p.err);
          tc_fence_after();
          if (!*abort_flag) {
            // A = Q and B = K, both K-major 8 x 8 core matrices: 128 B along
            // d, 2048 B per 8 rows; a k-step of 16 moves both by 256 B.
            const uint64_t ad = smem_desc(qa, 128, 2048, 0);
            const uint64_t bd = smem_desc(smem_addr(smem + OFF_K + slot * STAGE), 128, 2048, 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_bf16(tmem + col_s(slot), ad + (uint64_t)(kk * 16), bd + (uint64_t)(kk * 16),
                        IDESC_QK, kk > 0 ? 1u : 0u);
          }
          umma_commit(&s_full[slot]);
          umma_commit(&empty_k[slot]);
          mbar_arrive(&m_ready[slot]);  // hands the stage mask (acquired with full_k) on
        }
        if (i >= 1) {
          const int j = i - 1, slot = j & 1;
          wait_or_abort(&p_full[slot], (uint32_t)(j >> 1) & 1u, abort_flag, p.err);
          wait_or_abort(&full_v[slot], (uint32_t)(j >> 1) & 1u, abort_flag, p.err);
          tc_fence_after();
          if (!*abort_flag) {
            // A = P (K-major, tokens along K), B = V (MN-major: 8 d per
            // 16-byte row, 128 B to the next 8 d, 2048 B to the next 8
            // tokens); a k-step of 16 tokens moves P by 256 B, V by 4096 B.
            const uint64_t ad = smem_desc(smem_addr(smem + OFF_P + slot * ROWS * 256), 128, 2048, 0);
            const uint64_t bd = smem_desc(smem_addr(smem + OFF_V + slot * STAGE), 2048, 128, 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_bf16(tmem + COL_O, ad + (uint64_t)(kk * 16), bd + (uint64_t)(kk * 256),
                        IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&empty_v[slot]);
          umma_commit(&p_free[slot]);
        }
      }
      umma_commit(o_done);
    }
  } else if (warp < 8) {
    // -------------------------------------- softmax, two threads per row
    constexpr int TH = TOKP / 2;      // token columns per thread
    const int sh = warp >> 2;         // token half (and output-dims half) of this thread
    const int rr = (warp & 3) * 32 + lane;  // row (= tensor-memory lane)
    const bool rok = rr < rows;
    const int rbr = first + s0 + rr / G, rhr = g * G + rr % G;
    const size_t slot_r = ((size_t)rbr * p.n_q + rhr) * p.n_tsplit + ts;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    float *xmax = reinterpret_cast<float *>(smem + OFF_X);  // [parity][half][row]
    float m_ref = -INFINITY, l = 0.f;
    for (int st = 0; st < nst; ++st) {
      const int slot = st & 1;
      const int nb = min(SB, nblk - st * SB);
      wait_or_abort(&s_full[slot], (uint32_t)(st >> 1) & 1u, abort_flag, p.err);
      wait_or_abort(&m_ready[slot], (uint32_t)(st >> 1) & 1u, abort_flag, p.err);
      const int mask = stage_mask[st & 3];
      tc_fence_after();
      float sv[TH];
#pragma unroll
      for (int c = 0; c < TH / 32; ++c)
        tmem_ld32(tmem + lane_base + col_s(slot) + sh * TH + c * 32, sv + c * 32);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[slot]);
      // Scores stay unscaled (the scale is > 0, so the maximum commutes with
      // it); columns past the stage's blocks or in a block with a bad id are
      // -inf.  A full stage needs no mask.
      if (nb < SB || mask) {
#pragma unroll
        for (int c = 0; c < TH; ++c) {
          const int blk = (sh * TH + c) / BS;
          if (blk >= nb || ((mask >> blk) & 1)) sv[c] = -INFINITY;
        }
      }
      float hm[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
      for (int c = 4; c < TH; ++c) hm[c & 3] = fmaxf(hm[c & 3], sv[c]);
      const float hmax = fmaxf(fmaxf(hm[0], hm[1]), fmaxf(hm[2], hm[3])) * p.qk_scale_log2;
      // the row maximum: this half's and the pair's (one exchange a stage, by
      // stage parity so that no second barrier is needed)
      xmax[((st & 1) * 2 + sh) * ROWS + rr] = hmax;
      named_barrier_sync(1, 256);
      const float rmax = fmaxf(hmax, xmax[((st & 1) * 2 + (sh ^ 1)) * ROWS + rr]);
      // move the row's reference when exceeded by 2^8; the O rows of the
      // warp are rescaled together (tensor-memory access is warp-wide), by 1
      // in the rows that keep their reference
      const bool need = rmax > m_ref + tc::kRescaleLog2;
      float alpha = 1.f;
      if (need) {
        alpha = (m_ref == -INFINITY) ? 0.f : exp2f(m_ref - rmax);
        m_ref = rmax;
        l *= alpha;
      }
      if (st > 0 && __any_sync(kFullMask, need)) {
        // once the previous p.v has completed
        wait_or_abort(&p_free[(st - 1) & 1], (uint32_t)((st - 1) >> 1) & 1u, abort_flag, p.err);
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {  // this thread's 64 of the 128 O columns
          float ov[32];
          const uint32_t col = COL_O + (uint32_t)(sh * 64 + c * 32);
          tmem_ld32(tmem + lane_base + col, ov);
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] *= alpha;
          tmem_st32(tmem + lane_base + col, ov);
        }
        tc_fence_before();
      }
      // probabilities 2^(s * scale - m) in bf16 (one fma and one ex2 each; a
      // masked -inf score gives 0), summed as the tensor cores see them
      uint32_t pk[TH / 2];
      {
        const float mb = (m_ref == -INFINITY) ? 0.f : m_ref;  // (every score masked so far)
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < TH; c += 2) {
          const __nv_bfloat162 pr =
              __floats2bfloat162_rn(ex2_approx(fmaf(sv[c], p.qk_scale_log2, -mb)),
                                    ex2_approx(fmaf(sv[c + 1], p.qk_scale_log2, -mb)));
          pk[c / 2] = *reinterpret_cast<const uint32_t *>(&pr);
          ls[(c / 2) & 3] += bf16lo(pk[c / 2]) + bf16hi(pk[c / 2]);
        }
        l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      }
      wait_or_abort(&p_free[slot], ((uint32_t)(st >> 1) & 1u) ^ 1u, abort_flag, p.err);
      unsigned char *prow = smem + OFF_P + slot * ROWS * 256 + (rr >> 3) * 2048 +
                            (sh * (TH / 8)) * 128 + (rr & 7) * 16;
#pragma unroll
      for (int c = 0; c < TH / 8; ++c)
        *reinterpret_cast<uint4 *>(prow + c * 128) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      if (nb < SB || mask) {
        // V rows that are not valid tokens must not feed NaN into p.v
        // (the threads of row r clear token row r of the stage, half each)
        wait_or_abort(&full_v[slot], (uint32_t)(st >> 1) & 1u, abort_flag, p.err);
        if (rr / BS >= nb || ((mask >> (rr / BS)) & 1)) {
          uint4 *vrow = reinterpret_cast<uint4 *>(smem + OFF_V + slot * STAGE + (rr >> 3) * 2048 +
                                                  (rr & 7) * 16);
#pragma unroll
          for (int c = 0; c < 8; ++c) vrow[(sh * 8 + c) * 8] = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[slot]);
    }
    // ---- epilogue: the row's sum over both halves, then this thread's 64
    // dims of the row's partial state
    // [half][row] sums over the maxima of the parity the last stage did not
    // use (every thread read those before the last stage's barrier)
    float *lx = xmax + (nst & 1) * 2 * ROWS;
    lx[sh * ROWS + rr] = l;
    named_barrier_sync(1, 256);
    const float l_row = l + lx[(sh ^ 1) * ROWS + rr];
    wait_or_abort(o_done, 0, abort_flag, p.err);
    tc_fence_after();
    float4 *o = reinterpret_cast<float4 *>(p.pre_o + slot_r * kHeadDim + sh * 64);
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
      float ov[32];
      tmem_ld32(tmem + lane_base + COL_O + (uint32_t)(sh * 64 + c * 32), ov);  // warp-wide
      if (rok) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          o[c * 8 + i] = make_float4(ov[4 * i], ov[4 * i + 1], ov[4 * i + 2], ov[4 * i + 3]);
      }
    }
    if (rok && sh == 0)
      *reinterpret_cast<float2 *>(p.pre_ml + slot_r * 2) = make_float2(m_ref, l_row);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == WARP_MMA)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(TMEM_COLS)
                 : "memory");
}

template <int G, int BS>
static cudaError_t launch_g(const PrefixParams &p, int grid, cudaStream_t stream) {
  static volatile int done[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!(dev >= 0 && dev < 64 && done[dev])) {
    e = cudaFuncSetAttribute(prefix_attention_kernel<G, BS>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
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
  return cudaLaunchKernelEx(&cfg, prefix_attention_kernel<G, BS>, p);
}

// Final merge of a cascade call: one CTA per output row (sequence b, query
// head h) with a shared prefix, one thread per dim: the row's suffix parts,
// then its prefix parts, folded by log-sum-exp into the bf16 output.  Parts
// are read PPG at a time, every load of a group issued before any is used.
template <int G>
__global__ void __launch_bounds__(kHeadDim) cascade_combine_kernel(const CombineParams p) {
  pdl_wait();  // the suffix pass, which waits for the prefix pass, has completed
  const int row = (int)blockIdx.x;  // b * n_q + h
  const int b = row / p.n_q, h = row % p.n_q;
  const int unit = b * p.n_kv + h / G, hh = h % G;
  if (b >= p.B) return;
  // Sequences the suffix pass rejected (flagged there) have no parts.
  const int s0 = __ldg(p.seq_prefix_blocks + b), c = __ldg(p.ctx + b);
  if (s0 <= 0 || c < 1 || c > p.MB * p.bs || s0 >= (c + p.bs - 1) / p.bs) return;
  const int e = threadIdx.x;
  const int2 info = __ldcg(p.part_info + unit);
  if (info.x < 0 || info.y < 1 || info.x + info.y > p.parts) return;
  const int n_dec = info.y, n_all = n_dec + p.n_tsplit;
  const float2 *dec_ml = reinterpret_cast<const float2 *>(p.part_ml);
  const float2 *pre_ml = reinterpret_cast<const float2 *>(p.pre_ml);
  float Mx = -INFINITY, Lm = 0.f, O = 0.f;
  constexpr int PPG = 8;
#pragma unroll 1
  for (int i0 = 0; i0 < n_all; i0 += PPG) {
    float2 ml[PPG];
    float o[PPG];
#pragma unroll
    for (int i = 0; i < PPG; ++i) {
      const int j = i0 + i;
      if (j < n_dec) {
        const size_t r = ((size_t)unit + (size_t)(info.x + j)) * G + hh;
        ml[i] = __ldcg(dec_ml + r);
        o[i] = __ldcg(p.part_o + r * kHeadDim + e);
      } else if (j < n_all) {
        const size_t r = (size_t)row * p.n_tsplit + (j - n_dec);
        ml[i] = __ldcg(pre_ml + r);
        o[i] = __ldcg(p.pre_o + r * kHeadDim + e);
      } else {
        ml[i] = make_float2(-INFINITY, 0.f);
        o[i] = 0.f;
      }
    }
    float nm = Mx;
#pragma unroll
    for (int i = 0; i < PPG; ++i) nm = fmaxf(nm, ml[i].x);
    if (nm == -INFINITY) continue;
    const float ca = (Mx == -INFINITY) ? 0.f : exp2f(Mx - nm);
    Lm *= ca;
    O *= ca;
#pragma unroll
    for (int i = 0; i < PPG; ++i) {
      const float cb = (ml[i].x == -INFINITY) ? 0.f : exp2f(ml[i].x - nm);
      Lm = fmaf(ml[i].y, cb, Lm);
      O = fmaf(o[i], cb, O);
    }
    Mx = nm;
  }
  p.out[(size_t)row * kHeadDim + e] = __float2bfloat16_rn(O / Lm);
}

template <int G>
static cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * p.n_q));
  cfg.blockDim = dim3(kHeadDim);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, cascade_combine_kernel<G>, p);
}

}  // namespace pf

cudaError_t cascade_combine_launch(const CombineParams &p, int G, cudaStream_t stream) {
  switch (G) {
    case 1: return pf::launch_combine<1>(p, stream);
    case 2: return pf::launch_combine<2>(p, stream);
    case 4: return pf::launch_combine<4>(p, stream);
    case 8: return pf::launch_combine<8>(p, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t prefix_attention_launch(const PrefixParams &p, int G, int bs, int grid,
                                    cudaStream_t stream) {
#define PGD_CASE(G_, BS_) \
  if (G == G_ && bs == BS_) return pf::launch_g<G_, BS_>(p, grid, stream);
  PGD_CASE(1, 16) PGD_CASE(2, 16) PGD_CASE(4, 16) PGD_CASE(8, 16)
  PGD_CASE(1, 32) PGD_CASE(2, 32) PGD_CASE(4, 32) PGD_CASE(8, 32)
#undef PGD_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pgd
