// attention.cu -- paged GQA decode attention for sm_103a.
//
// What it computes ("Module 10: inference and serving", section "Attention
// reads a different cache per sequence"; "The math of Transformer inference",
// section 4): for every sequence b and query head h,
//   out[b][h] = sum_t softmax_t(scale * q[b][h] . k_t) v_t over the
//   context_lens[b] cached positions, K/V head h / G, read through the block
//   table ("Module 10", section "Mapping logical positions to physical
//   blocks").
//
// Work decomposition.  A unit is one (sequence, KV head); its K/V tiles are
// read once and serve all G query heads.  The units' blocks are laid end to
// end (sequence-major, then KV head, then block) into one range of X blocks,
// and CTA c of P takes blocks [X*c/P, X*(c+1)/P): every CTA streams the same
// number of bytes (+-1 block) whatever the length mix.  A CTA walks its range
// unit by unit ("segments").  A segment that covers a whole unit writes the
// output; otherwise it writes its (max, sum, weighted sum) state and the last
// CTA of the unit to arrive merges the states by log-sum-exp ("The math of
// Transformer inference", section 8: split the sequence, attend locally,
// merge by log-sum-exp; the state update is the one in "LLM inference
// systems engineering", 2.8.3).  Arrival uses an atomic counter per unit; no
// CTA ever waits for another.
//
// Inside a CTA: one producer warp streams (block, head) K and V tiles -- each
// a contiguous bs*256-byte run -- into a ring of shared-memory stages with
// bulk copies on the TMA engine, signalled by mbarriers.  NW consumer warps
// take stages round robin; each keeps its own online-softmax state in
// registers (fp32) and the warps' states are merged at the end of a segment.
//
// Consumer lane layout for q.k: 16 lanes cover one token (8 head-dim
// elements each, one 16-byte shared load), two tokens per pass; the G partial
// dot products are reduce-scattered over the 16 lanes so that each lane ends
// with one (token, head) score.  For p.v each lane owns 4 of the 128 output
// elements of all G heads.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <math.h>

#include "pgd_device.cuh"

namespace pgd {

template <int N>
struct Log2 { static constexpr int value = 1 + Log2<N / 2>::value; };
template <>
struct Log2<1> { static constexpr int value = 0; };

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int G_, int BS_, int NW_, int NS_>
struct AttnCfg {
  static constexpr int G = G_, BS = BS_, NW = NW_, NS = NS_;
  static constexpr int D = kHeadDim;
  static constexpr int THREADS = (NW + 1) * 32;
  static constexpr int TILE_ELEMS = BS * D;
  static constexpr int TILE_BYTES = TILE_ELEMS * 2;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K tile then V tile
  static constexpr int OFF_BARS = NS * STAGE_BYTES;   // full[NS], empty[NS]
  static constexpr int OFF_BAD = OFF_BARS + 2 * NS * 8;
  static constexpr int OFF_PBUF = align_up(OFF_BAD + NS * 4, 16);   // f32 [NW][BS][G]
  static constexpr int OFF_ABUF = OFF_PBUF + NW * BS * G * 4;       // f32 [NW][G]
  static constexpr int OFF_MM = OFF_ABUF + NW * G * 4;              // f32 [NW][G]
  static constexpr int OFF_ML = OFF_MM + NW * G * 4;                // f32 [NW][G]
  static constexpr int OFF_MO = align_up(OFF_ML + NW * G * 4, 16);  // f32 [NW][G][D]
  static constexpr int OFF_FLAG = OFF_MO + NW * G * D * 4;          // int [4]
  static constexpr int OFF_PRE = OFF_FLAG + 16;                     // int [B + 1]
  static size_t smem_bytes(int B) { return (size_t)OFF_PRE + (size_t)(B + 1) * 4; }
};

// Segment: the part of the CTA's block range that lies in one unit.
struct Segment {
  int b, g, j0, nblk, n;
  long long unit_start, unit_end;
};

__device__ __forceinline__ Segment locate(const int *pre, int B, int n_kv, long long x,
                                          long long x_end) {
  int lo = 0, hi = B - 1;  // largest b with n_kv * pre[b] <= x
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((long long)n_kv * pre[mid] <= x) lo = mid; else hi = mid - 1;
  }
  Segment s;
  s.b = lo;
  s.nblk = pre[lo + 1] - pre[lo];
  const long long base = (long long)n_kv * pre[lo];
  const long long r = x - base;
  s.g = (int)(r / s.nblk);
  s.j0 = (int)(r % s.nblk);
  s.unit_start = base + (long long)s.g * s.nblk;
  s.unit_end = s.unit_start + s.nblk;
  const long long e = x_end < s.unit_end ? x_end : s.unit_end;
  s.n = (int)(e - x);
  return s;
}

// Reduce-scatter G partial sums over the 16 lanes of a half warp (lane bits
// 3..0).  Level k halves the vector along lane bit 3-k; the lanes then hold
// one value for head ((lane & 15) >> (4 - log2 G)), and the remaining bits
// all-reduce it.
template <int G>
__device__ __forceinline__ float reduce_scatter16(float (&a)[G], int lane) {
  constexpr int LG = Log2<G>::value;
  float w[G];
#pragma unroll
  for (int i = 0; i < G; ++i) w[i] = a[i];
#pragma unroll
  for (int k = 0; k < LG; ++k) {
    const int bit = 3 - k;
    const int half = G >> (k + 1);
    const bool upper = (lane >> bit) & 1;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? w[i] : w[i + half];
      const float keep = upper ? w[i + half] : w[i];
      w[i] = keep + __shfl_xor_sync(kFullMask, send, 1 << bit);
    }
  }
  float v = w[0];
#pragma unroll
  for (int bit = 3 - LG; bit >= 0; --bit) v += __shfl_xor_sync(kFullMask, v, 1 << bit);
  return v;
}

template <class C>
__global__ void __launch_bounds__(C::THREADS)
paged_attention_kernel(const AttnParams p) {
  constexpr int G = C::G, BS = C::BS, NW = C::NW, NS = C::NS, D = C::D;
  constexpr int LG = Log2<G>::value;
  constexpr int DUPMASK = (1 << (4 - LG)) - 1;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BARS);
  uint64_t *empty = full + NS;
  volatile int *bad = reinterpret_cast<volatile int *>(smem + C::OFF_BAD);
  volatile int *flag = reinterpret_cast<volatile int *>(smem + C::OFF_FLAG);
  int *pre = reinterpret_cast<int *>(smem + C::OFF_PRE);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init_fence();
    flag[0] = 0;  // abort
  }
  // Blocks per sequence, then an exclusive prefix over the batch.
  const int max_tokens = p.MB * BS;
  bool bad_ctx = false;
  for (int b = tid; b < p.B; b += C::THREADS) {
    const int c = p.ctx[b];
    int nb = 0;
    if (c >= 1 && c <= max_tokens) nb = (c + BS - 1) / BS; else bad_ctx = true;
    pre[b + 1] = nb;
  }
  if (bad_ctx && blockIdx.x == 0) atomicOr(p.err, PGD_DEVERR_BAD_CONTEXT);
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < p.B; base += 32) {
      const int i = base + lane;
      int v = (i < p.B) ? pre[i + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFullMask, v, o);
        if (lane >= o) v += n;
      }
      if (i < p.B) pre[i + 1] = v + carry;
      carry += __shfl_sync(kFullMask, v, 31);
    }
    if (lane == 0) pre[0] = 0;
  }
  __syncthreads();

  const long long X = (long long)p.n_kv * pre[p.B];
  const long long P = X < (long long)gridDim.x ? X : (long long)gridDim.x;
  const long long cta = blockIdx.x;
  if (cta >= P) return;  // more CTAs than blocks: the spare ones have nothing to do
  const long long x_begin = X * cta / P, x_end = X * (cta + 1) / P;

  if (warp == NW) {
    // ------------------------------------------------------------ producer
    const uint64_t policy = l2_policy_evict_first();
    int s = 0;
    bool abort = false;
    for (long long x = x_begin; x < x_end && !abort;) {
      const Segment sg = locate(pre, p.B, p.n_kv, x, x_end);
      const int32_t *trow = p.tables + (size_t)sg.b * p.MB + sg.j0;
      for (int base = 0; base < sg.n && !abort; base += 32) {
        const int cnt = min(32, sg.n - base);
        const int my_blk = (lane < cnt) ? __ldg(trow + base + lane) : 0;
        for (int k = 0; k < cnt; ++k) {
          const int blk = __shfl_sync(kFullMask, my_blk, k);
          int stop = 0;
          if (lane == 0) {
            const int slot = s % NS;
            const uint32_t phase = (uint32_t)(s / NS) & 1u;
            if (flag[0] || !mbar_wait_bounded(&empty[slot], phase ^ 1u)) {
              if (!flag[0]) atomicOr(p.err, PGD_DEVERR_TIMEOUT);
              flag[0] = 1;
              stop = 1;
            } else if ((unsigned)blk >= (unsigned)p.NB) {
              bad[slot] = 1;
              atomicOr(p.err, PGD_DEVERR_BAD_BLOCK_ID);
              mbar_arrive(&full[slot]);
            } else {
              bad[slot] = 0;
              unsigned char *dst = smem + (size_t)slot * C::STAGE_BYTES;
              const size_t tile = ((size_t)blk * p.n_kv + sg.g) * C::TILE_ELEMS;
              mbar_arrive_expect_tx(&full[slot], C::STAGE_BYTES);
              bulk_copy_g2s(dst, p.k_cache + tile, C::TILE_BYTES, &full[slot], policy);
              bulk_copy_g2s(dst + C::TILE_BYTES, p.v_cache + tile, C::TILE_BYTES, &full[slot],
                            policy);
            }
          }
          stop = __shfl_sync(kFullMask, stop, 0);
          if (stop) { abort = true; break; }
          ++s;
        }
      }
      x += sg.n;
    }
    // Never leave a copy in flight into this CTA's shared memory: wait for
    // the last phase issued on every slot (immediate unless aborted).
    if (lane == 0) {
      for (int k = 1; k <= NS && k <= s; ++k) {
        const int last = s - k;
        mbar_wait_bounded(&full[last % NS], (uint32_t)(last / NS) & 1u);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int w = warp;
  const int part = lane & 15;   // head-dim elements [8 part, 8 part + 8) for q.k
  const int jj = lane >> 4;     // token within a pass
  const int hsel = (lane & 15) >> (4 - LG);
  float *pbuf = reinterpret_cast<float *>(smem + C::OFF_PBUF) + w * BS * G;
  float *abuf = reinterpret_cast<float *>(smem + C::OFF_ABUF) + w * G;
  float *mrg_m = reinterpret_cast<float *>(smem + C::OFF_MM);
  float *mrg_l = reinterpret_cast<float *>(smem + C::OFF_ML);
  float *mrg_o = reinterpret_cast<float *>(smem + C::OFF_MO);
  const int ct = w * 32 + lane;  // consumer thread index
  constexpr int NCT = NW * 32;

  int s = 0;
  for (long long x = x_begin; x < x_end;) {
    const Segment sg = locate(pre, p.B, p.n_kv, x, x_end);
    const int unit = sg.b * p.n_kv + sg.g;
    const int ctx_b = __ldg(p.ctx + sg.b);

    float qr[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(
          p.q + ((size_t)sg.b * p.n_q + sg.g * G + h) * D + 8 * part));
      float f[8];
      unpack8(raw, f);
#pragma unroll
      for (int e = 0; e < 8; ++e) qr[h][e] = f[e] * p.qk_scale_log2;
    }
    float m_run = -INFINITY, l_run = 0.f;
    float o[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[h][e] = 0.f;

    const int first = ((w - s) % NW + NW) % NW;
    for (int i = first; i < sg.n; i += NW) {
      const int S = s + i;
      const int slot = S % NS;
      const uint32_t phase = (uint32_t)(S / NS) & 1u;
      bool ok = !flag[0] && mbar_wait_bounded(&full[slot], phase);
      ok = __all_sync(kFullMask, ok);
      if (!ok) {
        if (lane == 0 && !flag[0]) atomicOr(p.err, PGD_DEVERR_TIMEOUT);
        flag[0] = 1;
      } else if (!bad[slot]) {
        const __nv_bfloat16 *Ks =
            reinterpret_cast<const __nv_bfloat16 *>(smem + (size_t)slot * C::STAGE_BYTES);
        const __nv_bfloat16 *Vs = Ks + C::TILE_ELEMS;
        const int nvalid = min(BS, ctx_b - (sg.j0 + i) * BS);

        // scores (log2 domain), one (token, head) per lane per pass
        float sc[BS / 2];
#pragma unroll
        for (int it = 0; it < BS / 2; ++it) {
          const int t = 2 * it + jj;
          const uint4 raw = *reinterpret_cast<const uint4 *>(Ks + t * D + 8 * part);
          float kf[8];
          unpack8(raw, kf);
          float acc[G];
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float a = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) a = fmaf(qr[h][e], kf[e], a);
            acc[h] = a;
          }
          const float v = reduce_scatter16<G>(acc, lane);
          sc[it] = (t < nvalid) ? v : -INFINITY;
        }
        // online softmax update for this lane's head
        float tmax = sc[0];
#pragma unroll
        for (int it = 1; it < BS / 2; ++it) tmax = fmaxf(tmax, sc[it]);
        tmax = fmaxf(tmax, __shfl_xor_sync(kFullMask, tmax, 16));
        const float m_new = fmaxf(m_run, tmax);
        const float alpha = exp2f(m_run - m_new);
        float psum = 0.f;
#pragma unroll
        for (int it = 0; it < BS / 2; ++it) {
          const float pv = exp2f(sc[it] - m_new);
          psum += pv;
          if ((lane & DUPMASK) == 0) pbuf[(2 * it + jj) * G + hsel] = pv;
        }
        l_run = l_run * alpha + psum;
        m_run = m_new;
        if (lane < 16 && (lane & DUPMASK) == 0) abuf[hsel] = alpha;
        __syncwarp();

        // o = alpha * o + sum_t p_t v_t over the valid tokens only
        float al[G];
#pragma unroll
        for (int h = 0; h < G; ++h) al[h] = abuf[h];
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[h][e] *= al[h];
#pragma unroll 4
        for (int t = 0; t < nvalid; ++t) {
          const uint2 raw = *reinterpret_cast<const uint2 *>(Vs + t * D + 4 * lane);
          float vf[4];
          unpack4(raw, vf);
          float pp[G];
#pragma unroll
          for (int h = 0; h < G; ++h) pp[h] = pbuf[t * G + h];
#pragma unroll
          for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[h][e] = fmaf(pp[h], vf[e], o[h][e]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
    s += sg.n;

    // ---- merge the NW warp states of this segment
    const float l_tot = l_run + __shfl_xor_sync(kFullMask, l_run, 16);
    if (lane < 16 && (lane & DUPMASK) == 0) {
      mrg_m[w * G + hsel] = m_run;
      mrg_l[w * G + hsel] = l_tot;
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
      *reinterpret_cast<float4 *>(mrg_o + (w * G + h) * D + 4 * lane) =
          make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
    named_barrier_sync(1, NCT);

    const bool whole = (x == sg.unit_start) && (x + sg.n == sg.unit_end);
    const size_t out_row = (size_t)sg.b * p.n_q + (size_t)sg.g * G;
    const size_t slot_row = ((size_t)unit + (size_t)cta) * G;
    for (int k = ct; k < G * D / 2; k += NCT) {
      const int h = k / (D / 2), e = 2 * (k % (D / 2));
      float M = -INFINITY;
#pragma unroll
      for (int ww = 0; ww < NW; ++ww) M = fmaxf(M, mrg_m[ww * G + h]);
      float L = 0.f, O0 = 0.f, O1 = 0.f;
#pragma unroll
      for (int ww = 0; ww < NW; ++ww) {
        const float mw = mrg_m[ww * G + h];
        if (mw == -INFINITY) continue;
        const float cf = exp2f(mw - M);
        L = fmaf(cf, mrg_l[ww * G + h], L);
        O0 = fmaf(cf, mrg_o[(ww * G + h) * D + e], O0);
        O1 = fmaf(cf, mrg_o[(ww * G + h) * D + e + 1], O1);
      }
      if (whole) {
        const float inv = 1.f / L;
        *reinterpret_cast<__nv_bfloat162 *>(p.out + (out_row + h) * D + e) =
            __floats2bfloat162_rn(O0 * inv, O1 * inv);
      } else {
        *reinterpret_cast<float2 *>(p.part_o + (slot_row + h) * D + e) = make_float2(O0, O1);
        if (e == 0)
          *reinterpret_cast<float2 *>(p.part_ml + (slot_row + h) * 2) = make_float2(M, L);
      }
    }

    if (!whole) {
      // Publish this part; the last part of the unit to arrive merges all.
      __threadfence();
      named_barrier_sync(1, NCT);
      if (ct == 0) {
        const long long c_first = (P * (sg.unit_start + 1) - 1) / X;
        const long long c_last = (P * sg.unit_end - 1) / X;
        const int n_parts = (int)(c_last - c_first + 1);
        const int before = atomicAdd(p.counters + unit, 1);
        const int last = (before == n_parts - 1);
        if (last) atomicExch(p.counters + unit, 0);  // ready for the next call
        flag[1] = last;
        flag[2] = (int)c_first;
        flag[3] = n_parts;
      }
      named_barrier_sync(1, NCT);
      if (flag[1]) {
        __threadfence();
        const int c_first = flag[2], n_parts = flag[3];
        const size_t row0 = ((size_t)unit + (size_t)c_first) * G;
        for (int k = ct; k < G * D / 2; k += NCT) {
          const int h = k / (D / 2), e = 2 * (k % (D / 2));
          float M = -INFINITY;
          for (int i = 0; i < n_parts; ++i)
            M = fmaxf(M, __ldcg(p.part_ml + (row0 + (size_t)i * G + h) * 2));
          float L = 0.f, O0 = 0.f, O1 = 0.f;
          for (int i = 0; i < n_parts; ++i) {
            const size_t r = row0 + (size_t)i * G + h;
            const float mi = __ldcg(p.part_ml + r * 2);
            if (mi == -INFINITY) continue;
            const float cf = exp2f(mi - M);
            L = fmaf(cf, __ldcg(p.part_ml + r * 2 + 1), L);
            const float2 oi = __ldcg(reinterpret_cast<const float2 *>(p.part_o + r * D + e));
            O0 = fmaf(cf, oi.x, O0);
            O1 = fmaf(cf, oi.y, O1);
          }
          const float inv = 1.f / L;
          *reinterpret_cast<__nv_bfloat162 *>(p.out + (out_row + h) * D + e) =
              __floats2bfloat162_rn(O0 * inv, O1 * inv);
        }
      }
    }
    named_barrier_sync(1, NCT);  // merge buffers and flags are reused next segment
    x += sg.n;
  }
}

// ---------------------------------------------------------------- launcher
// The dynamic shared-memory limit is raised once per device, to the size the
// largest accepted batch needs.
template <class C>
static cudaError_t ensure_smem_limit() {
  static volatile int done[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(paged_attention_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)C::smem_bytes(PGD_MAX_BATCH));
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = 1;
  return e;
}

template <class C>
static cudaError_t launch_cfg(const AttnParams &p, int grid, cudaStream_t stream) {
  cudaError_t e = ensure_smem_limit<C>();
  if (e != cudaSuccess) return e;
  paged_attention_kernel<C><<<grid, C::THREADS, C::smem_bytes(p.B), stream>>>(p);
  return cudaGetLastError();
}

template <class C>
static int occupancy_cfg(int B) {
  if (ensure_smem_limit<C>() != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, paged_attention_kernel<C>, C::THREADS,
                                                    C::smem_bytes(B)) != cudaSuccess)
    return 0;
  return n;
}

// Consumer warps and ring depth per (G, bs): 4 consumer warps; the ring holds
// 64 KiB of K/V per CTA.
template <int G, int BS>
using Cfg = AttnCfg<G, BS, 4, (BS == 16 ? 8 : 4)>;

#define PGD_DISPATCH(G_, BS_, CALL)                     \
  if (G == G_ && bs == BS_) { using C = Cfg<G_, BS_>; CALL; }

int attention_ctas_per_sm(int G, int bs, int B) {
  PGD_DISPATCH(1, 16, return occupancy_cfg<C>(B))
  PGD_DISPATCH(2, 16, return occupancy_cfg<C>(B))
  PGD_DISPATCH(4, 16, return occupancy_cfg<C>(B))
  PGD_DISPATCH(8, 16, return occupancy_cfg<C>(B))
  PGD_DISPATCH(1, 32, return occupancy_cfg<C>(B))
  PGD_DISPATCH(2, 32, return occupancy_cfg<C>(B))
  PGD_DISPATCH(4, 32, return occupancy_cfg<C>(B))
  PGD_DISPATCH(8, 32, return occupancy_cfg<C>(B))
  return 0;
}

cudaError_t attention_launch(const AttnParams &p, int G, int bs, int grid, cudaStream_t stream) {
  PGD_DISPATCH(1, 16, return launch_cfg<C>(p, grid, stream))
  PGD_DISPATCH(2, 16, return launch_cfg<C>(p, grid, stream))
  PGD_DISPATCH(4, 16, return launch_cfg<C>(p, grid, stream))
  PGD_DISPATCH(8, 16, return launch_cfg<C>(p, grid, stream))
  PGD_DISPATCH(1, 32, return launch_cfg<C>(p, grid, stream))
  PGD_DISPATCH(2, 32, return launch_cfg<C>(p, grid, stream))
  PGD_DISPATCH(4, 32, return launch_cfg<C>(p, grid, stream))
  PGD_DISPATCH(8, 32, return launch_cfg<C>(p, grid, stream))
  return cudaErrorInvalidValue;
}

#undef PGD_DISPATCH

}  // namespace pgd
