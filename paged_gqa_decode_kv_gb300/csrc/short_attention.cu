// short_attention.cu -- decode attention for short contexts, latency first.
//
// The same operation as the tensor-core decode kernel ("Module 10: inference
// and serving", section "Attention reads a different cache per sequence";
// "The math of Transformer inference", section 4):
//     out[b][h] = sum_t softmax_t(scale * q[b][h] . k_t) v_t,  t < ctx[b],
// with k_t / v_t of KV head h / G read through the block table from the same
// tiled pool.  When every context is short the call is bound by latency, not
// bytes: the large kernel's start-up (tensor-memory allocation, barrier
// rings, the split schedule, a long instruction stream) costs several
// microseconds before its first copy, more than the whole job.  This kernel
// keeps the start-up to a few dependent loads:
//
// - one cluster of CL = 8 CTAs per (sequence, KV head); CTA r of the cluster
//   takes the contiguous token range [r ctx / CL, (r + 1) ctx / CL) in
//   pieces of 64 tokens (at most two pieces in the sizes routed here);
// - per piece, K and V rows go straight from global memory into registers
//   (16-byte loads, all issued before the first use); q.k on the CUDA cores
//   with two threads per token (64 dims each), an online softmax over the
//   pieces (exact exp2, fp32), and p.v with one thread per output dim from V
//   staged in shared memory;
// - the CTAs' (max, sum, output) states are merged by log-sum-exp ("The math
//   of Transformer inference", section 8, sharding the KV cache along the
//   sequence; "LLM inference systems engineering", 2.8.3) through distributed
//   shared memory: after a cluster barrier CTA r reads the eight states of
//   output dims [16 r, 16 r + 16) and writes them; a second barrier keeps
//   every CTA's shared memory alive until its peers have read it.
//
// With k_new / v_new given, the new token's K/V are first written at
// position ctx - 1 exactly as kv_append does ("LLM inference systems
// engineering", 2.1.3), by the CTA whose range holds that position (always
// the last of the cluster), which also keeps the token's values in shared
// memory for its own loads: one launch for the whole decode step.
//
// Tokens are masked exactly as in the large kernel: positions past the
// context and blocks whose id is outside [0, NB) (flagged) take no weight.
// A context length outside [1, MB bs] is flagged and its rows are zero.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "kv_quant.cuh"
#include "short_attention.cuh"

namespace pgd {
namespace sc {

constexpr int CL = 8;         // CTAs per (sequence, KV head): one cluster
constexpr int CH = 64;        // tokens per piece
constexpr int THREADS = 128;  // = the head dim: one thread per output dim in p.v
constexpr int MAXB = 64;      // table entries of a sequence held in shared memory

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Full barrier of the cluster; the release/acquire pair orders each CTA's
// shared-memory writes before the peers' reads that follow.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// A 32-bit load from the shared memory of CTA `rank` of the cluster, at the
// offset that `local` has in this CTA's.
__device__ __forceinline__ float ld_cluster_f32(const float *local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

template <int G, int BS, bool FP8>
__global__ void __launch_bounds__(THREADS) short_attention_kernel(const ShortParams p) {
  constexpr int VEC = kHeadDim * 2 / 16;  // 16-byte chunks per bf16 row
  // bytes of one (block, KV head) tile: bf16 rows, or 8-token groups of
  // codes and scales
  constexpr size_t TILE = FP8 ? (size_t)(BS / 8) * kGroupBytes8 : (size_t)BS * kHeadDim * 2;
  using VT = typename std::conditional<FP8, unsigned char, __nv_bfloat16>::type;
  __shared__ __align__(16) float qs[G][kHeadDim];        // query rows, fp32
  __shared__ __align__(16) VT vs[CH][kHeadDim];          // V rows of a piece (bf16, or codes)
  __shared__ float vsc[CH];                              // their scales (8-bit cache)
  __shared__ __align__(16) float ps[CH][G];              // probabilities of a piece
  __shared__ float red[4][G];                            // per-warp maxima
  __shared__ int tbl[MAXB];                              // the sequence's table row
  __shared__ float st_m[G], st_l[G];                     // this CTA's state, for the merge
  __shared__ float st_o[G][kHeadDim];
  __shared__ __align__(16) unsigned char nk8[kHeadDim], nv8[kHeadDim];  // the appended token,
  __shared__ float nks, nvs;                                            // quantised (8-bit)
  __shared__ uint4 nkb[kHeadDim / 8], nvb[kHeadDim / 8];  // the appended token (bf16)

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int unit = (int)blockIdx.x / CL;
  const int b = unit / p.n_kv, g = unit % p.n_kv;
  // Context length, query rows and (in warp 0 of the cluster's last CTA,
  // whose range always holds the appended token) the new token's K/V row:
  // all loads in flight together.  They may come from the previous kernel
  // of the stream, so they wait for it -- unless they live in caller memory
  // that no kernel writes (`early`), where they overlap its end.
  const bool appender = p.k_new != nullptr && rank == CL - 1 && warp == 0;
  int c = 0;
  uint4 raw_new = make_uint4(0, 0, 0, 0);
  auto load_inputs = [&]() {
    c = __ldg(p.ctx + b);
    if (appender)
      raw_new = __ldg(reinterpret_cast<const uint4 *>(lane < 16 ? p.k_new : p.v_new) +
                      (size_t)unit * VEC + (lane & 15));
    const uint4 *qsrc = reinterpret_cast<const uint4 *>(p.q + ((size_t)b * p.n_q + g * G) * kHeadDim);
    for (int i = tid; i < G * VEC; i += THREADS) {
      float f[8];
      unpack8(__ldg(qsrc + i), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) qs[i / VEC][(i % VEC) * 8 + e] = f[e];
    }
  };
  // (The next launch is let in only after the wait either way: triggered
  // before the loads, the next step's CTAs queue on the SMs beside these and
  // the host-buffer step measured 8.0 us against 5.9.)
  if (p.early) load_inputs();
  pdl_wait();
  pdl_launch_dependents();
  if (!p.early) load_inputs();
  // the table row (device memory a previous kernel may write)
  const int32_t *trow = p.tables + (size_t)b * p.MB;
  if (tid < p.MB && tid < MAXB) tbl[tid] = __ldg(trow + tid);
  const bool ctx_ok = c >= 1 && c <= p.MB * BS;
  if (!ctx_ok && tid == 0 && rank == 0 && g == 0) {
    atomicOr(p.err, PGD_DEVERR_BAD_CONTEXT);
    if (p.k_new) atomicOr(p.err, PGD_DEVERR_BAD_POSITION);
  }
  const int n = ctx_ok ? c : 0;
  const int t_lo = (int)((long long)n * rank / CL), t_hi = (int)((long long)n * (rank + 1) / CL);
  const int t_new = (p.k_new && ctx_ok) ? n - 1 : -1;  // appended token (in the last range)
  __syncthreads();

  // The fused append, by warp 0 of the CTA whose range holds t_new: the
  // token row of slot t_new % BS in tile (table[b][t_new / BS], g) becomes
  // k_new[b][g] (and V) bit for bit -- or, for the 8-bit cache, its codes and
  // scale, quantised exactly as kv_append_fp8 does (lanes 0-15 K, 16-31 V);
  // the 8-bit rows are also kept here for this CTA's own use.
  if (t_new >= t_lo && t_new < t_hi && warp == 0) {
    const int blk = tbl[t_new / BS];
    const bool blk_ok = (unsigned)blk < (unsigned)p.NB;
    const int slot = t_new % BS, v = lane & 15;
    const uint4 raw = raw_new;  // (this warp is the appender)
    unsigned char *pool = lane < 16 ? p.k_cache : p.v_cache;
    if constexpr (FP8) {
      uint32_t w[2];
      float scale;
      quantize_row_e4m3(raw, w, scale);
      *reinterpret_cast<uint2 *>((lane < 16 ? nk8 : nv8) + 8 * v) = make_uint2(w[0], w[1]);
      if (v == 0) *(lane < 16 ? &nks : &nvs) = scale;
      if (blk_ok) {
        unsigned char *group = pool + (size_t)blk * p.n_kv * TILE + (size_t)g * TILE +
                               (size_t)(slot / 8) * kGroupBytes8;
        *reinterpret_cast<uint2 *>(group + code_offset8(slot, v)) = make_uint2(w[0], w[1]);
        if (v == 0) *reinterpret_cast<float *>(group + scale_offset8(slot)) = scale;
      }
    } else {
      (lane < 16 ? nkb : nvb)[v] = raw;
      if (blk_ok) {
        const size_t dst = ((size_t)blk * p.n_kv + g) * (TILE / 16) +
                           (size_t)(slot >> 3) * 128 + (size_t)v * 8 + (size_t)(slot & 7);
        reinterpret_cast<uint4 *>(pool)[dst] = raw;
      }
    }
    if (!blk_ok && lane == 0) atomicOr(p.err, PGD_DEVERR_BAD_BLOCK_ID);
  }
  __syncthreads();  // the appended row is read from shared memory by the loaders below

  // Thread roles in a piece: q.k -- token j = tid / 2, dims [64 hf, 64 hf + 64);
  // V staging -- bf16: token rows 8 k + tid / 16 (k < 8), 16-byte chunk
  // tid % 16; 8-bit: rows 16 k + tid / 8 (k < 4), 16-code chunk tid % 8, and
  // the scale of row tid (tid < 64); p.v -- output dim tid.
  const int j = tid >> 1, hf = tid & 1;
  float m_run[G], l_run[G], o_acc[G];
#pragma unroll
  for (int h = 0; h < G; ++h) { m_run[h] = -INFINITY; l_run[h] = 0.f; o_acc[h] = 0.f; }
  bool bad_seen = false;

  for (int tb = t_lo; tb < t_hi; tb += CH) {
    const int nt = min(CH, t_hi - tb);
    // ---- loads first, all in flight together: K of token tb + j (this
    // thread's 64 dims), then this thread's share of the piece's V rows
    // (zeros, and scale 0, for rows that take no weight, so that no NaN
    // reaches p.v)
    constexpr int NKV = FP8 ? 4 : 8;        // 16-byte K pieces per thread
    constexpr int NVV = FP8 ? CH / 16 : CH / 8;  // 16-byte V pieces per thread
    uint4 kr[NKV], vr[NVV];
    float ksc = 0.f, vscl = 0.f;
    const int t = tb + j;
    const int kblk = (j < nt) ? tbl[t / BS] : -1;
    const bool kval = j < nt && (unsigned)kblk < (unsigned)p.NB;
    if (j < nt && !kval) bad_seen = true;
#pragma unroll
    for (int k = 0; k < NKV; ++k) kr[k] = make_uint4(0, 0, 0, 0);
    if (kval) {
      const int slot = t % BS;
      const unsigned char *tile = p.k_cache + ((size_t)kblk * p.n_kv + g) * TILE;
      if constexpr (FP8) {
        // 4 chunks of 16 codes (dims 64 hf + 16 k ..) and the token's scale
        if (t == t_new) {
#pragma unroll
          for (int k = 0; k < 4; ++k) kr[k] = *reinterpret_cast<const uint4 *>(nk8 + 64 * hf + 16 * k);
          ksc = nks;
        } else {
          const unsigned char *group = tile + (size_t)(slot / 8) * kGroupBytes8;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            kr[k] = __ldg(reinterpret_cast<const uint4 *>(group + (4 * hf + k) * 128 + (slot & 7) * 16));
          ksc = __ldg(reinterpret_cast<const float *>(group + scale_offset8(slot)));
        }
      } else if (t == t_new) {
#pragma unroll
        for (int k = 0; k < 8; ++k) kr[k] = nkb[hf * 8 + k];
      } else {
        const uint4 *src = reinterpret_cast<const uint4 *>(tile) + (size_t)(slot >> 3) * 128 +
                           (size_t)(hf * 8) * 8 + (size_t)(slot & 7);
#pragma unroll
        for (int k = 0; k < 8; ++k) kr[k] = __ldg(src + (size_t)k * 8);  // chunks 128 B apart
      }
    }
#pragma unroll
    for (int k = 0; k < NVV; ++k) {
      // bf16: row 8 k + tid / 16, chunk tid % 16; 8-bit: row 16 k + tid / 8,
      // 16-code chunk tid % 8
      const int jj = FP8 ? 16 * k + (tid >> 3) : 8 * k + (tid >> 4);
      const int cv = FP8 ? (tid & 7) : (tid & 15);
      const int tv = tb + jj;
      vr[k] = make_uint4(0, 0, 0, 0);
      if (jj < nt) {
        const int blk = tbl[tv / BS];
        if ((unsigned)blk < (unsigned)p.NB) {
          const int slot = tv % BS;
          const unsigned char *tile = p.v_cache + ((size_t)blk * p.n_kv + g) * TILE;
          if constexpr (FP8) {
            vr[k] = (tv == t_new) ? *reinterpret_cast<const uint4 *>(nv8 + 16 * cv)
                                  : __ldg(reinterpret_cast<const uint4 *>(
                                        tile + (size_t)(slot / 8) * kGroupBytes8 + cv * 128 +
                                        (slot & 7) * 16));
          } else {
            vr[k] = (tv == t_new)
                ? nvb[cv]
                : __ldg(reinterpret_cast<const uint4 *>(tile) + (size_t)(slot >> 3) * 128 +
                        (size_t)cv * 8 + (size_t)(slot & 7));
          }
        }
      }
    }
    if (FP8 && tid < CH && tid < nt) {  // the V scale of row tid
      const int tv = tb + tid, blk = tbl[tv / BS];
      if ((unsigned)blk < (unsigned)p.NB) {
        const int slot = tv % BS;
        vscl = (tv == t_new) ? nvs
                             : __ldg(reinterpret_cast<const float *>(
                                   p.v_cache + ((size_t)blk * p.n_kv + g) * TILE +
                                   (size_t)(slot / 8) * kGroupBytes8 + scale_offset8(slot)));
      }
    }
    // ---- q.k over this thread's 64 dims
    float s[G];
#pragma unroll
    for (int h = 0; h < G; ++h) s[h] = 0.f;
    if constexpr (FP8) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t wd[4] = {kr[k].x, kr[k].y, kr[k].z, kr[k].w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 f2 = e4m3x2_to_f32x2((uint16_t)(wd[e >> 1] >> ((e & 1) * 16)));
          const int d = 64 * hf + 16 * k + 2 * e;
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float2 q2 = *reinterpret_cast<const float2 *>(&qs[h][d]);
            s[h] = fmaf(q2.x, f2.x, s[h]);
            s[h] = fmaf(q2.y, f2.y, s[h]);
          }
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h) s[h] *= ksc;
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float f[8];
        unpack8(kr[k], f);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float4 a = *reinterpret_cast<const float4 *>(&qs[h][hf * 64 + k * 8]);
          const float4 bq = *reinterpret_cast<const float4 *>(&qs[h][hf * 64 + k * 8 + 4]);
          s[h] = fmaf(a.x, f[0], s[h]);
          s[h] = fmaf(a.y, f[1], s[h]);
          s[h] = fmaf(a.z, f[2], s[h]);
          s[h] = fmaf(a.w, f[3], s[h]);
          s[h] = fmaf(bq.x, f[4], s[h]);
          s[h] = fmaf(bq.y, f[5], s[h]);
          s[h] = fmaf(bq.z, f[6], s[h]);
          s[h] = fmaf(bq.w, f[7], s[h]);
        }
      }
    }
    // ---- V rows into shared memory (bf16: a warp writes two whole rows,
    // 512 contiguous bytes; 8-bit: four rows of 128 codes)
#pragma unroll
    for (int k = 0; k < NVV; ++k) {
      const int jj = FP8 ? 16 * k + (tid >> 3) : 8 * k + (tid >> 4);
      const int col = FP8 ? 16 * (tid & 7) : 8 * (tid & 15);
      *reinterpret_cast<uint4 *>(&vs[jj][col]) = vr[k];
    }
    if (FP8 && tid < CH) vsc[tid] = vscl;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      s[h] += __shfl_xor_sync(kFullMask, s[h], 1);
      s[h] = kval ? s[h] * p.qk_scale_log2 : -INFINITY;  // log2 domain
    }
    // the piece's maximum of each row
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float m = s[h];
#pragma unroll
      for (int o = 2; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(kFullMask, m, o));
      if (lane == 0) red[warp][h] = m;
    }
    __syncthreads();
    float alpha[G], m_new[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float mc = fmaxf(fmaxf(red[0][h], red[1][h]), fmaxf(red[2][h], red[3][h]));
      m_new[h] = fmaxf(m_run[h], mc);
      // (a row still without a valid token keeps -inf and weight 0)
      alpha[h] = (m_run[h] == -INFINITY) ? 0.f : exp2f(m_run[h] - m_new[h]);
      m_run[h] = m_new[h];
    }
    if (hf == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h)
        ps[j][h] = (s[h] == -INFINITY) ? 0.f : exp2f(s[h] - m_new[h]);
    }
    __syncthreads();
    // p.v for output dim tid, and the row sums (alike in every thread)
    float acc[G], lsum[G];
#pragma unroll
    for (int h = 0; h < G; ++h) { acc[h] = 0.f; lsum[h] = 0.f; }
    for (int jj = 0; jj < nt; ++jj) {
      float v;
      if constexpr (FP8) {
        const __half h = __half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)vs[jj][tid], __NV_E4M3));
        v = __half2float(h) * vsc[jj];
      } else {
        v = __bfloat162float(vs[jj][tid]);
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float pw = ps[jj][h];
        acc[h] = fmaf(pw, v, acc[h]);
        lsum[h] += pw;
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      o_acc[h] = o_acc[h] * alpha[h] + acc[h];
      l_run[h] = l_run[h] * alpha[h] + lsum[h];
    }
    __syncthreads();  // vs, vsc, ps and red are rewritten by the next piece
  }
  if (bad_seen) atomicOr(p.err, PGD_DEVERR_BAD_BLOCK_ID);

  // This CTA's state, then the merge of the cluster's eight by output dims.
#pragma unroll
  for (int h = 0; h < G; ++h) st_o[h][tid] = o_acc[h];
  if (tid == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) { st_m[h] = m_run[h]; st_l[h] = l_run[h]; }
  }
  cluster_sync();
  if (tid < 16 * G) {
    const int h = tid / 16, d = (int)rank * 16 + (tid % 16);
    float mk[CL], lk[CL], ok[CL];
#pragma unroll
    for (int k = 0; k < CL; ++k) {
      mk[k] = ld_cluster_f32(&st_m[h], (uint32_t)k);
      lk[k] = ld_cluster_f32(&st_l[h], (uint32_t)k);
      ok[k] = ld_cluster_f32(&st_o[h][d], (uint32_t)k);
    }
    float M = mk[0];
#pragma unroll
    for (int k = 1; k < CL; ++k) M = fmaxf(M, mk[k]);
    float num = 0.f, den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int k = 0; k < CL; ++k) {
        const float w = (mk[k] == -INFINITY) ? 0.f : exp2f(mk[k] - M);
        num = fmaf(w, ok[k], num);
        den = fmaf(w, lk[k], den);
      }
    }
    const float o = den > 0.f ? num / den : 0.f;
    p.out[((size_t)b * p.n_q + g * G + h) * kHeadDim + d] = __float2bfloat16_rn(o);
  }
  cluster_sync();  // peers may still be reading this CTA's state
}

template <int G, int BS, bool FP8>
static cudaError_t launch_g(const ShortParams &p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * p.n_kv * CL));
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, short_attention_kernel<G, BS, FP8>, p);
}

template <int BS, bool FP8>
static cudaError_t launch_bs(const ShortParams &p, int G, cudaStream_t stream) {
  switch (G) {
    case 1: return launch_g<1, BS, FP8>(p, stream);
    case 2: return launch_g<2, BS, FP8>(p, stream);
    case 4: return launch_g<4, BS, FP8>(p, stream);
    case 8: return launch_g<8, BS, FP8>(p, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace sc

// Largest table width (MB * bs tokens), number of (sequence, KV head) units
// and units x width the short-context kernel takes: at most two 64-token
// pieces per CTA, about one wave of clusters (3 CTAs of 128 threads per SM by
// registers), and the work below which it measured faster than the
// tensor-core kernel (device time per append + attention step, bf16 and
// 8-bit: 8 units x 512 tokens 5.7 against 11.6 us, 32 x 1024 13.1 / 18.8,
// 64 x 512 11.7 / 13.8; beyond: 64 x 1024 19.3 / 16.6, 128 x 256 16.5 / 13.1).
int short_max_tokens() { return sc::CL * 2 * sc::CH; }
int short_max_units() { return 64; }
long long short_max_work() { return 40960; }

cudaError_t short_attention_launch(const ShortParams &p, int G, int bs, cudaStream_t stream) {
  if (p.B * p.n_kv == 0) return cudaSuccess;
  if ((long long)p.MB * bs > short_max_tokens() || p.MB > sc::MAXB) return cudaErrorInvalidValue;
  if (p.fp8)
    return bs == 16 ? sc::launch_bs<16, true>(p, G, stream)
         : bs == 32 ? sc::launch_bs<32, true>(p, G, stream)
                    : cudaErrorInvalidValue;
  return bs == 16 ? sc::launch_bs<16, false>(p, G, stream)
       : bs == 32 ? sc::launch_bs<32, false>(p, G, stream)
                  : cudaErrorInvalidValue;
}

}  // namespace pgd
