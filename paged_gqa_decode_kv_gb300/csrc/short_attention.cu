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
// the last of the cluster), which also takes the token's values from k_new /
// v_new directly: one launch for the whole decode step.
//
// Tokens are masked exactly as in the large kernel: positions past the
// context and blocks whose id is outside [0, NB) (flagged) take no weight.
// A context length outside [1, MB bs] is flagged and its rows are zero.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

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

template <int G, int BS>
__global__ void __launch_bounds__(THREADS) short_attention_kernel(const ShortParams p) {
  constexpr int VEC = kHeadDim * 2 / 16;  // 16-byte chunks per 256-byte row
  constexpr uint32_t TILE_VEC = BS * VEC;
  __shared__ __align__(16) float qs[G][kHeadDim];        // query rows, fp32
  __shared__ __align__(16) __nv_bfloat16 vs[CH][kHeadDim];  // V rows of a piece
  __shared__ __align__(16) float ps[CH][G];              // probabilities of a piece
  __shared__ float red[4][G];                            // per-warp maxima
  __shared__ int tbl[MAXB];                              // the sequence's table row
  __shared__ float st_m[G], st_l[G];                     // this CTA's state, for the merge
  __shared__ float st_o[G][kHeadDim];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int unit = (int)blockIdx.x / CL;
  const int b = unit / p.n_kv, g = unit % p.n_kv;
  // Inputs may come from the previous kernel of the stream.
  pdl_wait();
  pdl_launch_dependents();

  // Context length, table row and query rows, all loads in flight together.
  const int c = __ldg(p.ctx + b);
  const int32_t *trow = p.tables + (size_t)b * p.MB;
  if (tid < p.MB && tid < MAXB) tbl[tid] = __ldg(trow + tid);
  {
    const uint4 *qsrc = reinterpret_cast<const uint4 *>(p.q + ((size_t)b * p.n_q + g * G) * kHeadDim);
    for (int i = tid; i < G * VEC; i += THREADS) {
      float f[8];
      unpack8(__ldg(qsrc + i), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) qs[i / VEC][(i % VEC) * 8 + e] = f[e];
    }
  }
  const bool ctx_ok = c >= 1 && c <= p.MB * BS;
  if (!ctx_ok && tid == 0 && rank == 0 && g == 0) {
    atomicOr(p.err, PGD_DEVERR_BAD_CONTEXT);
    if (p.k_new) atomicOr(p.err, PGD_DEVERR_BAD_POSITION);
  }
  const int n = ctx_ok ? c : 0;
  const int t_lo = (int)((long long)n * rank / CL), t_hi = (int)((long long)n * (rank + 1) / CL);
  const int t_new = (p.k_new && ctx_ok) ? n - 1 : -1;  // appended token (in the last range)
  __syncthreads();

  // The fused append: the token row of slot t_new % BS in tile
  // (table[b][t_new / BS], g) becomes k_new[b][g] (and V), bit for bit.
  if (t_new >= t_lo && t_new < t_hi && tid < 32) {
    const int blk = tbl[t_new / BS];
    if ((unsigned)blk < (unsigned)p.NB) {
      const int slot = t_new % BS, v = lane & 15;
      const size_t dst = ((size_t)blk * p.n_kv + g) * TILE_VEC + (size_t)(slot >> 3) * 128 +
                         (size_t)v * 8 + (size_t)(slot & 7);
      const uint4 *src = reinterpret_cast<const uint4 *>(lane < 16 ? p.k_new : p.v_new) +
                         (size_t)unit * VEC + v;
      reinterpret_cast<uint4 *>(lane < 16 ? p.k_cache : p.v_cache)[dst] = __ldg(src);
    } else if (lane == 0) {
      atomicOr(p.err, PGD_DEVERR_BAD_BLOCK_ID);
    }
  }

  // Thread roles in a piece: q.k -- token j = tid / 2, dims [64 hf, 64 hf + 64);
  // V staging -- token rows 8 k + tid / 16 (k < 8), chunk tid % 16; p.v --
  // output dim tid.
  const int j = tid >> 1, hf = tid & 1;
  float m_run[G], l_run[G], o_acc[G];
#pragma unroll
  for (int h = 0; h < G; ++h) { m_run[h] = -INFINITY; l_run[h] = 0.f; o_acc[h] = 0.f; }
  bool bad_seen = false;

  for (int tb = t_lo; tb < t_hi; tb += CH) {
    const int nt = min(CH, t_hi - tb);
    // K: this thread's 8 chunks of token tb + j
    uint4 kr[8];
    bool kval = false;
    {
      const int t = tb + j;
      if (j < nt) {
        const int blk = tbl[t / BS];
        if (t == t_new) {
          const uint4 *src = reinterpret_cast<const uint4 *>(p.k_new) + (size_t)unit * VEC + hf * 8;
#pragma unroll
          for (int k = 0; k < 8; ++k) kr[k] = __ldg(src + k);
          kval = (unsigned)blk < (unsigned)p.NB;
        } else if ((unsigned)blk < (unsigned)p.NB) {
          const int slot = t % BS;
          const uint4 *src = reinterpret_cast<const uint4 *>(p.k_cache) +
                             ((size_t)blk * p.n_kv + g) * TILE_VEC + (size_t)(slot >> 3) * 128 +
                             (size_t)(hf * 8) * 8 + (size_t)(slot & 7);
#pragma unroll
          for (int k = 0; k < 8; ++k) kr[k] = __ldg(src + (size_t)k * 8);
          kval = true;
        } else {
          bad_seen = true;
        }
      }
      if (!kval) {
#pragma unroll
        for (int k = 0; k < 8; ++k) kr[k] = make_uint4(0, 0, 0, 0);
      }
    }
    // V: rows 8 k + tid / 16 of the piece, chunk tid % 16 (zeros for rows
    // that take no weight, so that no NaN reaches p.v)
    uint4 vr[CH / 8];
    {
      const int cv = tid & 15;
#pragma unroll
      for (int k = 0; k < CH / 8; ++k) {
        const int jj = 8 * k + (tid >> 4), t = tb + jj;
        vr[k] = make_uint4(0, 0, 0, 0);
        if (jj < nt) {
          const int blk = tbl[t / BS];
          if ((unsigned)blk < (unsigned)p.NB) {
            if (t == t_new) {
              vr[k] = __ldg(reinterpret_cast<const uint4 *>(p.v_new) + (size_t)unit * VEC + cv);
            } else {
              const int slot = t % BS;
              vr[k] = __ldg(reinterpret_cast<const uint4 *>(p.v_cache) +
                            ((size_t)blk * p.n_kv + g) * TILE_VEC + (size_t)(slot >> 3) * 128 +
                            (size_t)cv * 8 + (size_t)(slot & 7));
            }
          }
        }
      }
    }
    // q.k over this thread's 64 dims, then the pair's sum
    float s[G];
#pragma unroll
    for (int h = 0; h < G; ++h) s[h] = 0.f;
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
    // stage V rows (row jj, chunk cv: 16 B at column 8 cv; a warp writes two
    // whole rows, 512 contiguous bytes)
#pragma unroll
    for (int k = 0; k < CH / 8; ++k)
      *reinterpret_cast<uint4 *>(&vs[8 * k + (tid >> 4)][(tid & 15) * 8]) = vr[k];
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
    if (hf == 0 && j < CH) {
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
      const float v = __bfloat162float(vs[jj][tid]);
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
    __syncthreads();  // vs, ps and red are rewritten by the next piece
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

template <int G, int BS>
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
  return cudaLaunchKernelEx(&cfg, short_attention_kernel<G, BS>, p);
}

template <int BS>
static cudaError_t launch_bs(const ShortParams &p, int G, cudaStream_t stream) {
  switch (G) {
    case 1: return launch_g<1, BS>(p, stream);
    case 2: return launch_g<2, BS>(p, stream);
    case 4: return launch_g<4, BS>(p, stream);
    case 8: return launch_g<8, BS>(p, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace sc

// Largest context (MB * bs tokens) and number of (sequence, KV head) units
// the short-context kernel takes: at most two 64-token pieces per CTA, and
// one wave of clusters.
int short_max_tokens() { return sc::CL * 2 * sc::CH; }
int short_max_units() { return 128; }

cudaError_t short_attention_launch(const ShortParams &p, int G, int bs, cudaStream_t stream) {
  if (p.B * p.n_kv == 0) return cudaSuccess;
  if ((long long)p.MB * bs > short_max_tokens() || p.MB > sc::MAXB) return cudaErrorInvalidValue;
  return bs == 16 ? sc::launch_bs<16>(p, G, stream)
       : bs == 32 ? sc::launch_bs<32>(p, G, stream)
                  : cudaErrorInvalidValue;
}

}  // namespace pgd
