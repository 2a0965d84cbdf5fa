// kv_append.cu -- write each sequence's new K/V into its paged slot, and the
// device half of copy-on-write (whole-block copies).
//
// kv_append ("LLM inference systems engineering", 2.1.3: the step commits the
// pending token's K/V; "The math of Transformer inference", section 1: decode
// appends its own K and V to the cache): for sequence b at position p, the
// token row of slot p % bs in tile (table[b][p / bs], g) becomes k_new[b][g]
// (and V).  Tiles hold 8 x 8 core matrices, so the 256-byte row is sixteen
// 16-byte chunks 128 bytes apart.  A multi-query call appends T tokens per
// sequence (k_new [B][T][n_kv][d]) at positions p .. p + T - 1.  One warp per
// (sequence, token, KV head): lanes 0-15 move the K chunks and lanes 16-31
// the V chunks.  A pure copy, bit exact.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "kv_quant.cuh"
#include "pgd_device.cuh"

namespace pgd {

// 128-thread launch with programmatic stream serialization: the kernel may be
// scheduled while the previous kernel of the stream finishes (it waits for it,
// griddepcontrol.wait, before touching memory), which takes the launch
// latency off the step.
template <typename... P, typename... A>
static cudaError_t launch_pdl(void (*kernel)(P...), dim3 grid, cudaStream_t stream, A... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

__global__ void __launch_bounds__(128)
kv_append_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                 uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                 const int32_t *__restrict__ tables, const int32_t *__restrict__ pos,
                 int pos_offset, int B, int T, int n_kv, int bs, int MB, int NB, int32_t *err) {
  constexpr int kVecPerRow = kHeadDim * 2 / 16;  // 16 uint4 per 256-byte row
  pdl_wait();               // the previous kernel (which may read these slots) has completed
  pdl_launch_dependents();  // the attention that follows may start its prologue
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);  // (b * T + j) * n_kv + g
  const int lane = threadIdx.x & 31;
  if (row >= B * T * n_kv) return;
  const int bj = row / n_kv, g = row % n_kv;
  const int b = bj / T, j = bj % T;
  const long long pl = (long long)__ldg(pos + b) + pos_offset + j;
  if (pl < 0 || pl >= (long long)MB * bs) {
    if (lane == 0 && g == 0) atomicOr(err, PGD_DEVERR_BAD_POSITION);
    return;
  }
  const int p = (int)pl;
  const int blk = __ldg(tables + (size_t)b * MB + p / bs);
  if ((unsigned)blk >= (unsigned)NB) {
    if (lane == 0 && g == 0) atomicOr(err, PGD_DEVERR_BAD_BLOCK_ID);
    return;
  }
  // Tile of (blk, g), then the token's slot inside it: 16-byte chunk v of the
  // row sits in core matrix (slot / 8, v), row slot % 8 -- 128 uint4 per
  // 8-token group, 8 uint4 per core matrix.
  const int slot = p % bs;
  const size_t tile = ((size_t)blk * n_kv + g) * (size_t)bs * kVecPerRow;
  const size_t src = (size_t)row * kVecPerRow;
  const int v = lane & 15;
  const size_t dst = tile + (size_t)(slot >> 3) * 128 + (size_t)v * 8 + (size_t)(slot & 7);
  if (lane < 16)
    k_cache[dst] = __ldg(k_new + src + v);
  else
    v_cache[dst] = __ldg(v_new + src + v);
}

cudaError_t kv_append_launch(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                             const int32_t *tables, const int32_t *pos, int pos_offset, int B,
                             int T, int n_kv, int bs, int MB, int NB, int32_t *err,
                             cudaStream_t stream) {
  const long long rows = (long long)B * T * n_kv;
  if (rows == 0) return cudaSuccess;
  const int grid = (int)((rows + 3) / 4);
  return launch_pdl(kv_append_kernel, dim3(grid), stream, static_cast<const uint4 *>(k_new),
                    static_cast<const uint4 *>(v_new), static_cast<uint4 *>(k_cache),
                    static_cast<uint4 *>(v_cache), tables, pos, pos_offset, B, T, n_kv, bs, MB, NB,
                    err);
}

// kv_append into an 8-bit cache ("Ch. 6 Inference efficiency and serving",
// 6.6.1: symmetric quantisation, the scale from the largest absolute value,
// a zero row takes a positive scale; "The math of Transformer inference",
// section 11: KV scales per head and per token).  For each (sequence, KV
// head) row x of 128 bf16 values: scale = max|x| / 448 (1 if that is 0),
// code_i = E4M3(x_i / scale), both divisions IEEE binary32, the conversion
// rounding to nearest even and saturating to +-448.  The pool keeps each
// 8-token group as its codes (8-row x 16-byte core matrices) then its 8
// fp32 scales.  One warp per row pair: lanes 0-15 quantise K, 16-31 V, 8
// values per lane; the max is a shuffle reduction inside each 16-lane half.
__global__ void __launch_bounds__(128)
kv_append_fp8_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                     unsigned char *__restrict__ k_cache, unsigned char *__restrict__ v_cache,
                     const int32_t *__restrict__ tables, const int32_t *__restrict__ pos,
                     int pos_offset, int B, int n_kv, int bs, int MB, int NB, int32_t *err) {
  pdl_wait();               // the previous kernel (which may read these slots) has completed
  pdl_launch_dependents();  // the attention that follows may start its prologue
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= B * n_kv) return;
  const int b = row / n_kv, g = row % n_kv;
  const int p = __ldg(pos + b) + pos_offset;
  if (p < 0 || p >= MB * bs) {
    if (lane == 0 && g == 0) atomicOr(err, PGD_DEVERR_BAD_POSITION);
    return;
  }
  const int blk = __ldg(tables + (size_t)b * MB + p / bs);
  if ((unsigned)blk >= (unsigned)NB) {
    if (lane == 0 && g == 0) atomicOr(err, PGD_DEVERR_BAD_BLOCK_ID);
    return;
  }
  const int l = lane & 15;
  const uint4 raw = __ldg((lane < 16 ? k_new : v_new) + (size_t)row * 16 + l);
  uint32_t w[2];
  float scale;
  quantize_row_e4m3(raw, w, scale);
  const int slot = p % bs;
  unsigned char *group = (lane < 16 ? k_cache : v_cache) +
                         (((size_t)blk * n_kv + g) * (size_t)(bs / 8) + (size_t)(slot / 8)) *
                             (size_t)kGroupBytes8;
  *reinterpret_cast<uint2 *>(group + code_offset8(slot, l)) = make_uint2(w[0], w[1]);
  if (l == 0) *reinterpret_cast<float *>(group + scale_offset8(slot)) = scale;
}

cudaError_t kv_append_fp8_launch(const void *k_new, const void *v_new, void *k_cache,
                                 void *v_cache, const int32_t *tables, const int32_t *pos,
                                 int pos_offset, int B, int n_kv, int bs, int MB, int NB,
                                 int32_t *err, cudaStream_t stream) {
  const int rows = B * n_kv;
  if (rows == 0) return cudaSuccess;
  const int grid = (rows + 3) / 4;
  return launch_pdl(kv_append_fp8_kernel, dim3(grid), stream, static_cast<const uint4 *>(k_new),
                    static_cast<const uint4 *>(v_new), static_cast<unsigned char *>(k_cache),
                    static_cast<unsigned char *>(v_cache), tables, pos, pos_offset, B, n_kv, bs,
                    MB, NB, err);
}

// Copy-on-write ("Module 10: inference and serving", section "Share only
// identical state"): block src_ids[i] -> dst_ids[i], every KV head and slot,
// K and V.  grid.x = pairs, grid.y = chunks of the block; 16-byte vectors.
__global__ void __launch_bounds__(256)
copy_blocks_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                   const int32_t *__restrict__ src_ids, const int32_t *__restrict__ dst_ids,
                   int block_vecs, int NB, int32_t *err) {
  const int i = blockIdx.x;
  const int src = __ldg(src_ids + i), dst = __ldg(dst_ids + i);
  if ((unsigned)src >= (unsigned)NB || (unsigned)dst >= (unsigned)NB) {
    if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(err, PGD_DEVERR_BAD_BLOCK_ID);
    return;
  }
  const size_t s0 = (size_t)src * block_vecs, d0 = (size_t)dst * block_vecs;
  for (int v = blockIdx.y * blockDim.x + threadIdx.x; v < block_vecs;
       v += gridDim.y * blockDim.x) {
    k_cache[d0 + v] = k_cache[s0 + v];
    v_cache[d0 + v] = v_cache[s0 + v];
  }
}

cudaError_t copy_blocks_launch(void *k_cache, void *v_cache, const int32_t *src_ids,
                               const int32_t *dst_ids, int n, int n_kv, int bs, int NB,
                               int32_t *err, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const int block_vecs = n_kv * bs * kHeadDim * 2 / 16;
  int chunks = (block_vecs + 255) / 256;
  if (chunks > 64) chunks = 64;
  dim3 grid(n, chunks);
  copy_blocks_kernel<<<grid, 256, 0, stream>>>(static_cast<uint4 *>(k_cache),
                                               static_cast<uint4 *>(v_cache), src_ids, dst_ids,
                                               block_vecs, NB, err);
  return cudaGetLastError();
}

}  // namespace pgd
