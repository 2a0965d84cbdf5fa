// read_stream.cu -- read-only streaming kernels: the HBM read bandwidth a
// kernel that only reads can reach on this GPU, measured in the same job as
// the attention kernels so that their roofline fractions have a denominator
// of the same kind ("LLM inference systems engineering", 3.8.2: keep peak and
// sustained bandwidth apart and calibrate against the access pattern being
// measured).  Two access patterns:
//   mode 0  16-byte vector loads (non-coherent, no L1 allocation) by every
//           thread of a grid of four 512-thread CTAs per SM, eight loads in
//           flight per thread, folded into a value that decides one store;
//   mode 1  the attention kernels' pattern: one CTA per SM streams its share
//           as 4 KiB bulk copies (TMA engine) into a three-stage ring of
//           64 KiB shared-memory stages, L2 evict-first; a stage is refilled
//           once its previous copies have landed.
// Each byte of the source is read once per pass.
#include <cuda_runtime.h>

#include "pgd_device.cuh"

namespace pgd {
namespace rs {

constexpr int kLoadThreads = 512, kLoadCtasPerSm = 4, kUnroll = 8;
constexpr int kPiece = 4096;                  // bytes per bulk copy
constexpr int kPiecesPerStage = 16;           // 64 KiB stages
constexpr int kStages = 3;
constexpr int kStageBytes = kPiece * kPiecesPerStage;
constexpr int kBulkSmem = kStages * kStageBytes + 1024;

// Written only if the folded value hits one particular pattern: the loads
// cannot be dropped, and in practice nothing is stored.
__device__ uint32_t g_read_sink;

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__global__ void __launch_bounds__(kLoadThreads) read_loads_kernel(const uint4 *__restrict__ src,
                                                                   size_t n16) {
  const size_t stride = (size_t)gridDim.x * kLoadThreads;
  size_t i = (size_t)blockIdx.x * kLoadThreads + threadIdx.x;
  uint32_t acc = 0;
  for (; i + (kUnroll - 1) * stride < n16; i += kUnroll * stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = ld_stream(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n16; i += stride) {
    const uint4 v = ld_stream(src + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (acc == 0x9e3779b9u) g_read_sink = acc;
}

// One warp per CTA; lanes 0..15 each issue one 4 KiB copy per stage.  CTA c
// reads pieces [n * c / grid, n * (c + 1) / grid) of the n pieces.
__global__ void __launch_bounds__(32, 1) read_bulk_kernel(const unsigned char *__restrict__ src,
                                                           long long n_pieces, int32_t *err) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *ring = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full[kStages];
  const int lane = threadIdx.x;
  if (lane == 0) {
    for (int i = 0; i < kStages; ++i) mbar_init(&full[i], 1);
    mbar_init_fence();
  }
  __syncwarp();
  const long long p0 = n_pieces * blockIdx.x / gridDim.x;
  const long long p1 = n_pieces * (blockIdx.x + 1) / gridDim.x;
  const long long n_st = (p1 - p0 + kPiecesPerStage - 1) / kPiecesPerStage;
  const uint64_t policy = l2_policy_evict_first();
  long long s = 0;
  bool failed = false;
  for (; s < n_st; ++s) {
    const int slot = (int)(s % kStages);
    const long long use = s / kStages;
    // the slot's previous copies must have landed before it is refilled
    int ok = 1;
    if (lane == 0 && use > 0)
      ok = mbar_wait_bounded(&full[slot], (uint32_t)((use - 1) & 1)) ? 1 : 0;
    ok = __shfl_sync(kFullMask, ok, 0);
    if (!ok) {
      failed = true;
      break;
    }
    const long long first = p0 + s * kPiecesPerStage;
    const int n = (int)min((long long)kPiecesPerStage, p1 - first);
    if (lane == 0) mbar_arrive_expect_tx(&full[slot], (uint32_t)(n * kPiece));
    __syncwarp();
    if (lane < n)
      bulk_copy_g2s(ring + (size_t)slot * kStageBytes + (size_t)lane * kPiece,
                    src + (size_t)(first + lane) * kPiece, kPiece, &full[slot], policy);
  }
  // no copy may still be landing when the CTA exits (phases armed: 0 .. s-1)
  if (lane == 0) {
    for (long long k = 1; k <= kStages && k <= s; ++k) {
      const long long last = s - k;
      if (!mbar_wait_bounded(&full[last % kStages], (uint32_t)((last / kStages) & 1)))
        failed = true;
    }
    if (failed) atomicOr(err, PGD_DEVERR_TIMEOUT);
  }
}

}  // namespace rs

cudaError_t read_stream_launch(const void *src, size_t bytes, int mode, int32_t *err,
                               cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (mode == 0) {
    rs::read_loads_kernel<<<sms * rs::kLoadCtasPerSm, rs::kLoadThreads, 0, stream>>>(
        static_cast<const uint4 *>(src), bytes / 16);
    return cudaGetLastError();
  }
  e = cudaFuncSetAttribute(rs::read_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           rs::kBulkSmem);
  if (e != cudaSuccess) return e;
  rs::read_bulk_kernel<<<sms, 32, rs::kBulkSmem, stream>>>(
      static_cast<const unsigned char *>(src), (long long)(bytes / rs::kPiece), err);
  return cudaGetLastError();
}

}  // namespace pgd
