// noalloc.cu -- paged decode attention for callers that cannot allocate
// device memory.
//
// Some callers of this library cannot call cudaMalloc: code that runs as a
// plugin or callback inside another runtime's execution step (an inference
// engine's enqueue hook, for example) is handed its inputs and outputs but no
// scratch, and must not allocate there, because cudaMalloc/cudaFree can
// synchronize the device, can fail under the host runtime's memory budget,
// and fight the host runtime's own caching allocator.  For them this file
// keeps the attention kernel's split-merge scratch in a fixed array in device
// memory that belongs to the library itself.
//
// The array is a file-scope __device__ object of PGD_NOALLOC_SCRATCH_BYTES,
// present on every GPU that loads the library until the process exits.  Host
// code cannot use the array's name as a device address (on the host it names
// a stand-in), so its address is looked up with cudaGetSymbolAddress once per
// device, with that device current, on the first call made on that device.
// Every call shares the array: it keeps the contents the last call left, the
// per-unit arrival counters are cleared on the stream before each launch, and
// calls that overlap on the same GPU (issued on different streams, say) race
// on it.  Each GPU has its own copy, so calls on different GPUs do not.
#include <cuda_runtime.h>

#include <mutex>

#include "pgd_device.cuh"

namespace pgd {
pgd_status paged_attention_with_scratch(void *out, const void *q, const void *k_cache,
                                        const void *v_cache, const int32_t *tables,
                                        const int32_t *ctx, int32_t B, int32_t n_q, int32_t n_kv,
                                        int32_t d, int32_t bs, int32_t MB, int32_t NB,
                                        float scale, int32_t num_splits, void *scratch,
                                        size_t scratch_bytes, cudaStream_t stream);
pgd_status attention_args_status(const void *out, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *tables, const int32_t *ctx,
                                 int32_t B, int32_t n_q, int32_t n_kv, int32_t d, int32_t bs,
                                 int32_t MB, int32_t NB, float scale, int32_t num_splits);
pgd_status set_status_detail(pgd_status s, const char *msg);
}  // namespace pgd

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[PGD_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
pgd_status scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return pgd::set_status_detail(PGD_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices)
    return pgd::set_status_detail(PGD_ERR_UNSUPPORTED, "device index out of range");
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return pgd::set_status_detail(PGD_ERR_CUDA, "cudaGetSymbolAddress(scratch) failed");
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PGD_OK;
}

}  // namespace

extern "C" pgd_status pgd_paged_decode_attention_noalloc(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, int32_t B, int32_t n_q,
    int32_t n_kv, int32_t d, int32_t bs, int32_t MB, int32_t NB, float scale,
    int32_t num_splits, void *stream) {
  // The same checks, in the same order, as pgd_paged_decode_attention: a call
  // it would refuse is refused here with the same status before the scratch
  // is looked up, cleared or sized.
  pgd_status s = pgd::attention_args_status(out, q, k_cache, v_cache, block_tables, context_lens,
                                            B, n_q, n_kv, d, bs, MB, NB, scale, num_splits);
  if (s != PGD_OK || B == 0) return s;
  const size_t need = pgd_attention_workspace_size(B, n_q, n_kv, d, num_splits);
  if (need == 0 || need > (size_t)PGD_NOALLOC_SCRATCH_BYTES)
    return pgd::set_status_detail(
        PGD_ERR_WORKSPACE,
        "these sizes need more scratch than the fixed PGD_NOALLOC_SCRATCH_BYTES array holds");
  void *scratch = nullptr;
  s = scratch_address(&scratch);
  if (s != PGD_OK) return s;
  // The arrival counters (first B * n_kv int32 of the scratch) must start at
  // zero; clear them on the caller's stream.
  cudaError_t e = cudaMemsetAsync(scratch, 0, (size_t)B * n_kv * sizeof(int32_t),
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return pgd::set_status_detail(PGD_ERR_CUDA, "cudaMemsetAsync(scratch counters) failed");
  return pgd::paged_attention_with_scratch(out, q, k_cache, v_cache, block_tables, context_lens,
                                           B, n_q, n_kv, d, bs, MB, NB, scale, num_splits,
                                           scratch, (size_t)PGD_NOALLOC_SCRATCH_BYTES,
                                           static_cast<cudaStream_t>(stream));
}
