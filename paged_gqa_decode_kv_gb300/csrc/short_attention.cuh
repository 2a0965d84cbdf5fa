// short_attention.cuh -- parameter block of the short-context decode kernel
// (short_attention.cu), shared with the host code that launches it.
#pragma once

#include "pgd_device.cuh"

namespace pgd {

// One cluster of CTAs per (sequence, KV head), optionally appending the new
// token first.
struct ShortParams {
  __nv_bfloat16 *out;            // [B][n_q][D]
  const __nv_bfloat16 *q;        // [B][n_q][D]
  unsigned char *k_cache;        // bf16 tiled pools or 8-bit pools (codes + scales), written
                                 // only by the fused append
  unsigned char *v_cache;
  const __nv_bfloat16 *k_new;    // [B][n_kv][D] token to append at ctx - 1, or null
  const __nv_bfloat16 *v_new;
  const int32_t *tables;         // [B][MB]
  const int32_t *ctx;            // [B]
  int B, n_q, n_kv, MB, NB;
  float qk_scale_log2;           // scale * log2(e)
  int fp8;                       // 1: 8-bit pools
  int early;                     // 1: q, k_new, v_new and ctx live in caller memory that no
                                 // earlier kernel of the stream writes (page-locked host
                                 // buffers): read before waiting for the previous kernel
  int32_t *err;
};

cudaError_t short_attention_launch(const ShortParams &p, int G, int bs, cudaStream_t stream);
int short_max_tokens();
int short_max_units();
long long short_max_work();

}  // namespace pgd
