// attention_fp8.cu -- the paged decode attention kernel for an 8-bit cache
// (E4M3 codes with per-(token, head) scales; instantiated from
// attention_kernel.cuh).
#include "attention_kernel.cuh"

namespace pgd {

int attention_ctas_per_sm_fp8(int G, int bs, int B) {
  return attention_ctas_per_sm_t<true>(G, bs, B);
}

cudaError_t attention_launch_fp8(const AttnParams &p, int G, int bs, int grid,
                                 cudaStream_t stream) {
  return attention_launch_t<true>(p, G, bs, grid, stream);
}

}  // namespace pgd
