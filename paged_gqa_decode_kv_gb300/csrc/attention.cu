// attention.cu -- the paged decode attention kernel for a bf16 cache
// (instantiated from attention_kernel.cuh).
#include "attention_kernel.cuh"

namespace pgd {

int attention_ctas_per_sm(int G, int bs, int B) { return attention_ctas_per_sm_t<false>(G, bs, B); }

cudaError_t attention_launch(const AttnParams &p, int G, int bs, int grid, cudaStream_t stream) {
  return attention_launch_t<false>(p, G, bs, grid, stream);
}

}  // namespace pgd
