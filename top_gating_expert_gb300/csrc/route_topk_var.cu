// Instantiates route_topk_kernel (routing from logits in memory) for the routing variants
// (see route_kernels.cuh).
#include "route_kernels.cuh"

namespace moe {

int launch_topk_chunks_variants(const RouteArgs& a, int n_chunks, cudaStream_t st) {
  return launch_topk_any_k<true>(a, n_chunks, st);
}

}  // namespace moe
