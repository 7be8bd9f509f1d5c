// Instantiates router_topk_kernel (router projection fused with the routing) for the
// default routing (see route_kernels.cuh).
#include "route_kernels.cuh"

namespace moe {

int launch_router_chunks(const CUtensorMap& tx, const CUtensorMap& tw, const RouteArgs& a,
                         const FusedRouterArgs& f, int n_chunks, cudaStream_t st) {
  return launch_router_topk_any_k<false>(tx, tw, a, f, n_chunks, st);
}

}  // namespace moe
