// moe_route_noalloc: routing for callers that cannot allocate device memory.
//
// The routing kernels need scratch (per-chunk histograms and ranks, partial sums, the
// status word). moe_route takes it from a caller-allocated workspace; this entry point
// takes it from a fixed array that lives in the library's own module instead, so the
// caller passes only inputs and outputs and nothing is allocated or freed per call.
//
// The array is a file-scope __device__ variable: every GPU that loads this library holds
// kNoAllocScratchBytes of it until the process exits. In host code its name is only a
// host-side stand-in, never a device address, so its device address is looked up with
// cudaGetSymbolAddress once per device (with that device current) and cached here.
#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_route_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};  // device address of g_route_scratch, per device

// Device address of the scratch array on the current device (looked up on first use).
int scratch_address(void** addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" int moe_route_noalloc(const moe_config_t* cfg, const float* logits, const float* u,
                                 const moe_route_out_t* out, int32_t* device_status,
                                 moe_stream_t stream) {
  int32_t C = 0;
  int rc = moe_capacity(cfg, &C);  // validates the configuration
  if (rc != MOE_OK) return rc;
  size_t need = 0;
  rc = moe_workspace_bytes(cfg, MOE_WS_STEP, &need);
  if (rc != MOE_OK) return rc;
  if (need > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;  // beyond the fixed maximum
  if (!logits || (cfg->random_routing && !u)) return MOE_ERR_INVALID_ARG;
  if (!out || !out->expert_id || !out->gate || !out->pos || !out->drop_reason || !out->row ||
      !out->counts || !out->counts_routed || !out->expert_offsets || !out->token_of ||
      !out->w_perm || !out->aux_loss || !out->z_loss)
    return MOE_ERR_INVALID_ARG;
  void* ws = nullptr;
  rc = scratch_address(&ws);
  if (rc != MOE_OK) return rc;
  const moe::WsLayout L = moe::ws_layout(*cfg, C);
  // The array keeps the previous call's contents: the status word must start at zero
  // (the routing kernels reset their own ticket counter).
  if (cudaMemsetAsync(static_cast<char*>(ws) + L.status, 0, sizeof(uint32_t), stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  rc = moe::launch_route(*cfg, C, logits, cfg->random_routing ? u : nullptr, *out,
                         static_cast<char*>(ws), L, stream);
  if (rc != MOE_OK) return rc;
  if (device_status &&
      cudaMemcpyAsync(device_status, static_cast<char*>(ws) + L.status, sizeof(uint32_t),
                      cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
