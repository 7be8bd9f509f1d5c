// fp32 path for small layers: router projection and grouped expert FFN with plain FMA
// (no tensor cores: bf16/tf32 tensor inputs cannot meet an fp32 tolerance).
//
// MegaBlocks router chapter §2: the router is a linear layer without bias. GShard summary
// page, "MoE Transformer": every expert is a two-layer FFN of the dense FFN's shape.
// Lec16 Systems for MoE Models, "DeepSeek V3 MoE": SwiGLU expert, (Swish(x W1) * (x W2)) W3.
#include <math.h>

#include "internal.h"
#include "simt_f32.cuh"

namespace moe {
namespace {

__global__ void router_f32_kernel(const float* __restrict__ x, const float* __restrict__ W_g,
                                  const float* __restrict__ bias, int S, int E, int M,
                                  float* __restrict__ logits) {
  pdl_wait();
  pdl_trigger();
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= int64_t(S) * E) return;
  const int64_t t = idx / E;
  const int e = int(idx % E);
  const float* xr = x + t * M;
  const float* wr = W_g + int64_t(e) * M;
  float acc = dot_in_order(xr, wr, M, 0.f);
  if (bias) acc += bias[e];
  logits[idx] = acc;
}

// h[r, j] = act(A[r] . W[g] rows), W packed as by moe_pack_weights.
__global__ void ffn_up_f32_kernel(const float* __restrict__ A, const int32_t* __restrict__ offsets,
                                  int groups, int rows_dense, int64_t rows_cap, int M, int H,
                                  int swiglu, const float* __restrict__ W, float* __restrict__ h) {
  pdl_wait();
  pdl_trigger();
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t r = idx / H;
  const int j = int(idx % H);
  if (r >= rows_cap) return;
  int g = 0;
  if (offsets) {
    g = group_of(offsets, groups, r);
    if (g < 0) return;
  } else if (r >= rows_dense) {
    return;
  }
  const int NR = swiglu ? 2 * H : H;
  const int gate_row = swiglu ? (j / 128) * 256 + (j % 128) : j;
  const float* a = A + r * M;
  const float* wg = W + (int64_t(g) * NR + gate_row) * M;
  const float acc = dot_in_order(a, wg, M, 0.f);
  float out;
  if (swiglu) {
    const float* wu = wg + int64_t(128) * M;
    const float up = dot_in_order(a, wu, M, 0.f);
    out = acc / (1.f + expf(-acc)) * up;
  } else {
    out = acc > 0.f ? acc : 0.f;
  }
  h[r * H + j] = out;
}

// y[r, m] = scale[r] * (h[r] . W_out[g][m]).
__global__ void ffn_down_f32_kernel(const float* __restrict__ h, const int32_t* __restrict__ offsets,
                                    int groups, int rows_dense, int64_t rows_cap, int M, int H,
                                    const float* __restrict__ scale, const float* __restrict__ W,
                                    float* __restrict__ y) {
  pdl_wait();
  pdl_trigger();
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t r = idx / M;
  const int m = int(idx % M);
  if (r >= rows_cap) return;
  int g = 0;
  if (offsets) {
    g = group_of(offsets, groups, r);
    if (g < 0) return;
  } else if (r >= rows_dense) {
    return;
  }
  const float* hr = h + r * H;
  const float* w = W + (int64_t(g) * M + m) * H;
  const float acc = dot_in_order(hr, w, H, 0.f);
  y[r * M + m] = scale ? acc * scale[r] : acc;
}

}  // namespace

int launch_router_f32(const moe_config_t& c, const float* x, const float* W_g, const float* bias,
                      float* logits, cudaStream_t st) {
  const int64_t n = int64_t(c.S) * c.E;
  return launch_kernel(router_f32_kernel, dim3(unsigned((n + 255) / 256)), dim3(256), 0, st, x, W_g,
                       bias, c.S, c.E, c.M, logits);
}

int launch_ffn_up_f32(const moe_config_t& c, int H, const float* A, const int32_t* offsets,
                      int groups, int rows_dense, int64_t rows_cap, const float* W_packed,
                      float* h, unsigned* /*status*/, cudaStream_t st) {
  const int64_t n = rows_cap * H;
  return launch_kernel(ffn_up_f32_kernel, dim3(unsigned((n + 255) / 256)), dim3(256), 0, st, A,
                       offsets, groups, rows_dense, rows_cap, c.M, H, int(c.act == MOE_ACT_SWIGLU),
                       W_packed, h);
}

int launch_ffn_down_f32(const moe_config_t& c, int H, const float* h, const int32_t* offsets,
                        int groups, int rows_dense, int64_t rows_cap, const float* row_scale,
                        const float* W_out, float* y, unsigned* /*status*/, cudaStream_t st) {
  const int64_t n = rows_cap * c.M;
  return launch_kernel(ffn_down_f32_kernel, dim3(unsigned((n + 255) / 256)), dim3(256), 0, st, h,
                       offsets, groups, rows_dense, rows_cap, c.M, H, row_scale, W_out, y);
}

}  // namespace moe
