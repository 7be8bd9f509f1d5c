// The backward pass of the fp32 path (small layers), on plain FMA like its forward
// (simt_f32.cu): one thread an output element, every sum in a fixed order. The steps are
// those of the bf16 backward (api.cu, backward.cu), on row-major fp32 operands:
//   D = dy_perm . W_out (per expert), the gate partial sum_j D * h per row, the ReLU mask or
//   the SwiGLU derivative from the recomputed pre-activations, dx_perm = da . W_in; the
//   weights' gradients dW_out = (w dy)^T h and dW_in = da^T x summed over each expert's rows
//   in row order; the router's dx = dlogits . W_g and dW_g = dlogits^T x.
// MegaBlocks router chapter §3 (the gradient through the router scores); GShard summary
// page, "MoE Transformer" (the expert FFN and the gate-weighted combine).
#include <math.h>

#include "internal.h"
#include "simt_f32.cuh"

namespace moe {
namespace {

constexpr int kThreadsF32 = 256;

// The group of row r, or -1 past the last group's rows (dense: group 0 below dense_rows).
__device__ __forceinline__ int row_group(const int32_t* offsets, int groups, int dense_rows, int64_t r) {
  if (offsets) return group_of(offsets, groups, r);
  return r < dense_rows ? 0 : -1;
}

// The transposed packs of the fp32 backward, row-major [groups][N][K]:
//   mode 0: dst[g][n][k] = W[g or part][k][j], n = part * Hp + j (W_out transposed; the shared
//           experts' Hp-wide parts side by side);
//   mode 1: dst[g][n][k] = W[g][h(k)][n] with the forward pack's K order (SwiGLU: 128 gate
//           columns, then the same 128 up columns from W2, block by block).
__global__ void pack_transposed_f32_kernel(const float* __restrict__ W, const float* __restrict__ W2,
                                           int mode, int swiglu, int groups, int N, int K, int M,
                                           int Hp, int parts, float* __restrict__ dst) {
  const int64_t total = int64_t(groups) * N * K;
  for (int64_t u = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; u < total;
       u += int64_t(gridDim.x) * blockDim.x) {
    const int k = int(u % K);
    const int64_t gn = u / K;
    const int n = int(gn % N);
    const int g = int(gn / N);
    const float* base = W;
    int64_t src;
    if (mode == 0) {
      const int part = n / Hp, j = n % Hp;
      src = (int64_t(parts > 1 ? part : g) * M + k) * Hp + j;
    } else {
      int h = k;
      if (swiglu) {
        const int c = k & 255;
        h = (k >> 8) * 128 + (c & 127);
        if (c >= 128) base = W2;
      }
      src = (int64_t(g) * (swiglu ? K / 2 : K) + h) * M + n;
    }
    dst[u] = base[src];
  }
}

// D[r][j] = dy_rows[r] . Wt_out[g][j] (the gradient through GEMM 2 before the gate), into
// the first Hn columns of row r of D (row stride ldD).
__global__ void bwd_f32_d_kernel(const float* __restrict__ dy_rows, const int32_t* __restrict__ offsets,
                                 int groups, int dense_rows, int64_t rows_cap, int M, int Hn,
                                 const float* __restrict__ Wt_out, float* __restrict__ D, int ldD) {
  pdl_wait();
  pdl_trigger();
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t r = idx / Hn;
  const int j = int(idx % Hn);
  if (r >= rows_cap) return;
  const int g = row_group(offsets, groups, dense_rows, r);
  if (g < 0) return;
  D[r * ldD + j] = dot_in_order(dy_rows + r * M, Wt_out + (int64_t(g) * Hn + j) * M, M, 0.f);
}

// One warp a row: the gate partial sum_j D[r][j] h[r][j] (lanes take j = lane, lane + 32, ...
// in order, then a fixed xor tree) into gpart[r][0] (the other n_tiles - 1 entries 0); then
// with the row's gate w_r: ReLU, D[r][j] <- w_r D[r][j] where h > 0, else 0 (da, in place);
// SwiGLU, dh[r][j] = w_r D[r][j].
__global__ void bwd_f32_row_kernel(float* __restrict__ D, int ldD, const float* __restrict__ h, int Hn,
                                   const int32_t* __restrict__ offsets, int groups, int dense_rows,
                                   int64_t rows_cap, const float* __restrict__ w,
                                   float* __restrict__ gpart, int n_tiles, int swiglu,
                                   float* __restrict__ dh) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (r >= rows_cap || row_group(offsets, groups, dense_rows, r) < 0) return;
  float* d = D + r * ldD;
  const float* hr = h + r * Hn;
  float s = 0.f;
  for (int j = lane; j < Hn; j += 32) s = fmaf(d[j], hr[j], s);
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (gpart && lane == 0)
    for (int nt = 0; nt < n_tiles; ++nt) gpart[r * n_tiles + nt] = nt == 0 ? s : 0.f;
  const float scale = w ? w[r] : 1.f;
  for (int j = lane; j < Hn; j += 32) {
    const float v = scale * d[j];
    if (swiglu) dh[r * Hn + j] = v;
    else d[j] = hr[j] > 0.f ? v : 0.f;
  }
}

// SwiGLU: the pre-activations a (gate) and b (up) recomputed from x_rows and the forward's
// pack (rows of 128 gate units, then their 128 up units), and with dh: da = dh b silu'(a),
// db = dh silu(a), written at the same interleaved columns of dab (row stride 2 Hn).
__global__ void bwd_f32_swiglu_kernel(const float* __restrict__ x_rows, const int32_t* __restrict__ offsets,
                                      int groups, int dense_rows, int64_t rows_cap, int M, int Hn,
                                      const float* __restrict__ W_packed, const float* __restrict__ dh,
                                      float* __restrict__ dab) {
  pdl_wait();
  pdl_trigger();
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t r = idx / Hn;
  const int j = int(idx % Hn);
  if (r >= rows_cap) return;
  const int g = row_group(offsets, groups, dense_rows, r);
  if (g < 0) return;
  const int col = (j / 128) * 256 + (j % 128);
  const float* xr = x_rows + r * M;
  const float* wg = W_packed + (int64_t(g) * 2 * Hn + col) * M;
  const float a = dot_in_order(xr, wg, M, 0.f);
  const float b = dot_in_order(xr, wg + int64_t(128) * M, M, 0.f);
  const float d = dh[r * Hn + j];
  const float sg = 1.f / (1.f + expf(-a));
  dab[r * 2 * Hn + col] = d * b * sg * (1.f + a * (1.f - sg));
  dab[r * 2 * Hn + col + 128] = d * a * sg;
}

// dx_rows[r][m] = dab[r] . Wt_in[g][m] (the gradient through GEMM 1).
__global__ void bwd_f32_dx_kernel(const float* __restrict__ dab, int F, const int32_t* __restrict__ offsets,
                                  int groups, int dense_rows, int64_t rows_cap, int M,
                                  const float* __restrict__ Wt_in, float* __restrict__ dx_rows) {
  pdl_wait();
  pdl_trigger();
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t r = idx / M;
  const int m = int(idx % M);
  if (r >= rows_cap) return;
  const int g = row_group(offsets, groups, dense_rows, r);
  if (g < 0) return;
  dx_rows[r * M + m] = dot_in_order(dab + r * F, Wt_in + (int64_t(g) * M + m) * F, F, 0.f);
}

// out[g][a][b] = sum over the rows r of group g, in increasing r, of s_r P[r][pc(a)] Q[r][b]
// (s_r = scale[r], or 1 when scale is null). pc(a) = a (pmode 0), or SwiGLU's interleaved
// column of gate unit a (pmode 1) or of up unit a (pmode 2).
__global__ void bwd_f32_wgrad_kernel(const float* __restrict__ P, int ldP, const float* __restrict__ scale,
                                     int pmode, const float* __restrict__ Q, int ldQ,
                                     const int32_t* __restrict__ offsets, int groups, int dense_rows,
                                     int A, int Bn, float* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= int64_t(groups) * A * Bn) return;
  const int b = int(idx % Bn);
  const int a = int((idx / Bn) % A);
  const int g = int(idx / (int64_t(A) * Bn));
  const int r0 = offsets ? offsets[g] : 0, r1 = offsets ? offsets[g + 1] : dense_rows;
  const int pc = pmode == 0 ? a : (a / 128) * 256 + (a % 128) + (pmode == 2 ? 128 : 0);
  float acc = 0.f;
  for (int r = r0; r < r1; ++r) {
    const float p = scale ? scale[r] * P[int64_t(r) * ldP + pc] : P[int64_t(r) * ldP + pc];
    acc = fmaf(p, Q[int64_t(r) * ldQ + b], acc);
  }
  out[idx] = acc;
}

// The router's data and weight gradients from dlogits [S][E]:
// dx_r[t][m] = sum_e dl[t][e] W_g[e][m]; dW_g[e][m] = sum_t dl[t][e] x[t][m] (in order).
__global__ void router_dx_f32_kernel(const float* __restrict__ dl, const float* __restrict__ W_g, int S,
                                     int E, int M, float* __restrict__ dx_r) {
  pdl_wait();
  pdl_trigger();
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= int64_t(S) * M) return;
  const int64_t t = idx / M;
  const int m = int(idx % M);
  float acc = 0.f;
  for (int e = 0; e < E; ++e) acc = fmaf(dl[t * E + e], W_g[int64_t(e) * M + m], acc);
  dx_r[idx] = acc;
}

__global__ void router_dw_f32_kernel(const float* __restrict__ dl, const float* __restrict__ x, int S,
                                     int E, int M, float* __restrict__ dW_g) {
  pdl_wait();
  pdl_trigger();
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= int64_t(E) * M) return;
  const int e = int(idx / M);
  const int m = int(idx % M);
  float acc = 0.f;
  for (int t = 0; t < S; ++t) acc = fmaf(dl[int64_t(t) * E + e], x[int64_t(t) * M + m], acc);
  dW_g[idx] = acc;
}

unsigned blocks_for(int64_t n) { return unsigned((n + kThreadsF32 - 1) / kThreadsF32); }

}  // namespace

int launch_pack_transposed_f32(int mode, int swiglu, int groups, int N, int K, int M, int Hp,
                               int parts, const void* W, const void* W2, void* dst,
                               cudaStream_t st) {
  if (groups < 1 || N < 1 || K < 1 || (mode == 1 && swiglu && K % 256)) return MOE_ERR_UNSUPPORTED;
  const int64_t total = int64_t(groups) * N * K;
  int64_t grid = (total + kThreadsF32 - 1) / kThreadsF32;
  if (grid > 4096) grid = 4096;
  pack_transposed_f32_kernel<<<unsigned(grid), kThreadsF32, 0, st>>>(
      static_cast<const float*>(W), static_cast<const float*>(W2), mode, swiglu, groups, N, K, M,
      Hp, parts, static_cast<float*>(dst));
  MOE_CUDA_CHECK(cudaGetLastError());
  return MOE_OK;
}

int ffn_backward_data_f32(const FfnBwdF32& f, cudaStream_t st) {
  const int Hn = f.Hn, M = f.M, F = f.swiglu ? 2 * Hn : Hn;
  float* D = static_cast<float*>(f.dab);  // D in dab's first Hn columns, then da (ReLU)
  int rc = launch_kernel(bwd_f32_d_kernel, dim3(blocks_for(f.rows_cap * Hn)), dim3(kThreadsF32), 0, st,
                         static_cast<const float*>(f.dy_rows), f.offsets, f.groups, f.dense_rows,
                         f.rows_cap, M, Hn, static_cast<const float*>(f.Wt_out), D, F);
  if (rc != MOE_OK) return rc;
  rc = launch_kernel(bwd_f32_row_kernel, dim3(blocks_for(f.rows_cap * 32)), dim3(kThreadsF32), 0, st, D,
                     F, static_cast<const float*>(f.h), Hn, f.offsets, f.groups, f.dense_rows,
                     f.rows_cap, f.w, f.gpart, f.n_tiles, f.swiglu, static_cast<float*>(f.dh));
  if (rc != MOE_OK) return rc;
  if (f.swiglu &&
      (rc = launch_kernel(bwd_f32_swiglu_kernel, dim3(blocks_for(f.rows_cap * Hn)), dim3(kThreadsF32), 0,
                          st, static_cast<const float*>(f.x_rows), f.offsets, f.groups, f.dense_rows,
                          f.rows_cap, M, Hn, static_cast<const float*>(f.W_in_packed),
                          static_cast<const float*>(f.dh), D)) != MOE_OK)
    return rc;
  return launch_kernel(bwd_f32_dx_kernel, dim3(blocks_for(f.rows_cap * M)), dim3(kThreadsF32), 0, st,
                       static_cast<const float*>(f.dab), F, f.offsets, f.groups, f.dense_rows,
                       f.rows_cap, M, static_cast<const float*>(f.Wt_in),
                       static_cast<float*>(f.dx_rows));
}

int weight_grad_f32(const void* P, int ldP, const float* scale, int pmode, const void* Q, int ldQ,
                    const int32_t* offsets, int groups, int dense_rows, int A, int Bn, float* out,
                    cudaStream_t st) {
  return launch_kernel(bwd_f32_wgrad_kernel, dim3(blocks_for(int64_t(groups) * A * Bn)),
                       dim3(kThreadsF32), 0, st, static_cast<const float*>(P), ldP, scale, pmode,
                       static_cast<const float*>(Q), ldQ, offsets, groups, dense_rows, A, Bn, out);
}

int router_grads_f32(const moe_config_t& c, const float* dlogits, const void* x, const void* W_g,
                     float* dx_r, float* dW_g, cudaStream_t st) {
  int rc = launch_kernel(router_dx_f32_kernel, dim3(blocks_for(int64_t(c.S) * c.M)), dim3(kThreadsF32), 0,
                         st, dlogits, static_cast<const float*>(W_g), c.S, c.E, c.M, dx_r);
  if (rc != MOE_OK) return rc;
  return launch_kernel(router_dw_f32_kernel, dim3(blocks_for(int64_t(c.E) * c.M)), dim3(kThreadsF32), 0,
                       st, dlogits, static_cast<const float*>(x), c.S, c.E, c.M, dW_g);
}

}  // namespace moe
