// Dispatch (gather into expert-contiguous rows), combine (gate-weighted scatter back to
// token order) and the one-time weight packing.
//
// GShard summary page: the dispatch path "dispatch -> local expert computation -> combine
// -> residual"; "Expert capacity": an overflow token gets no expert computation and passes
// through the residual connection. MegaBlocks router chapter §4: ops.gather / ops.scatter
// move token rows into and out of expert order. Lec16 Systems for MoE Models, "共享专家 vs.
// 路由专家": output = SharedFFN(h) + sum_i g_i Expert_i(h).
//
// All three are HBM-bound row copies: 16-byte vector accesses, one warp per row, a grid
// of a few CTAs per SM striding over rows, so every warp keeps several 16-byte loads in
// flight and every access is fully coalesced.
#include <cuda_bf16.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint4 ld_nc(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// x_perm[r] = x[token_of[r]] for r < offsets[E]; `units` 16-byte units per row.
__global__ void __launch_bounds__(kThreads) dispatch_kernel(const uint4* __restrict__ x,
                                                            const int32_t* __restrict__ token_of,
                                                            const int32_t* __restrict__ offsets,
                                                            int E, int S, int units, int64_t R_max,
                                                            uint4* __restrict__ x_perm) {
  pdl_wait();
  pdl_trigger();
  int64_t R = offsets[E];
  R = R < 0 ? 0 : (R > R_max ? R_max : R);
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * kThreads) >> 5;
  for (int64_t r = warp0; r < R; r += nwarps) {
    const int t = token_of[r];
    if (unsigned(t) >= unsigned(S)) continue;
    const uint4* src = x + int64_t(t) * units;
    uint4* dst = x_perm + r * units;
    int q = lane;
    for (; q + 96 < units; q += 128) {
      const uint4 a = ld_nc(src + q), b = ld_nc(src + q + 32), c = ld_nc(src + q + 64),
                  d = ld_nc(src + q + 96);
      st_stream(dst + q, a);
      st_stream(dst + q + 32, b);
      st_stream(dst + q + 64, c);
      st_stream(dst + q + 96, d);
    }
    for (; q < units; q += 32) st_stream(dst + q, ld_nc(src + q));
  }
}

template <bool kBF16>
struct Vec8 {  // 16 bytes of elements, widened to fp32
  static constexpr int n = kBF16 ? 8 : 4;
  float v[8];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.f;
  }
  __device__ __forceinline__ void add(const uint4& u) {
    if constexpr (kBF16) {
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[2 * i] += f.x;
        v[2 * i + 1] += f.y;
      }
    } else {
      v[0] += __uint_as_float(u.x);
      v[1] += __uint_as_float(u.y);
      v[2] += __uint_as_float(u.z);
      v[3] += __uint_as_float(u.w);
    }
  }
  // n fp32 values (8 for bf16 rows, 4 for fp32 rows), 16-byte aligned
  __device__ __forceinline__ void add_f32(const float* p) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    v[0] += a.x; v[1] += a.y; v[2] += a.z; v[3] += a.w;
    if constexpr (kBF16) {
      const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
      v[4] += b.x; v[5] += b.y; v[6] += b.z; v[7] += b.w;
    }
  }
  __device__ __forceinline__ uint4 pack() const {
    uint4 u;
    if constexpr (kBF16) {
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
      for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    } else {
      u.x = __float_as_uint(v[0]);
      u.y = __float_as_uint(v[1]);
      u.z = __float_as_uint(v[2]);
      u.w = __float_as_uint(v[3]);
    }
    return u;
  }
};

// y[t] = sum_{j kept, ascending} y_perm[row[t,j]] (+ shared[t]) (+ residual[t]); fp32 sum,
// one rounding. One warp per token; each lane owns 16-byte units q, q+32, ...; for two
// units at a time every row's loads are issued before any is added (KMAX >= k rows).
template <bool kBF16, int KMAX>
__global__ void __launch_bounds__(kThreads) combine_kernel(
    const uint4* __restrict__ y_perm, const int32_t* __restrict__ row, int k, int S, int units,
    int64_t R_max, const uint4* __restrict__ shared, const uint4* __restrict__ residual,
    const float* __restrict__ add32, uint4* __restrict__ y) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * kThreads) >> 5;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t t = warp0; t < S; t += nwarps) {
    int rows[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      rows[j] = -1;
      if (j < k) {
        const int r = __ldg(row + t * k + j);
        rows[j] = (r >= 0 && r < R_max) ? r : -1;
      }
    }
    for (int q0 = lane; q0 < units; q0 += 64) {
      const int q1 = q0 + 32;
      const bool has1 = q1 < units;
      uint4 v0[KMAX], v1[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        const uint4* src = y_perm + int64_t(rows[j] < 0 ? 0 : rows[j]) * units;
        v0[j] = rows[j] >= 0 ? __ldg(src + q0) : zero;
        v1[j] = (rows[j] >= 0 && has1) ? __ldg(src + q1) : zero;
      }
      const uint4 s0 = shared ? __ldg(shared + t * units + q0) : zero;
      const uint4 s1 = (shared && has1) ? __ldg(shared + t * units + q1) : zero;
      const uint4 r0 = residual ? __ldg(residual + t * units + q0) : zero;
      const uint4 r1 = (residual && has1) ? __ldg(residual + t * units + q1) : zero;
      Vec8<kBF16> a0, a1;
      a0.zero();
      a1.zero();
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (rows[j] >= 0) {
          a0.add(v0[j]);
          a1.add(v1[j]);
        }
      }
      if (shared) {
        a0.add(s0);
        a1.add(s1);
      }
      if (residual) {
        a0.add(r0);
        a1.add(r1);
      }
      if (add32) {  // an fp32 term, added before the one rounding
        constexpr int n = Vec8<kBF16>::n;
        a0.add_f32(add32 + (t * units + q0) * n);
        if (has1) a1.add_f32(add32 + (t * units + q1) * n);
      }
      __stcs(y + t * units + q0, a0.pack());
      if (has1) __stcs(y + t * units + q1, a1.pack());
    }
  }
}

// Weight packing, one pass over the destination in 16-byte units (coalesced stores).
// mode 0, first layer: logical row n of group g is W_in[g][n] (ReLU) or, for SwiGLU, in
//   blocks of 256 rows, W_in[g][128b + i] for i < 128 and W_up[g][128b + i - 128] after;
//   K = M.
// mode 1, second layer: logical row m, column k = s*H + h of group g is W[g*parts + s][m][h]
//   (parts = 1 for routed experts; the n_shared shared experts side by side).
// TILED (bf16): destination [g][N/BN][K/64][BN][64], one contiguous block per GEMM box;
// otherwise row-major [g][N][K].
template <bool TILED>
__global__ void __launch_bounds__(kThreads) pack_kernel(const uint4* __restrict__ W,
                                                        const uint4* __restrict__ W2, int mode,
                                                        int swiglu, int groups, int N, int K,
                                                        int H, int parts, int BN, int epu,
                                                        uint4* __restrict__ dst) {
  const int kunits = K / epu;
  const int64_t total = int64_t(groups) * N * kunits;
  for (int64_t u = int64_t(blockIdx.x) * kThreads + threadIdx.x; u < total;
       u += int64_t(gridDim.x) * kThreads) {
    int64_t g;
    int n, kq;
    if (TILED) {  // 8 units of 8 bf16 per 64-wide box row
      const int cu = int(u % 8);
      int64_t rest = u / 8;
      const int r = int(rest % BN);
      rest /= BN;
      const int KB = K / 64;
      const int kb = int(rest % KB);
      rest /= KB;
      const int NT = N / BN;
      const int nt = int(rest % NT);
      g = rest / NT;
      n = nt * BN + r;
      kq = kb * 8 + cu;
    } else {
      kq = int(u % kunits);
      const int64_t rest = u / kunits;
      n = int(rest % N);
      g = rest / N;
    }
    if (mode == 0) {
      const uint4* base = W;
      int srow = n;
      if (swiglu) {
        const int b = n / 256, i = n % 256;
        srow = b * 128 + (i & 127);
        if (i >= 128) base = W2;
      }
      dst[u] = base[(g * H + srow) * kunits + kq];
    } else {
      const int k = kq * epu;
      const int part = k / H, h = k % H;
      dst[u] = W[((g * parts + part) * N + n) * (H / epu) + h / epu];
    }
  }
}

unsigned grid_for(int64_t warps_needed) {
  const int64_t cap = int64_t(num_sms()) * 8;
  int64_t blocks = (warps_needed * 32 + kThreads - 1) / kThreads;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return unsigned(blocks);
}

}  // namespace

int launch_dispatch(const moe_config_t& c, int64_t R_max, const void* x, const int32_t* token_of,
                    const int32_t* offsets, void* x_perm, cudaStream_t st) {
  const int units = int(c.M * elem_bytes(c) / 16);
  return launch_kernel(dispatch_kernel, dim3(grid_for(R_max)), dim3(kThreads), 0, st,
                       static_cast<const uint4*>(x), token_of, offsets, c.E, c.S, units, R_max,
                       static_cast<uint4*>(x_perm));
}

template <bool kBF16>
int combine_dispatch_k(int k, unsigned grid, cudaStream_t st, const uint4* yp, const int32_t* row,
                       int S, int units, int64_t R_max, const uint4* sh, const uint4* res,
                       const float* add32, uint4* y) {
  auto kern = k <= 2 ? combine_kernel<kBF16, 2> : (k <= 4 ? combine_kernel<kBF16, 4> : combine_kernel<kBF16, 8>);
  return launch_kernel(kern, dim3(grid), dim3(kThreads), 0, st, yp, row, k, S, units, R_max, sh, res,
                       add32, y);
}

int launch_combine(const moe_config_t& c, const void* y_perm, const int32_t* row,
                   const void* shared_out, const void* residual, void* y, int64_t R_max,
                   cudaStream_t st, const float* add32) {
  const int units = int(c.M * elem_bytes(c) / 16);
  const unsigned grid = grid_for(c.S);
  auto yp = static_cast<const uint4*>(y_perm);
  auto sh = static_cast<const uint4*>(shared_out);
  auto res = static_cast<const uint4*>(residual);
  auto yo = static_cast<uint4*>(y);
  if (c.dtype == MOE_BF16)
    return combine_dispatch_k<true>(c.k, grid, st, yp, row, c.S, units, R_max, sh, res, add32, yo);
  return combine_dispatch_k<false>(c.k, grid, st, yp, row, c.S, units, R_max, sh, res, add32, yo);
}

namespace {
int run_pack(const moe_config_t& c, const void* W, const void* W2, int mode, int swiglu, int groups,
             int N, int K, int H, int parts, int BN, void* dst, cudaStream_t st) {
  const int epu = int(16 / elem_bytes(c));
  if (K % epu || (mode == 1 && H % epu)) return MOE_ERR_UNSUPPORTED;
  const int64_t total = int64_t(groups) * N * (K / epu);
  const unsigned grid = grid_for((total + 31) / 32);
  if (c.dtype == MOE_BF16) {
    if (BN <= 0 || N % BN || K % 64) return MOE_ERR_UNSUPPORTED;
    pack_kernel<true><<<grid, kThreads, 0, st>>>(static_cast<const uint4*>(W),
                                                 static_cast<const uint4*>(W2), mode, swiglu,
                                                 groups, N, K, H, parts, BN, epu,
                                                 static_cast<uint4*>(dst));
  } else {
    pack_kernel<false><<<grid, kThreads, 0, st>>>(static_cast<const uint4*>(W),
                                                  static_cast<const uint4*>(W2), mode, swiglu,
                                                  groups, N, K, H, parts, 0, epu,
                                                  static_cast<uint4*>(dst));
  }
  MOE_CUDA_CHECK(cudaGetLastError());
  return MOE_OK;
}
}  // namespace

int launch_pack_in(const moe_config_t& c, int groups, int H, const void* W_in, const void* W_up,
                   void* packed, cudaStream_t st) {
  const int swiglu = c.act == MOE_ACT_SWIGLU;
  const int N = swiglu ? 2 * H : H;
  const int BN = gemm_bn(N, swiglu ? EPI_SWIGLU : EPI_RELU);
  return run_pack(c, W_in, W_up, 0, swiglu, groups, N, c.M, H, 1, BN, packed, st);
}

int launch_pack_out(const moe_config_t& c, int groups, int H, int n_parts, const void* W_out,
                    void* packed, cudaStream_t st) {
  const int BN = gemm_bn(c.M, EPI_SCALE);
  return run_pack(c, W_out, nullptr, 1, 0, groups, c.M, H * n_parts, H, n_parts, BN, packed, st);
}

}  // namespace moe
