// Plain-FMA helpers of the fp32 path (simt_f32.cu, backward_f32.cu).
#pragma once
#include <stdint.h>

namespace moe {

// acc + sum over i < n of a[i] * w[i], one fmaf at a time in increasing i (the scalar loop's
// order and rounding, so the result is the same bit for bit). When n is a multiple of 4 and
// both rows are 16-byte aligned, 32 floats of each row are loaded (eight 16-byte loads)
// before their 32 FMAs: the loads of a round are in flight together instead of a few at a
// time, which is what these small, latency-bound kernels wait on.
__device__ __forceinline__ float dot_in_order(const float* __restrict__ a,
                                              const float* __restrict__ w, int n, float acc) {
  int i = 0;
  if ((n & 3) == 0 &&
      ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(w)) & 15u) == 0) {
    constexpr int kRound = 32;
    for (; i + kRound <= n; i += kRound) {
      float4 av[kRound / 4], wv[kRound / 4];
#pragma unroll
      for (int q = 0; q < kRound / 4; ++q) {
        av[q] = __ldg(reinterpret_cast<const float4*>(a + i) + q);
        wv[q] = __ldg(reinterpret_cast<const float4*>(w + i) + q);
      }
#pragma unroll
      for (int q = 0; q < kRound / 4; ++q) {
        acc = fmaf(av[q].x, wv[q].x, acc);
        acc = fmaf(av[q].y, wv[q].y, acc);
        acc = fmaf(av[q].z, wv[q].z, acc);
        acc = fmaf(av[q].w, wv[q].w, acc);
      }
    }
  }
  for (; i < n; ++i) acc = fmaf(a[i], w[i], acc);
  return acc;
}

// Group (expert) of row r: the g with offsets[g] <= r < offsets[g+1]; -1 if r >= offsets[G].
__device__ __forceinline__ int group_of(const int32_t* offsets, int groups, int64_t r) {
  if (r >= offsets[groups]) return -1;
  int lo = 0, hi = groups;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (offsets[mid] <= r) lo = mid;
    else hi = mid;
  }
  return lo;
}

}  // namespace moe
