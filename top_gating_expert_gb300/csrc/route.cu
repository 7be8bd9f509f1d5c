// Routing: softmax / logsumexp, top-k gates, random 2nd-expert dispatch, per-(group,
// expert) capacity slots, expert-contiguous rows, aux and z losses.
//
// GShard summary page, "Top-2 gating": Expert capacity (assignments beyond an expert's
// capacity are dropped), Local group dispatching (groups of S/G consecutive tokens are
// routed independently), Random routing (the 2nd expert is dispatched with probability
// proportional to its gate), Auxiliary loss; the dispatch path's "capacity / token
// position assignment". Lec16 Systems for MoE Models, "Switch Transformer": gates =
// Softmax(KeepTopK(logits)); "MoE Kernel 优化": softmax, top-k and the token-to-expert
// table fused instead of one kernel each. MegaBlocks router chapter §2: z-loss =
// mean(logsumexp(logits)^2); §3: load-balancing loss.
//
// Three launches, all on one stream:
//   1. route_topk_kernel   one CTA per chunk of 256 tokens of one group. A sub-warp per
//      token computes max / sum-exp / top-k / gates / random-routing decision; the CTA then
//      ranks its candidates per (choice rank j, expert) with warp match + a scan over warps,
//      and writes per-chunk histograms, routed counts, softmax-probability partial sums and
//      logsumexp^2 partial sums.
//   2. route_scan_kernel   one CTA per group: exclusive scan of the chunk histograms in
//      (choice rank, chunk) order -- the GShard queue order -- giving each chunk's first slot
//      per (j, expert); kept counts per (group, expert); per-group aux-loss term. The last
//      CTA to finish (atomic ticket, no waiting) forms expert_offsets, the per-(group,
//      expert) first rows, and the two loss scalars.
//   3. route_finalize_kernel  one thread per assignment: slot, keep/drop, row, inverse map.
// Every integer output is a pure function of the logits and u: no atomics decide an order.
#include <float.h>
#include <math.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kThreads = kRouteChunk;  // one token per thread in the rank phase
constexpr int kWarps = kThreads / 32;
constexpr int kMaxE = 256;
constexpr int kMaxK = 8;

struct RouteArgs {
  const float* logits;
  const float* u;
  int S, G, E, k, Sg, n_cpg, rr, C;
  int64_t R_max;
  int32_t* expert_id;
  float* gate;
  int32_t* pos;
  uint8_t* drop;
  int32_t* row;
  int32_t* counts;
  int32_t* counts_routed;
  int32_t* offsets;
  int32_t* token_of;
  float* w_perm;
  float* aux;
  float* z;
  unsigned* status;
  unsigned* done;
  int32_t* hist;    // [n_chunks][k][E]: candidates per chunk, then each chunk's first slot
  int32_t* hroute;  // [n_chunks][E]: top-k choices per chunk (before random routing)
  float* ppart;     // [n_chunks][E]: sum of softmax probabilities per chunk
  float* zpart;     // [n_chunks]: sum of logsumexp^2 per chunk
  int32_t* rank;    // [S][k]: rank among the chunk's candidates of the same (j, e); -1 if none
  int32_t* gbase;   // [G][E]: first row of (group, expert)
  float* gaux;      // [G]
  float* gz;        // [G]
};

template <int VPL>
__global__ void __launch_bounds__(kThreads) route_topk_kernel(RouteArgs a) {
  __shared__ uint8_t s_id[kRouteChunk * kMaxK];
  __shared__ uint8_t s_cand[kRouteChunk];
  __shared__ int s_wc[kWarps][kMaxE];
  __shared__ float s_pacc[kWarps][kMaxE];
  __shared__ float s_z[kWarps];
  __shared__ int s_route[kMaxE];

  const int c = blockIdx.x;
  const int g = c / a.n_cpg, cc = c % a.n_cpg;
  const int t0 = g * a.Sg + cc * kRouteChunk;
  const int nt = min(kRouteChunk, a.Sg - cc * kRouteChunk);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, k = a.k;

  if (c == 0 && tid == 0) *a.done = 0u;  // ticket counter of route_scan_kernel
  for (int e = tid; e < E; e += kThreads) s_route[e] = 0;
  __syncthreads();

  // A sub-warp of W lanes handles one token; lane sl holds experts sl, sl+W, ...
  int W = 32;
  if (VPL == 1) {
    W = 1;
    while (W < E) W <<= 1;
  }
  const int sub = lane / W, sl = lane % W, spw = 32 / W;
  const unsigned sub_mask = (W == 32) ? 0xffffffffu : (((1u << W) - 1u) << (sub * W));

  float pacc[VPL];
#pragma unroll
  for (int v = 0; v < VPL; ++v) pacc[v] = 0.f;
  float zacc = 0.f;

  for (int i = warp * spw + sub; i < nt; i += kWarps * spw) {
    const int t = t0 + i;
    const float* lrow = a.logits + size_t(t) * E;
    float val[VPL];
    bool bad = false;
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      const int e = sl + v * W;
      float x = -INFINITY;
      if (e < E) {
        x = __ldg(lrow + e);
        if (!isfinite(x)) {
          bad = true;
          x = -INFINITY;
        }
      }
      val[v] = x;
    }
    if (bad) atomicOr(a.status, kStatusNonfinite);

    // softmax pieces
    float mx = -INFINITY;
#pragma unroll
    for (int v = 0; v < VPL; ++v) mx = fmaxf(mx, val[v]);
    for (int off = W >> 1; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(sub_mask, mx, off, W));
    if (mx == -INFINITY) mx = 0.f;  // only when every logit was non-finite (already flagged)
    float ex[VPL], sum = 0.f;
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      ex[v] = expf(val[v] - mx);
      sum += ex[v];
    }
    for (int off = W >> 1; off > 0; off >>= 1) sum += __shfl_xor_sync(sub_mask, sum, off, W);
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
#pragma unroll
    for (int v = 0; v < VPL; ++v) pacc[v] += ex[v] * inv;
    if (sl == 0) {
      const float lse = mx + logf(sum);
      zacc += lse * lse;
    }

    // top-k: k rounds of a sub-warp argmax (larger value first, then lower index)
    unsigned chosen = 0u;
    int ids[kMaxK];
    float top[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j < k) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
          const int e = sl + v * W;
          if (e < E && !((chosen >> v) & 1u) && (val[v] > bv || (val[v] == bv && e < bi))) {
            bv = val[v];
            bi = e;
          }
        }
        for (int off = W >> 1; off > 0; off >>= 1) {
          const float ov = __shfl_xor_sync(sub_mask, bv, off, W);
          const int oi = __shfl_xor_sync(sub_mask, bi, off, W);
          if (ov > bv || (ov == bv && oi < bi)) {
            bv = ov;
            bi = oi;
          }
        }
        ids[j] = bi;
        top[j] = bv;
        if (bi % W == sl) chosen |= 1u << (bi / W);
      }
    }

    if (sl == 0) {
      // gates: softmax over the k selected logits
      float gw[kMaxK], gsum = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < k) {
          gw[j] = (top[0] > -INFINITY) ? expf(top[j] - top[0]) : (j == 0 ? 1.f : 0.f);
          gsum += gw[j];
        }
      }
      unsigned cand = 0xffu;
      if (a.rr) {
        // keep the 2nd choice iff u < 2 * g2, g2 = 1 / (1 + exp(l1 - l2)), in fp64
        const double thr = 2.0 / (1.0 + exp(double(top[0]) - double(top[1])));
        if (!(double(a.u[t]) < thr)) cand &= ~2u;
      }
      s_cand[i] = uint8_t(cand);
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < k) {
          a.expert_id[size_t(t) * k + j] = ids[j];
          a.gate[size_t(t) * k + j] = gw[j] / gsum;
          s_id[i * kMaxK + j] = uint8_t(ids[j]);
          atomicAdd(&s_route[ids[j]], 1);
        }
      }
    }
  }

  // per-chunk softmax-probability sums (fixed reduction order: deterministic)
#pragma unroll
  for (int v = 0; v < VPL; ++v)
    for (int off = W; off < 32; off <<= 1) pacc[v] += __shfl_xor_sync(0xffffffffu, pacc[v], off);
  if (sub == 0) {
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      const int e = sl + v * W;
      if (e < E) s_pacc[warp][e] = pacc[v];
    }
  }
  for (int off = 16; off > 0; off >>= 1) zacc += __shfl_xor_sync(0xffffffffu, zacc, off);
  if (lane == 0) s_z[warp] = zacc;
  __syncthreads();
  for (int e = tid; e < E; e += kThreads) {
    float s = 0.f;
    for (int w = 0; w < kWarps; ++w) s += s_pacc[w][e];
    a.ppart[size_t(c) * E + e] = s;
    a.hroute[size_t(c) * E + e] = s_route[e];
  }
  if (tid == 0) {
    float s = 0.f;
    for (int w = 0; w < kWarps; ++w) s += s_z[w];
    a.zpart[c] = s;
  }

  // rank of each candidate among the chunk's earlier candidates of the same (j, e)
  const int i = tid;
  const bool valid = i < nt;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int j = 0; j < k; ++j) {
    for (int x = tid; x < kWarps * E; x += kThreads) s_wc[x / E][x % E] = 0;
    __syncthreads();
    const bool cand = valid && ((s_cand[i] >> j) & 1u);
    const int e = cand ? int(s_id[i * kMaxK + j]) : -1;
    const int key = cand ? e : (1024 + lane);
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const int rk = __popc(peers & lt_mask);
    if (cand && rk == 0) s_wc[warp][e] = __popc(peers);
    __syncthreads();
    for (int e2 = tid; e2 < E; e2 += kThreads) {
      int run = 0;
      for (int w = 0; w < kWarps; ++w) {
        const int v = s_wc[w][e2];
        s_wc[w][e2] = run;
        run += v;
      }
      a.hist[(size_t(c) * k + j) * E + e2] = run;
    }
    __syncthreads();
    if (valid) a.rank[size_t(t0 + i) * k + j] = cand ? s_wc[warp][e] + rk : -1;
    __syncthreads();
  }
}

// Sums of `ncol` columns over rows [0, n) of a row-major [n][ncol] array, in a fixed order:
// each of P segments of rows is summed in row order, then the segments in segment order.
template <typename T>
__device__ void column_sums(const T* base, int ncol, int n, T* s_part, T* out) {
  int P = 1024 / ncol;
  P = P < 1 ? 1 : (P > n ? n : P);
  if (P < 1) P = 1;
  const int L = (n + P - 1) / P;
  for (int idx = threadIdx.x; idx < ncol * P; idx += blockDim.x) {
    const int col = idx % ncol, s = idx / ncol;
    const int cb = s * L, ce = min(n, cb + L);
    T sum = T(0);
    for (int r = cb; r < ce; ++r) sum += base[size_t(r) * ncol + col];
    s_part[idx] = sum;
  }
  __syncthreads();
  for (int col = threadIdx.x; col < ncol; col += blockDim.x) {
    T sum = T(0);
    for (int s = 0; s < P; ++s) sum += s_part[s * ncol + col];
    out[col] = sum;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(1024) route_scan_kernel(RouteArgs a) {
  __shared__ int s_part[2 * 1024];
  __shared__ int s_tot[kMaxK * kMaxE];
  __shared__ int s_routed[kMaxE];
  __shared__ float s_fpart[1024];
  __shared__ float s_psum[kMaxE];
  __shared__ float s_zsum[1];
  __shared__ int s_last;

  const int g = blockIdx.x, tid = threadIdx.x;
  const int E = a.E, k = a.k, ncol = k * E, n = a.n_cpg;
  const size_t c0 = size_t(g) * n;

  // candidate histograms: exclusive scan over the group's chunks, per (j, e) column
  int P = 1024 / ncol;
  P = P < 1 ? 1 : (P > n ? n : P);
  const int L = (n + P - 1) / P;
  int32_t* hist = a.hist + c0 * ncol;
  for (int idx = tid; idx < ncol * P; idx += 1024) {
    const int col = idx % ncol, s = idx / ncol;
    const int cb = s * L, ce = min(n, cb + L);
    int sum = 0;
    for (int r = cb; r < ce; ++r) sum += hist[size_t(r) * ncol + col];
    s_part[idx] = sum;
  }
  __syncthreads();
  for (int col = tid; col < ncol; col += 1024) {
    int run = 0;
    for (int s = 0; s < P; ++s) {
      const int v = s_part[s * ncol + col];
      s_part[s * ncol + col] = run;
      run += v;
    }
    s_tot[col] = run;
  }
  __syncthreads();
  for (int idx = tid; idx < ncol * P; idx += 1024) {
    const int col = idx % ncol, s = idx / ncol;
    const int j = col / E, e = col % E;
    int run = s_part[idx];
    for (int jj = 0; jj < j; ++jj) run += s_tot[jj * E + e];  // earlier choice ranks first
    const int cb = s * L, ce = min(n, cb + L);
    for (int r = cb; r < ce; ++r) {
      const size_t o = size_t(r) * ncol + col;
      const int v = hist[o];
      hist[o] = run;
      run += v;
    }
  }
  for (int e = tid; e < E; e += 1024) {
    int cand = 0;
    for (int j = 0; j < k; ++j) cand += s_tot[j * E + e];
    a.counts[g * E + e] = (a.C >= 0 && cand > a.C) ? a.C : cand;
  }
  __syncthreads();

  // routed counts, probability sums and logsumexp^2 sum of the group
  column_sums<int>(a.hroute + c0 * E, E, n, s_part, s_routed);
  column_sums<float>(a.ppart + c0 * E, E, n, s_fpart, s_psum);
  column_sums<float>(a.zpart + c0, 1, n, s_fpart, s_zsum);
  for (int e = tid; e < E; e += 1024) a.counts_routed[g * E + e] = s_routed[e];
  if (tid == 0) {
    // E * sum_e (routed_e / (Sg*k)) * (psum_e / Sg)
    double acc = 0.0;
    for (int e = 0; e < E; ++e) acc += double(s_routed[e]) * double(s_psum[e]);
    a.gaux[g] = float(acc * double(E) / (double(a.Sg) * a.k * double(a.Sg)));
    a.gz[g] = s_zsum[0];
  }

  // the last group to finish forms the offsets and the loss scalars
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(a.done, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int e = tid; e < E; e += 1024) {
    int tot = 0;
    for (int gg = 0; gg < a.G; ++gg) tot += __ldcg(a.counts + gg * E + e);
    s_routed[e] = tot;
  }
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int e = 0; e < E; ++e) {
      const int v = s_routed[e];
      s_routed[e] = run;
      a.offsets[e] = run;
      run += v;
    }
    a.offsets[E] = run;
    double aux = 0.0, z = 0.0;
    for (int gg = 0; gg < a.G; ++gg) {
      aux += double(__ldcg(a.gaux + gg));
      z += double(__ldcg(a.gz + gg));
    }
    *a.aux = float(aux / a.G);
    *a.z = float(z / a.S);
    *a.done = 0u;
  }
  __syncthreads();
  for (int e = tid; e < E; e += 1024) {
    int run = s_routed[e];
    for (int gg = 0; gg < a.G; ++gg) {
      a.gbase[gg * E + e] = run;
      run += __ldcg(a.counts + gg * E + e);
    }
  }
}

__global__ void __launch_bounds__(256) route_finalize_kernel(RouteArgs a) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= int64_t(a.S) * a.k) return;
  const int t = int(idx / a.k), j = int(idx % a.k);
  const int e = a.expert_id[idx];
  const int g = t / a.Sg;
  const int c = g * a.n_cpg + (t - g * a.Sg) / kRouteChunk;
  const int rk = a.rank[idx];
  int pos = -1, row = -1;
  uint8_t reason = MOE_DROP_RANDOM;
  if (rk >= 0) {
    const int slot = a.hist[(size_t(c) * a.k + j) * a.E + e] + rk;
    if (a.C < 0 || slot < a.C) {
      pos = slot;
      row = a.gbase[g * a.E + e] + slot;
      reason = MOE_KEPT;
    } else {
      reason = MOE_DROP_CAPACITY;
    }
  }
  float gt = a.gate[idx];
  if (row >= 0 && row >= a.R_max) {  // cannot happen for consistent inputs
    atomicOr(a.status, kStatusDeviceData);
    row = -1;
    pos = -1;
  }
  if (row >= 0) {
    a.token_of[row] = t;
    a.w_perm[row] = gt;
  } else {
    gt = 0.f;
  }
  a.pos[idx] = pos;
  a.row[idx] = row;
  a.drop[idx] = reason;
  a.gate[idx] = gt;
}

}  // namespace

int launch_route(const moe_config_t& c, int C, const float* logits, const float* u,
                 const moe_route_out_t& out, char* ws, const WsLayout& L, cudaStream_t st) {
  RouteArgs a;
  a.logits = logits;
  a.u = u;
  a.S = c.S; a.G = c.G; a.E = c.E; a.k = c.k; a.Sg = c.S / c.G; a.n_cpg = L.n_cpg;
  a.rr = c.random_routing; a.C = C;
  a.R_max = rows_max(c, C);
  a.expert_id = out.expert_id; a.gate = out.gate; a.pos = out.pos; a.drop = out.drop_reason;
  a.row = out.row; a.counts = out.counts; a.counts_routed = out.counts_routed;
  a.offsets = out.expert_offsets; a.token_of = out.token_of; a.w_perm = out.w_perm;
  a.aux = out.aux_loss; a.z = out.z_loss;
  a.status = reinterpret_cast<unsigned*>(ws + L.status);
  a.done = reinterpret_cast<unsigned*>(ws + L.done);
  a.hist = reinterpret_cast<int32_t*>(ws + L.hist);
  a.hroute = reinterpret_cast<int32_t*>(ws + L.hroute);
  a.ppart = reinterpret_cast<float*>(ws + L.ppart);
  a.zpart = reinterpret_cast<float*>(ws + L.zpart);
  a.rank = reinterpret_cast<int32_t*>(ws + L.rank);
  a.gbase = reinterpret_cast<int32_t*>(ws + L.gbase);
  a.gaux = reinterpret_cast<float*>(ws + L.gaux);
  a.gz = reinterpret_cast<float*>(ws + L.gz);

  const dim3 g1(L.n_chunks);
  if (c.E <= 32) route_topk_kernel<1><<<g1, kThreads, 0, st>>>(a);
  else if (c.E <= 64) route_topk_kernel<2><<<g1, kThreads, 0, st>>>(a);
  else if (c.E <= 128) route_topk_kernel<4><<<g1, kThreads, 0, st>>>(a);
  else route_topk_kernel<8><<<g1, kThreads, 0, st>>>(a);
  MOE_CUDA_CHECK(cudaGetLastError());
  route_scan_kernel<<<c.G, 1024, 0, st>>>(a);
  MOE_CUDA_CHECK(cudaGetLastError());
  const int64_t n = int64_t(c.S) * c.k;
  route_finalize_kernel<<<unsigned((n + 255) / 256), 256, 0, st>>>(a);
  MOE_CUDA_CHECK(cudaGetLastError());
  return MOE_OK;
}

}  // namespace moe
