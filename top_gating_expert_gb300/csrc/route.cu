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
// Three launches, all on one stream (the per-chunk kernels live in route_kernels.cuh):
//   1. route_topk_kernel   one CTA per chunk of 128 tokens of one group. The chunk's logits
//      are staged into padded shared memory with coalesced loads; TPT consecutive threads
//      share a token, each keeping a sorted top-k of its slice of the experts (larger logit
//      first, lower index on ties), merged by K rounds of a TPT-lane shuffle arg-best; then
//      max, sum-exp, gates and the random-routing decision. The CTA ranks its candidates per
//      (choice rank j, expert) with warp match + a scan over warps, and writes per-chunk
//      histograms, routed counts, per-expert softmax-probability sums and the
//      logsumexp^2 sum (fixed summation orders: deterministic). router_topk_kernel does the
//      same after computing the chunk's logits itself on the tensor cores.
//   2. route_scan_kernel   X CTAs per group, each a slice of the experts: exclusive scans of
//      the chunk histograms in (choice rank, chunk) order -- the GShard queue order -- giving
//      each chunk's first slot per (j, expert); kept counts per (group, expert); the slice's
//      aux-loss term. The last CTA to finish (atomic ticket, no waiting) forms
//      expert_offsets, the per-(group, expert) first rows and the two loss scalars.
//   3. route_finalize_kernel  one thread per assignment: slot, keep/drop, row, inverse map.
// Every integer output is a pure function of the logits and u: no atomic decides an order.
#include <algorithm>

#include "route_kernels.cuh"

namespace moe {
namespace {

constexpr int kScanThreads = 256;
constexpr int kBatch = 16;  // loads kept in flight per thread in the scans

// Fixed-order block reduction of one float per thread (all threads participate).
__device__ float block_sum(float v, float* s_red) {
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  float r = 0.f;
  if (warp == 0) {
    r = lane < int(blockDim.x >> 5) ? s_red[lane] : 0.f;
    for (int off = 16; off > 0; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
  }
  __syncthreads();
  return r;  // valid in thread 0
}

// CTA (g, x) of a G x X grid takes group g's experts e0 .. e0 + nw - 1 (e0 = x * ew): the
// columns (j, e) of the chunk histograms, each an exclusive scan down the group's chunks
// offset by the group's candidates of choice ranks j' < j for e (the GShard queue order:
// all first choices, then all second choices, each in token order), and the sums over
// chunks of the routed counts and probability sums of its experts (the group's
// logsumexp^2 sum in the x = 0 CTA). A thread owns one (segment of chunks, column) and
// issues all its loads before using any. The last CTA to finish (atomic ticket, no
// waiting) forms expert_offsets, the first row of every (group, expert) and the two loss
// scalars. Every sum has a fixed order.
__global__ void __launch_bounds__(kScanThreads) route_scan_kernel(RouteArgs a, int X, int ew) {
  __shared__ int s_ph[kScanThreads];      // hist segment sums, then exclusive prefixes
  __shared__ int s_pr[kScanThreads];      // routed-count segment sums (j = 0 columns)
  __shared__ float s_pp[kScanThreads];    // probability segment sums (j = 0 columns)
  __shared__ float s_pz[kScanThreads];    // logsumexp^2 segment sums (column 0, x = 0)
  __shared__ int s_tot[kScanThreads];     // column totals
  __shared__ int s_routed[kScanThreads];
  __shared__ float s_psum[kScanThreads];
  __shared__ float s_red[kScanThreads / 32];
  __shared__ int s_wsum[kScanThreads / 32];
  __shared__ int s_last;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.x / X, x = blockIdx.x % X;
  const int E = a.E, k = a.k, n = a.n_cpg, KE = k * E;
  const int e0 = x * ew, nw = min(ew, E - e0);
  const int ncol = k * nw;  // <= kScanThreads (host)
  int P = kScanThreads / ncol;
  P = P < 1 ? 1 : (P > n ? n : P);
  const int L = (n + P - 1) / P;
  pdl_wait();
  pdl_trigger();

  const int col = tid % ncol, seg = tid / ncol;
  const bool active = seg < P;
  const int j = col / nw, el = col % nw, e = e0 + el;
  const bool lead = j == 0;
  const bool zl = x == 0 && col == 0;
  const int cb = min(n, seg * L), ce = min(n, cb + L);
  const size_t c0 = size_t(g) * n;
  int32_t* __restrict__ hist = a.hist + c0 * KE + size_t(j) * E + e;  // rows KE apart
  const int32_t* __restrict__ hr = a.hroute + c0 * E + e;
  const float* __restrict__ pp = a.ppart + c0 * E + e;
  const float* __restrict__ zp = a.zpart + c0;

  int keep[kBatch];
  int hs = 0, rs = 0;
  float ps = 0.f, zs = 0.f;
  if (active) {
    for (int r0 = cb; r0 < ce; r0 += kBatch) {
      int v[kBatch], w[kBatch];
      float p[kBatch], z[kBatch];
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const bool in = r0 + q < ce;
        v[q] = in ? hist[size_t(r0 + q) * KE] : 0;
        w[q] = (in && lead) ? hr[size_t(r0 + q) * E] : 0;
        p[q] = (in && lead) ? pp[size_t(r0 + q) * E] : 0.f;
        z[q] = (in && zl) ? zp[r0 + q] : 0.f;
      }
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        hs += v[q];
        rs += w[q];
        ps += p[q];
        zs += z[q];
        if (r0 == cb) keep[q] = v[q];
      }
    }
  }
  s_ph[tid] = hs;
  s_pr[tid] = rs;
  s_pp[tid] = ps;
  s_pz[tid] = zs;
  __syncthreads();

  // per column, over its P segments in order: exclusive prefix (in place) and totals
  if (P <= 8) {
    if (tid < ncol) {
      int run = 0, rr = 0;
      float pr = 0.f, zr = 0.f;
      for (int s = 0; s < P; ++s) {
        const int i = s * ncol + tid;
        const int v = s_ph[i];
        s_ph[i] = run;
        run += v;
        rr += s_pr[i];
        pr += s_pp[i];
        zr += s_pz[i];
      }
      s_tot[tid] = run;
      if (tid < nw) {
        s_routed[tid] = rr;
        s_psum[tid] = pr;
      }
      if (tid == 0 && x == 0) a.gz[g] = zr;
    }
  } else {  // one warp per column: lane l takes segments l*per .. l*per + per - 1
    const int per = (P + 31) / 32;
    for (int cl = warp; cl < ncol; cl += kScanThreads / 32) {
      const int s0 = lane * per, s1 = min(P, s0 + per);
      int loc = 0, rr = 0;
      float pr = 0.f, zr = 0.f;
      for (int s = s0; s < s1; ++s) {
        const int i = s * ncol + cl;
        loc += s_ph[i];
        rr += s_pr[i];
        pr += s_pp[i];
        zr += s_pz[i];
      }
      int inc = loc;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += v;
      }
      int run = inc - loc;
      for (int s = s0; s < s1; ++s) {
        const int i = s * ncol + cl;
        const int v = s_ph[i];
        s_ph[i] = run;
        run += v;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        rr += __shfl_xor_sync(0xffffffffu, rr, off);
        pr += __shfl_xor_sync(0xffffffffu, pr, off);
        zr += __shfl_xor_sync(0xffffffffu, zr, off);
      }
      if (lane == 31) s_tot[cl] = inc;
      if (lane == 0) {
        if (cl < nw) {
          s_routed[cl] = rr;
          s_psum[cl] = pr;
        }
        if (cl == 0 && x == 0) a.gz[g] = zr;
      }
    }
  }
  __syncthreads();

  // first slot of every (chunk, j, e) of the segment
  if (active && cb < ce) {
    int run = s_ph[seg * ncol + col];
    for (int jj = 0; jj < j; ++jj) run += s_tot[jj * nw + el];
    if (L <= kBatch) {
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        if (cb + q < ce) {
          hist[size_t(cb + q) * KE] = run;
          run += keep[q];
        }
      }
    } else {
      for (int r0 = cb; r0 < ce; r0 += kBatch) {
        int v[kBatch];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) v[q] = (r0 + q < ce) ? hist[size_t(r0 + q) * KE] : 0;
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
          if (r0 + q < ce) hist[size_t(r0 + q) * KE] = run;
          run += v[q];
        }
      }
    }
  }
  if (tid < nw) {
    int cand = 0;
    for (int jj = 0; jj < k; ++jj) cand += s_tot[jj * nw + tid];
    a.counts[g * E + e0 + tid] = (a.C >= 0 && cand > a.C) ? a.C : cand;
    a.counts_routed[g * E + e0 + tid] = s_routed[tid];
  }
  // this slice's share of the group's load-balancing term: sum over its experts of
  // routed_e * psum_e (lanes over experts, then a fixed tree)
  if (warp == 0) {
    float t = 0.f;
    for (int i = lane; i < nw; i += 32) t += float(s_routed[i]) * s_psum[i];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
    if (lane == 0) a.gaux[size_t(g) * X + x] = t;
  }

  // the last CTA to finish forms the offsets and the loss scalars
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(a.done, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int G = a.G;
  const int32_t* __restrict__ counts = a.counts;
  int tot = 0;  // rows of expert tid over all groups
  if (tid < E) {
    for (int g0 = 0; g0 < G; g0 += kBatch) {
      int v[kBatch];
#pragma unroll
      for (int q = 0; q < kBatch; ++q) v[q] = (g0 + q < G) ? __ldcg(counts + (g0 + q) * E + tid) : 0;
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        tot += v[q];
        if (g0 == 0) keep[q] = v[q];
      }
    }
  }
  // exclusive scan of tot over the experts (thread order)
  int inc = tot;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += v;
  }
  if (lane == 31) s_wsum[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int v = lane < kScanThreads / 32 ? s_wsum[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += u;
    }
    if (lane < kScanThreads / 32) s_wsum[lane] = v;  // inclusive over warps
  }
  __syncthreads();
  const int off_e = inc - tot + (warp > 0 ? s_wsum[warp - 1] : 0);
  if (tid < E) {
    a.offsets[tid] = off_e;
    if (tid == E - 1) a.offsets[E] = off_e + tot;
    int run = off_e;
    if (G <= kBatch) {
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        if (q < G) {
          a.gbase[q * E + tid] = run;
          run += keep[q];
        }
      }
    } else {
      for (int g0 = 0; g0 < G; g0 += kBatch) {
        int v[kBatch];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) v[q] = (g0 + q < G) ? __ldcg(counts + (g0 + q) * E + tid) : 0;
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
          if (g0 + q < G) a.gbase[(g0 + q) * E + tid] = run;
          run += v[q];
        }
      }
    }
  }
  // losses: aux = mean over groups of E * sum_e f_e P_e (f_e = routed_e / (Sg k),
  // P_e = psum_e / Sg); z = mean over tokens of logsumexp^2. Fixed-order sums.
  // With many expert slices a group (X > 8: few groups, as in single-group layers) a warp
  // sums a group's slices (lanes over slices, then a fixed shuffle tree) instead of one
  // thread walking them: those loads would otherwise form one long dependent chain.
  float ga = 0.f, gzs = 0.f;
  const double gscale = double(E) / (double(a.Sg) * a.k * double(a.Sg));
  if (X > 8) {
    for (int gg = warp; gg < G; gg += kScanThreads / 32) {
      float tsum = 0.f;
      for (int xx = lane; xx < X; xx += 32) tsum += __ldcg(a.gaux + size_t(gg) * X + xx);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) tsum += __shfl_xor_sync(0xffffffffu, tsum, off);
      if (lane == 0) {
        ga += float(double(tsum) * gscale);
        gzs += __ldcg(a.gz + gg);
      }
    }
  } else {
    for (int gg = tid; gg < G; gg += kScanThreads) {
      float tsum = 0.f;
      for (int xx = 0; xx < X; ++xx) tsum += __ldcg(a.gaux + size_t(gg) * X + xx);
      ga += float(double(tsum) * gscale);
      gzs += __ldcg(a.gz + gg);
    }
  }
  ga = block_sum(ga, s_red);
  gzs = block_sum(gzs, s_red);
  if (tid == 0) {
    *a.aux = ga / float(G);
    *a.z = gzs / float(a.S);
    *a.done = 0u;
  }
}

// Assignment idx = t * k + j: slot, keep/drop, row, inverse map. Returns the row (-1 if
// not kept).
__device__ __forceinline__ int finalize_assignment(const RouteArgs& a, int64_t idx) {
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
  return row;
}

__global__ void __launch_bounds__(256) route_finalize_kernel(RouteArgs a) {
  pdl_wait();
  pdl_trigger();
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= int64_t(a.S) * a.k) return;
  finalize_assignment(a, idx);
}

// The finalize step fused with the dispatch gather (the whole-layer path): one warp per
// token; lane j < k finalizes assignment (t, j), then the warp reads x[t] once (16-byte
// units, 128 a pass) and writes it to every kept row of x_perm. Read as a gather over rows
// (x_perm[r] = x[token_of[r]]) the dispatch reads x[t] once per kept choice; read from the
// token's side it reads it once.
// Before its wait on the scan, the kernel's first kPrefetchCtas CTAs bring the first
// prefetch_bytes of the next GEMM's weights into L2 (32 KB pieces), so that they stream
// from DRAM while the routing still runs (those weights do not depend on it).
constexpr int kPrefetchCtas = 512;
constexpr int64_t kPrefetchPiece = 32768;

__global__ void __launch_bounds__(256)
    route_finalize_dispatch_kernel(RouteArgs a, const uint4* __restrict__ x, int units,
                                   uint4* __restrict__ x_perm, const char* __restrict__ pf,
                                   int64_t pf_bytes, uint4* __restrict__ h_tail, int h_units) {
  if (pf_bytes > 0 && threadIdx.x == 0) {
    const int64_t pieces = (pf_bytes + kPrefetchPiece - 1) / kPrefetchPiece;
    const int nb = min(int(gridDim.x), kPrefetchCtas);
    for (int64_t i = blockIdx.x; i < pieces && int(blockIdx.x) < nb; i += nb) {
      const int64_t o = i * kPrefetchPiece;
      prefetch_l2_bulk(pf + o, uint32_t(min(kPrefetchPiece, pf_bytes - o)));
    }
  }
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (h_tail && t < 64) {  // the 64 rows of h after the kept ones: zeros (h is written later)
    int64_t R = a.offsets[a.E];
    R = R < 0 ? 0 : (R > a.R_max ? a.R_max : R);
    uint4* hr = h_tail + (R + t) * h_units;
    for (int q = lane; q < h_units; q += 32) hr[q] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (t >= a.S) return;
  int row = -1;
  if (lane < a.k) row = finalize_assignment(a, t * a.k + lane);
  const uint4* src = x + t * units;
  for (int q0 = 0; q0 < units; q0 += 128) {
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int q = q0 + lane + 32 * i;
      if (q < units) v[i] = ld_nc_v4(src + q);
    }
    for (int j = 0; j < a.k; ++j) {
      const int r = __shfl_sync(0xffffffffu, row, j);
      if (r < 0) continue;
      uint4* dst = x_perm + int64_t(r) * units;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int q = q0 + lane + 32 * i;
        if (q < units) st_v4(dst + q, v[i]);
      }
    }
  }
}

bool uses_variants(const moe_config_t& c) {
  return c.gate_norm != MOE_GATE_SOFTMAX_TOPK || c.n_expert_groups > 1 || c.uniform_assignment;
}

RouteArgs route_args(const moe_config_t& c, int C, const float* logits, const float* u,
                     const moe_route_out_t& out, char* ws, const WsLayout& L) {
  RouteArgs a;
  a.logits = logits;
  a.u = u;
  a.S = c.S; a.G = c.G; a.E = c.E; a.k = c.k; a.Sg = c.S / c.G; a.n_cpg = L.n_cpg;
  a.rr = c.random_routing; a.C = C;
  a.gate_norm = c.gate_norm; a.gate_p = c.gate_p;
  a.ng = c.n_expert_groups > 1 ? c.n_expert_groups : 1;
  a.tg = c.n_expert_groups > 1 ? c.topk_groups : 1;
  a.gsz = c.E / a.ng;
  a.uniform = c.uniform_assignment;
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
  return a;
}

// the two launches after the per-chunk kernel; with d, the finalize step also dispatches
int launch_scan_finalize(const moe_config_t& c, const RouteArgs& a, const DispatchFuse* d,
                         cudaStream_t st) {
  // experts per scan CTA: about 2048 values of a group per CTA, at most kScanThreads columns
  const int64_t vals = int64_t(a.n_cpg) * (int64_t(c.k) * c.E + 2 * c.E + 1);
  int X = int((vals + 2047) / 2048);
  if (X > c.E) X = c.E;
  if (X < 1) X = 1;
  int ew = (c.E + X - 1) / X;
  if (ew > kScanThreads / c.k) ew = kScanThreads / c.k;
  X = (c.E + ew - 1) / ew;
  int rc = launch_kernel(route_scan_kernel, dim3(unsigned(c.G * X)), dim3(kScanThreads), 0, st, a, X,
                         ew);
  if (rc != MOE_OK) return rc;
  if (d) {
    const int units = int(int64_t(c.M) * elem_bytes(c) / 16);
    const int64_t warps = std::max<int64_t>(c.S, d->h_tail ? 64 : 1);  // 64: h's tail rows
    return launch_kernel(route_finalize_dispatch_kernel, dim3(unsigned((warps * 32 + 255) / 256)),
                         dim3(256), 0, st, a, static_cast<const uint4*>(d->x), units,
                         static_cast<uint4*>(d->x_perm), static_cast<const char*>(d->prefetch),
                         d->prefetch ? (d->prefetch_bytes & ~int64_t(15)) : int64_t(0),
                         static_cast<uint4*>(d->h_tail), d->h_tail ? d->h_cols / 8 : 0);
  }
  const int64_t n = int64_t(c.S) * c.k;
  return launch_kernel(route_finalize_kernel, dim3(unsigned((n + 255) / 256)), dim3(256), 0, st, a);
}

}  // namespace

int launch_route(const moe_config_t& c, int C, const float* logits, const float* u,
                 const moe_route_out_t& out, char* ws, const WsLayout& L, cudaStream_t st,
                 const DispatchFuse* d) {
  if (reinterpret_cast<uintptr_t>(logits) % 16 != 0) return MOE_ERR_INVALID_ARG;
  const RouteArgs a = route_args(c, C, logits, u, out, ws, L);
  const int rc = uses_variants(c) ? launch_topk_chunks_variants(a, L.n_chunks, st)
                                  : launch_topk_chunks(a, L.n_chunks, st);
  if (rc != MOE_OK) return rc;
  return launch_scan_finalize(c, a, d, st);
}

int launch_router_route(const moe_config_t& c, int C, const void* x, const void* W_g,
                        const float* bias, const float* u, float* logits_out,
                        const moe_route_out_t& out, char* ws, const WsLayout& L, cudaStream_t st,
                        const DispatchFuse* d) {
  FusedRouterArgs f;
  f.bias = bias;
  f.logits_out = logits_out;
  f.Mdim = c.M;
  f.BN = gemm_bn(c.E, EPI_F32_BIAS);
  if (f.BN == 0 || c.M % 64 != 0 || c.M <= 0) return MOE_ERR_UNSUPPORTED;
  f.stages = 0;  // set per launch shape
  CUtensorMap tx, tw;
  int rc = make_tma_map_rows(&tx, x, c.S, c.M, 128);
  if (rc != MOE_OK) return rc;
  if ((rc = make_tma_map_rows(&tw, W_g, c.E, c.M, f.BN)) != MOE_OK) return rc;
  const RouteArgs a = route_args(c, C, nullptr, u, out, ws, L);
  rc = uses_variants(c) ? launch_router_chunks_variants(tx, tw, a, f, L.n_chunks, st)
                        : launch_router_chunks(tx, tw, a, f, L.n_chunks, st);
  if (rc != MOE_OK) return rc;
  return launch_scan_finalize(c, a, d, st);
}

}  // namespace moe
