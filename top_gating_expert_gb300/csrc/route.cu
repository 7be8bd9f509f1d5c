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
#include <float.h>
#include <math.h>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = kRouteChunk;  // one token per thread
constexpr int kWarps = kThreads / 32;
constexpr int kMaxE = 256;
constexpr int kMaxK = 8;
constexpr int kScanThreads = 256;
constexpr int kBatch = 16;  // loads kept in flight per thread in the scans

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
  float* gaux;      // [G][X]: aux-loss term of each expert slice of each group
  float* gz;        // [G]
};

// GShard random routing: keep the 2nd choice iff u < 2 * g2 with g2 = 1 / (1 + exp(l1 - l2)),
// the decision of the fp64 evaluation. fp32 decides whenever u lies outside a margin that
// bounds the fp32 threshold's error: d = l1 - l2 carries <= 2^-24 relative error, expf <= 2
// ulp, the add and the division <= 1/2 ulp each, so the relative error of the fp32
// threshold is below (6 + d) * 2^-24; the margin is (8 + d) * 2^-23. Inside it (or when the
// threshold underflows) the fp64 expression decides.
__device__ __forceinline__ bool rr_keep(float l1, float l2, float u) {
  const float d = l1 - l2;
  const float thr = 2.f / (1.f + expf(d));
  if (thr > 1e-30f) {
    const float margin = thr * (8.f + d) * 1.1920929e-7f;
    if (u < thr - margin) return true;
    if (u > thr + margin) return false;
  }
  return double(u) < 2.0 / (1.0 + exp(double(l1) - double(l2)));
}

// Larger logit first; equal logits: lower expert index first.
__device__ __forceinline__ bool ranks_before(float v, int i, float w, int j) {
  return v > w || (v == w && i < j);
}

// The random-routing draw of this thread's token when it is the token's first lane (read
// early, so that its latency hides behind the staging of the logits).
template <int K, int TPT>
__device__ __forceinline__ float token_u(const RouteArgs& a, int t0, int nt) {
  const int i = int(threadIdx.x) / TPT;
  return (K == 2 && a.rr && int(threadIdx.x) % TPT == 0 && i < nt) ? __ldg(a.u + t0 + i) : 0.f;
}

// The per-chunk routing work on a chunk's logits staged in shared memory (s_log: nt rows of
// E logits, row stride ld = E + TPT). TPT threads per token (consecutive lanes), each owning
// experts sub, sub + TPT, ...; the CTA has kThreads * TPT threads, all of which call this.
// Non-finite logits count as -inf (and are flagged); each staged logit is overwritten by
// exp(logit - max of its token).
template <int K, int TPT>
__device__ __forceinline__ void topk_chunk(const RouteArgs& a, float* s_log, int c, int t0, int nt,
                                           float u_tok) {
  constexpr int kT = kThreads * TPT;
  __shared__ float s_inv[kThreads], s_pp[kT];
  __shared__ uint8_t s_id[kThreads * kMaxK];
  __shared__ uint8_t s_cand[kThreads];
  __shared__ int s_wc[kWarps][kMaxE];
  __shared__ int s_route[kMaxE];
  __shared__ float s_z[kT / 32];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, ld = E + TPT;
  if (c == 0 && tid == 0) *a.done = 0u;  // ticket counter of route_scan_kernel
  for (int e = tid; e < E; e += kT) s_route[e] = 0;
  __syncthreads();

  // token i = tid / TPT; this thread's experts: sub, sub + TPT, ...
  const int i = tid / TPT, sub = tid % TPT;
  const bool tok = i < nt;
  const unsigned tmask = TPT == 32 ? 0xffffffffu : (((1u << TPT) - 1u) << (lane & ~(TPT - 1)));
  float zacc = 0.f;
  {
    float* rowp = s_log + i * ld;
    float top[K];
    int id[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
      top[j] = -INFINITY;
      id[j] = 0x7fffffff;
    }
    float m = -INFINITY;
    bool bad = false;
    if (tok) {
      for (int e = sub; e < E; e += TPT) {
        float v = rowp[e];
        if (!isfinite(v)) {
          bad = true;
          v = -INFINITY;
          rowp[e] = v;
        }
        m = fmaxf(m, v);
        // local sorted list; experts arrive in increasing index, so an equal logit ranks
        // after the ones already held. Once placed, the rest shift down one slot.
        if (ranks_before(v, e, top[K - 1], id[K - 1])) {
          float cv = v;
          int ci = e;
          bool placed = false;
#pragma unroll
          for (int j = 0; j < K; ++j) {
            if (placed || ranks_before(cv, ci, top[j], id[j])) {
              const float tv = top[j];
              const int ti = id[j];
              top[j] = cv;
              id[j] = ci;
              cv = tv;
              ci = ti;
              placed = true;
            }
          }
        }
      }
      if (bad) atomicOr(a.status, kStatusNonfinite);
    }
    // merge the TPT local lists: K rounds of a TPT-lane arg-best, the owner pops its head
    float bestv[K];
    int besti[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
      float bv = top[0];
      int bi = id[0];
#pragma unroll
      for (int off = TPT >> 1; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(tmask, bv, off, TPT);
        const int oi = __shfl_xor_sync(tmask, bi, off, TPT);
        if (ranks_before(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      bestv[j] = bv;
      besti[j] = bi;
      if (id[0] == bi) {
#pragma unroll
        for (int q = 0; q + 1 < K; ++q) {
          top[q] = top[q + 1];
          id[q] = id[q + 1];
        }
        top[K - 1] = -INFINITY;
        id[K - 1] = 0x7fffffff;
      }
    }
#pragma unroll
    for (int off = TPT >> 1; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(tmask, m, off, TPT));
    if (m == -INFINITY) m = 0.f;  // only when every logit was non-finite (already flagged)
    // sum of exp(l - m); each exp(l - m) replaces its logit in the row (the probability
    // sums below reuse it; the top-k logits are held in registers)
    float s = 0.f;
    if (tok)
      for (int e = sub; e < E; e += TPT) {
        const float v = expf(rowp[e] - m);
        rowp[e] = v;
        s += v;
      }
#pragma unroll
    for (int off = TPT >> 1; off > 0; off >>= 1) s += __shfl_xor_sync(tmask, s, off, TPT);

    if (tok && sub == 0) {
      const int t = t0 + i;
      s_inv[i] = s > 0.f ? 1.f / s : 0.f;
      const float lse = m + logf(s);
      zacc = lse * lse;
      // an id can only stay out of range when every logit was non-finite (flagged)
#pragma unroll
      for (int j = 0; j < K; ++j)
        if (besti[j] < 0 || besti[j] >= E) besti[j] = j;
      // gates: softmax over the K selected logits
      float gw[K], gsum = 0.f;
#pragma unroll
      for (int j = 0; j < K; ++j) {
        gw[j] = (bestv[0] > -INFINITY) ? expf(bestv[j] - bestv[0]) : (j == 0 ? 1.f : 0.f);
        gsum += gw[j];
      }
      unsigned cand = 0xffu;
      if (K == 2 && a.rr && !rr_keep(bestv[0], bestv[1], u_tok)) cand &= ~2u;
      s_cand[i] = uint8_t(cand);
      const float ginv = 1.f / gsum;
#pragma unroll
      for (int j = 0; j < K; ++j) {
        a.expert_id[size_t(t) * K + j] = besti[j];
        a.gate[size_t(t) * K + j] = gw[j] * ginv;
        s_id[i * kMaxK + j] = uint8_t(besti[j]);
        atomicAdd(&s_route[besti[j]], 1);
      }
    }
  }
  for (int off = 16; off > 0; off >>= 1) zacc += __shfl_xor_sync(0xffffffffu, zacc, off);
  if (lane == 0) s_z[warp] = zacc;
  __syncthreads();

  // per-expert softmax-probability sums over the chunk: tpe threads per expert, each a
  // strided subset of tokens, partials added in a fixed order
  {
    int tpe = kT / E;
    if (tpe < 1) tpe = 1;
    for (int base = 0; base < E * tpe; base += kT) {
      const int x = base + tid;
      const int e = x / tpe, sb = x % tpe;
      float acc = 0.f;
      if (e < E)
        for (int t = sb; t < nt; t += tpe) acc += s_log[t * ld + e] * s_inv[t];
      s_pp[tid] = acc;
      __syncthreads();
      if (e < E && sb == 0) {
        float sum = 0.f;
        for (int q = 0; q < tpe; ++q) sum += s_pp[tid + q];
        a.ppart[size_t(c) * E + e] = sum;
        a.hroute[size_t(c) * E + e] = s_route[e];
      }
      __syncthreads();
    }
  }
  if (tid == 0) {
    float sz = 0.f;
    for (int w = 0; w < kT / 32; ++w) sz += s_z[w];
    a.zpart[c] = sz;
  }

  // rank of each candidate among the chunk's earlier candidates of the same (j, e); the
  // first kThreads threads hold one token each
  const bool valid = tid < nt;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int j = 0; j < K; ++j) {
    for (int x = tid; x < kWarps * E; x += kT) s_wc[x / E][x % E] = 0;
    __syncthreads();
    int e = -1, rk = 0;
    if (tid < kThreads) {
      const bool cnd = valid && ((s_cand[tid] >> j) & 1u);
      e = cnd ? int(s_id[tid * kMaxK + j]) : -1;
      const int key = cnd ? e : (1024 + lane);
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      rk = __popc(peers & lt_mask);
      if (cnd && rk == 0) s_wc[warp][e] = __popc(peers);
    }
    __syncthreads();
    for (int e2 = tid; e2 < E; e2 += kT) {
      int run = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const int v = s_wc[w][e2];
        s_wc[w][e2] = run;
        run += v;
      }
      a.hist[(size_t(c) * K + j) * E + e2] = run;
    }
    __syncthreads();
    if (valid) a.rank[size_t(t0 + tid) * K + j] = e >= 0 ? s_wc[warp][e] + rk : -1;
    __syncthreads();
  }
}

// One CTA per chunk: stage the chunk's logits (contiguous rows t0..t0+nt-1, coalesced) into
// padded shared memory, then topk_chunk.
template <int K, int TPT>
__global__ void __launch_bounds__(kThreads * TPT) route_topk_kernel(RouteArgs a) {
  constexpr int kT = kThreads * TPT;
  extern __shared__ float s_log[];  // [kThreads][E + TPT] (padded: conflict-free lanes)
  const int c = blockIdx.x;
  const int g = c / a.n_cpg, cc = c % a.n_cpg;
  const int t0 = g * a.Sg + cc * kThreads;
  const int nt = min(kThreads, a.Sg - cc * kThreads);
  const int tid = threadIdx.x;
  const int E = a.E, ld = E + TPT;
  pdl_wait();
  pdl_trigger();
  const float u_tok = token_u<K, TPT>(a, t0, nt);
  const float* __restrict__ src = a.logits + size_t(t0) * E;
  const int n = nt * E;
  if ((E & 3) == 0 && (ld & 3) == 0) {
    const float4* __restrict__ src4 = reinterpret_cast<const float4*>(src);
#pragma unroll 4
    for (int q = tid; q < n / 4; q += kT) {
      const int idx = q * 4, r = idx / E, col = idx - r * E;
      *reinterpret_cast<float4*>(s_log + r * ld + col) = __ldg(src4 + q);
    }
  } else {
#pragma unroll 4
    for (int q = tid; q < n; q += kT) {
      const int r = q / E;
      s_log[r * ld + (q - r * E)] = __ldg(src + q);
    }
  }
  topk_chunk<K, TPT>(a, s_log, c, t0, nt, u_tok);  // its first barrier orders the staging
}

// ------------------------------------------------------------------ fused router + top-k
// The router projection and route_topk_kernel's work in one kernel (bf16 inputs). A CTA of
// kThreads * TPT threads takes one chunk: warp 0 streams the chunk's 128 rows of x and all
// of W_g through a ring of shared-memory stages with TMA, warp 1 accumulates the 128 x E
// logits tile with tcgen05.mma in tensor memory (fp32), warps 4..7 read it back (warp w
// reads TMEM lanes 32 (w % 4) ..) and add the bias into padded shared memory laid out as
// route_topk_kernel stages it (over the drained stage ring), optionally storing the logits
// to memory too; then the whole CTA runs topk_chunk. The logits never round-trip through
// HBM. The MMA sequence (64-wide k-blocks in order, four K = 16 steps each) and the bias
// addition are those of the router GEMM, so the logits equal moe_router's bit for bit.
// Lec16 Systems for MoE Models, "MoE Kernel 优化": the gating function as one fused kernel
// instead of one per step.
struct FusedRouterArgs {
  const float* bias;   // per-expert logit offset, nullable
  float* logits_out;   // [S, E] fp32, nullable
  int Mdim;            // contraction length (the model dimension)
  int BN;              // MMA N = smallest of 16, 32, .., 256 that is >= E
  int stages;
};

template <int K, int TPT>
__global__ void __launch_bounds__(kThreads * TPT, 1)
    router_topk_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                       RouteArgs a, FusedRouterArgs f) {
  using namespace sm100;
  static_assert(kThreads * TPT >= 256, "roles need warps 0, 1 and 4..7");
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[2 * 8 + 1];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int BN = f.BN, NS = f.stages;
  const int A_BYTES = 128 * 64 * 2, B_BYTES = BN * 64 * 2;
  uint8_t* sA = smem;
  uint8_t* sB = smem + NS * A_BYTES;
  float* s_log = reinterpret_cast<float*>(smem);  // reuses the ring once the MMAs are done
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * 8, done_bar = empty0 + 8 * 8;
  const int tcols = BN < 32 ? 32 : BN;

  const int c = blockIdx.x;
  const int g = c / a.n_cpg, cc = c % a.n_cpg;
  const int t0 = g * a.Sg + cc * kThreads;
  const int nt = min(kThreads, a.Sg - cc * kThreads);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E, ld = E + TPT;
  const int kblocks = f.Mdim / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(done_bar, 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_map(&tmX);
    tma_prefetch_map(&tmW);
  }
  if (warp == 1) tmem_alloc(smem_u32(&s_tmem), tcols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_wait();
  pdl_trigger();
  const float u_tok = token_u<K, TPT>(a, t0, nt);

  if (warp == 0) {
    // ---------------- TMA producer
    int stage = 0;
    uint32_t phase = 0, issued = 0, issued_par = 0;
    bool ok = true;
    for (int j = 0; j < kblocks; ++j) {
      ok = __all_sync(0xffffffffu, wait_bounded(empty0 + 8 * stage, phase ^ 1u, &s_abort, a.status));
      if (!ok) break;
      if (lane == 0) {
        const int kb = j;
        const uint32_t fb = full0 + 8 * stage;
        mbar_expect_tx(fb, A_BYTES + B_BYTES);
        tma_load_2d(smem_u32(sA + stage * A_BYTES), &tmX, kb * 64, t0, fb);
        tma_load_2d(smem_u32(sB + stage * B_BYTES), &tmW, kb * 64, 0, fb);
      }
      __syncwarp();
      issued |= 1u << stage;
      issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
      if (++stage == NS) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok && lane == 0)
      for (int s = 0; s < NS; ++s)
        if ((issued >> s) & 1u) wait_drain(full0 + 8 * s, (issued_par >> s) & 1u);
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer: one 128 x BN tile
    const uint32_t idesc = idesc_bf16(128, BN);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true, any = false;
    for (int j = 0; j < kblocks; ++j) {
      ok = __all_sync(0xffffffffu, wait_bounded(full0 + 8 * stage, phase, &s_abort, a.status));
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t a0 = smem_u32(sA + stage * A_BYTES), b0 = smem_u32(sB + stage * B_BYTES);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(tmem, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32), idesc,
                   (j | kk) != 0 ? 1u : 0u);
        mma_commit(empty0 + 8 * stage);
      }
      __syncwarp();
      any = true;
      if (++stage == NS) {
        stage = 0;
        phase ^= 1u;
      }
    }
    // done_bar completes once every MMA issued has finished (also after an abort, so that
    // shared and tensor memory are reused or freed only once nothing writes them)
    if (lane == 0 && any) mma_commit(done_bar);
    if (!ok && any && lane == 0) wait_drain(done_bar, 0u);
    __syncwarp();
  } else if (warp >= 4 && warp < 8) {
    // ---------------- drain: token i = 32 q + lane owns TMEM lane i
    const int q = warp & 3, i = q * 32 + lane;
    const uint32_t trow = tmem + (uint32_t(q * 32) << 16);
    const bool ok = __all_sync(0xffffffffu, wait_bounded(done_bar, 0u, &s_abort, a.status));
    if (ok) {
      tc_fence_after();
      const bool store = f.logits_out != nullptr && i < nt;
      float* dst = store ? f.logits_out + size_t(t0 + i) * E : nullptr;
      float* row = s_log + i * ld;
      for (int c0 = 0; c0 < BN; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(trow + c0, v);
        tmem_ld_wait();
        float l[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj)
          l[jj] = __uint_as_float(v[jj]) + ((f.bias && c0 + jj < E) ? f.bias[c0 + jj] : 0.f);
        if ((ld & 3) == 0 && c0 + 16 <= E) {  // 16-byte stores (rows are 16-byte aligned)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)
            reinterpret_cast<float4*>(row + c0)[jj] =
                make_float4(l[4 * jj], l[4 * jj + 1], l[4 * jj + 2], l[4 * jj + 3]);
        } else {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            if (c0 + jj < E) row[c0 + jj] = l[jj];
        }
        if (store) {
          if ((E & 3) == 0 && c0 + 16 <= E) {
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
              reinterpret_cast<float4*>(dst + c0)[jj] =
                  make_float4(l[4 * jj], l[4 * jj + 1], l[4 * jj + 2], l[4 * jj + 3]);
          } else {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj)
              if (c0 + jj < E) dst[c0 + jj] = l[jj];
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
  }
  // after a timeout (flagged in the status word) the routing below runs, in bounds, on
  // whatever the buffer holds rather than leaving its outputs unset
  topk_chunk<K, TPT>(a, s_log, c, t0, nt, u_tok);
}

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
  float ga = 0.f, gzs = 0.f;
  for (int gg = tid; gg < G; gg += kScanThreads) {
    float tsum = 0.f;
    for (int xx = 0; xx < X; ++xx) tsum += __ldcg(a.gaux + size_t(gg) * X + xx);
    ga += float(double(tsum) * double(E) / (double(a.Sg) * a.k * double(a.Sg)));
    gzs += __ldcg(a.gz + gg);
  }
  ga = block_sum(ga, s_red);
  gzs = block_sum(gzs, s_red);
  if (tid == 0) {
    *a.aux = ga / float(G);
    *a.z = gzs / float(a.S);
    *a.done = 0u;
  }
}

__global__ void __launch_bounds__(256) route_finalize_kernel(RouteArgs a) {
  pdl_wait();
  pdl_trigger();
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

template <int K, int TPT>
int launch_topk_t(const RouteArgs& a, int n_chunks, cudaStream_t st) {
  const size_t smem = size_t(kThreads) * (a.E + TPT) * sizeof(float);
  MOE_CUDA_CHECK(cudaFuncSetAttribute(route_topk_kernel<K, TPT>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
  return launch_kernel(route_topk_kernel<K, TPT>, dim3(n_chunks), dim3(kThreads * TPT), smem, st, a);
}

// threads per token: enough lanes that each holds at most 16 experts
template <int K>
int launch_topk(const RouteArgs& a, int n_chunks, cudaStream_t st) {
  if (a.E <= 16) return launch_topk_t<K, 1>(a, n_chunks, st);
  if (a.E <= 32) return launch_topk_t<K, 2>(a, n_chunks, st);
  if (a.E <= 64) return launch_topk_t<K, 4>(a, n_chunks, st);
  return launch_topk_t<K, 8>(a, n_chunks, st);
}

template <int K, int TPT>
int launch_router_topk_t(const CUtensorMap& tx, const CUtensorMap& tw, const RouteArgs& a,
                         FusedRouterArgs f, int n_chunks, cudaStream_t st) {
  // ring of (x, W_g) stages: with more chunks than SMs and <= 512 threads a CTA, two CTAs
  // share an SM (about 96 KB each), else one CTA takes about 192 KB
  const int stage_bytes = 128 * 64 * 2 + f.BN * 64 * 2;
  const bool two = n_chunks > num_sms() && kThreads * TPT <= 512;
  int stages = (two ? 96 * 1024 : 192 * 1024) / stage_bytes;
  stages = stages < 2 ? 2 : (stages > 8 ? 8 : stages);
  if (stages > f.Mdim / 64) stages = f.Mdim / 64;
  f.stages = stages;
  const size_t ring = size_t(f.stages) * stage_bytes;
  const size_t stage_log = size_t(kThreads) * (a.E + TPT) * sizeof(float);
  const size_t smem = (ring > stage_log ? ring : stage_log) + 1024;
  MOE_CUDA_CHECK(cudaFuncSetAttribute(router_topk_kernel<K, TPT>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
  return launch_kernel(router_topk_kernel<K, TPT>, dim3(n_chunks), dim3(kThreads * TPT), smem, st,
                       tx, tw, a, f);
}

// as launch_topk, with at least two threads per token (the roles need eight warps)
template <int K>
int launch_router_topk(const CUtensorMap& tx, const CUtensorMap& tw, const RouteArgs& a,
                       const FusedRouterArgs& f, int n_chunks, cudaStream_t st) {
  if (a.E <= 32) return launch_router_topk_t<K, 2>(tx, tw, a, f, n_chunks, st);
  if (a.E <= 64) return launch_router_topk_t<K, 4>(tx, tw, a, f, n_chunks, st);
  return launch_router_topk_t<K, 8>(tx, tw, a, f, n_chunks, st);
}

RouteArgs route_args(const moe_config_t& c, int C, const float* logits, const float* u,
                     const moe_route_out_t& out, char* ws, const WsLayout& L) {
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
  return a;
}

// the two launches after the per-chunk kernel
int launch_scan_finalize(const moe_config_t& c, const RouteArgs& a, cudaStream_t st) {
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
  const int64_t n = int64_t(c.S) * c.k;
  return launch_kernel(route_finalize_kernel, dim3(unsigned((n + 255) / 256)), dim3(256), 0, st, a);
}

}  // namespace

int launch_route(const moe_config_t& c, int C, const float* logits, const float* u,
                 const moe_route_out_t& out, char* ws, const WsLayout& L, cudaStream_t st) {
  if (reinterpret_cast<uintptr_t>(logits) % 16 != 0) return MOE_ERR_INVALID_ARG;
  const RouteArgs a = route_args(c, C, logits, u, out, ws, L);
  int rc;
  switch (c.k) {
    case 1: rc = launch_topk<1>(a, L.n_chunks, st); break;
    case 2: rc = launch_topk<2>(a, L.n_chunks, st); break;
    case 3: rc = launch_topk<3>(a, L.n_chunks, st); break;
    case 4: rc = launch_topk<4>(a, L.n_chunks, st); break;
    case 5: rc = launch_topk<5>(a, L.n_chunks, st); break;
    case 6: rc = launch_topk<6>(a, L.n_chunks, st); break;
    case 7: rc = launch_topk<7>(a, L.n_chunks, st); break;
    default: rc = launch_topk<8>(a, L.n_chunks, st); break;
  }
  if (rc != MOE_OK) return rc;
  return launch_scan_finalize(c, a, st);
}

int launch_router_route(const moe_config_t& c, int C, const void* x, const void* W_g,
                        const float* bias, const float* u, float* logits_out,
                        const moe_route_out_t& out, char* ws, const WsLayout& L, cudaStream_t st) {
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
  switch (c.k) {
    case 1: rc = launch_router_topk<1>(tx, tw, a, f, L.n_chunks, st); break;
    case 2: rc = launch_router_topk<2>(tx, tw, a, f, L.n_chunks, st); break;
    case 3: rc = launch_router_topk<3>(tx, tw, a, f, L.n_chunks, st); break;
    case 4: rc = launch_router_topk<4>(tx, tw, a, f, L.n_chunks, st); break;
    case 5: rc = launch_router_topk<5>(tx, tw, a, f, L.n_chunks, st); break;
    case 6: rc = launch_router_topk<6>(tx, tw, a, f, L.n_chunks, st); break;
    case 7: rc = launch_router_topk<7>(tx, tw, a, f, L.n_chunks, st); break;
    default: rc = launch_router_topk<8>(tx, tw, a, f, L.n_chunks, st); break;
  }
  if (rc != MOE_OK) return rc;
  return launch_scan_finalize(c, a, st);
}

}  // namespace moe
