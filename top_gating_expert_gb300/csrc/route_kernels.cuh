// The per-chunk routing kernels, shared by four translation units that each instantiate one
// of them: route_topk_kernel (routing from logits in memory) and router_topk_kernel (router
// projection fused with the routing), each for the default routing (VAR = false) and for
// the routing variants of moe_config_t (VAR = true: group-limited top-k, gate
// normalisations, uniform assignment), so that the default path carries none of the
// variants' code. route.cu holds the scan and finalize kernels and the launch order.
//
// GShard summary page, "Top-2 gating" (Random routing; Local group dispatching); Lec16
// Systems for MoE Models, "Switch Transformer" (gates = Softmax(KeepTopK(logits))),
// "DeepSeek V3 MoE" (expert groups, TopK(Softmax)), "MoE Kernel 优化" (softmax, top-k and
// the token-to-expert table fused); MegaBlocks router chapter §2 (p-norm gates, uniform
// assignment), §3 (load-balancing loss).
#pragma once
#include <cuda.h>
#include <float.h>
#include <math.h>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace moe {

constexpr int kThreads = kRouteChunk;  // one token per thread
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
  float* gaux;      // [G][X]: aux-loss term of each expert slice of each group
  float* gz;        // [G]
  // routing variants (moe_config_t)
  int gate_norm;    // MOE_GATE_*
  float gate_p;
  int ng, tg, gsz;  // expert groups (ng > 1: group-limited), groups kept, experts a group
  int uniform;      // ids replaced by (t*k + j) mod E
};

// Arguments of the fused router kernel beyond RouteArgs.
struct FusedRouterArgs {
  const float* bias;   // per-expert logit offset, nullable
  float* logits_out;   // [S, E] fp32, nullable
  int Mdim;            // contraction length (the model dimension)
  int BN;              // MMA N = smallest of 16, 32, .., 256 that is >= E
  int stages;
};

// entry points of the four kernel translation units (route_topk*.cu, route_fused*.cu)
int launch_topk_chunks(const RouteArgs& a, int n_chunks, cudaStream_t st);
int launch_topk_chunks_variants(const RouteArgs& a, int n_chunks, cudaStream_t st);
int launch_router_chunks(const CUtensorMap& tx, const CUtensorMap& tw, const RouteArgs& a,
                         const FusedRouterArgs& f, int n_chunks, cudaStream_t st);
int launch_router_chunks_variants(const CUtensorMap& tx, const CUtensorMap& tw, const RouteArgs& a,
                                  const FusedRouterArgs& f, int n_chunks, cudaStream_t st);

namespace {


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

// Group-limited routing (one call per token lane, all TPT lanes of a token together): the
// token's best logit in each of the ng contiguous expert groups of gsz (non-finite logits
// count as -inf), then the bit mask of the tg groups ranked first, ties to the lower
// group. Lane sub takes groups sub, sub + TPT, ... (it reads a group's logits from a
// rotated start, so the lanes of a warp fall on different banks), ranks each of them
// against the ng maxima broadcast one by one, and the lanes' bits are OR-ed together.
template <int TPT>
__device__ __forceinline__ unsigned group_mask(const float* rowp, bool tok, int sub, unsigned tmask,
                                            int ng, int tg, int gsz) {
  constexpr int kSlots = (16 + TPT - 1) / TPT;  // ng <= 16
  float gs[kSlots];
  int before[kSlots];
  const int rot = sub % gsz;
#pragma unroll
  for (int s = 0; s < kSlots; ++s) {
    const int g = sub + s * TPT;
    float lm = -INFINITY;
    if (tok && g < ng) {
      const float* gp = rowp + g * gsz;
      int r = rot;
      for (int q = 0; q < gsz; ++q) {
        const float v = gp[r];
        if (isfinite(v)) lm = fmaxf(lm, v);
        r = r + 1 == gsz ? 0 : r + 1;
      }
    }
    gs[s] = lm;
    before[s] = 0;
  }
  for (int h = 0; h < ng; ++h) {  // group h's maximum sits in lane h % TPT, slot h / TPT
    const int hs = h / TPT;
    float mine = gs[0];
#pragma unroll
    for (int s = 1; s < kSlots; ++s)
      if (s == hs) mine = gs[s];
    const float vh = __shfl_sync(tmask, mine, h % TPT, TPT);
#pragma unroll
    for (int s = 0; s < kSlots; ++s)
      if (vh > gs[s] || (vh == gs[s] && h < sub + s * TPT)) ++before[s];
  }
  unsigned mask = 0u;
#pragma unroll
  for (int s = 0; s < kSlots; ++s) {
    const int g = sub + s * TPT;
    if (g < ng && before[s] < tg) mask |= 1u << g;
  }
#pragma unroll
  for (int off = TPT >> 1; off > 0; off >>= 1) mask |= __shfl_xor_sync(tmask, mask, off, TPT);
  return mask;
}

// Gate normalisation of a token's K selected logits (best first, top = best[0]):
// MOE_GATE_NONE: exp(l_j - m) / s, the full-softmax probabilities (inv = 1/s);
// MOE_GATE_PNORM: exp(l_j - l_1) over the p-norm of those (the norm is scale-free).
template <int K>
__device__ __forceinline__ void variant_gates(const float* best, float m, float inv, int norm, float p,
                                           float* g) {
  if (norm == MOE_GATE_NONE) {
    for (int j = 0; j < K; ++j) g[j] = expf(best[j] - m) * inv;
    return;
  }
  float w[K], sp = 0.f;
  for (int j = 0; j < K; ++j) {
    w[j] = (best[0] > -INFINITY) ? expf(best[j] - best[0]) : (j == 0 ? 1.f : 0.f);
    sp += powf(w[j], p);
  }
  const float ginv = 1.f / powf(sp, 1.f / p);
  for (int j = 0; j < K; ++j) g[j] = w[j] * ginv;
}

// The random-routing draw of this thread's token when it is the token's first lane (read
// early, so that its latency hides behind the staging of the logits).
template <int K, int TPT>
__device__ __forceinline__ float token_u(const RouteArgs& a, int t0, int nt) {
  const int i = int(threadIdx.x) / TPT;
  return (K == 2 && a.rr && int(threadIdx.x) % TPT == 0 && i < nt) ? __ldg(a.u + t0 + i) : 0.f;
}

// The barrier of the routing body: the whole CTA (NB = 0), or named barrier 1 over the
// first NB threads when the CTA also runs warps of other roles.
template <int NB>
__device__ __forceinline__ void body_sync() {
  if constexpr (NB == 0) __syncthreads();
  else asm volatile("bar.sync 1, %0;" ::"n"(NB) : "memory");
}

// The per-chunk routing work on a chunk's logits staged in shared memory (s_log: nt rows of
// E logits, row stride ld = E + TPT). TPT threads per token (consecutive lanes), each owning
// experts sub, sub + TPT, ...; the CTA has kThreads * TPT threads, all of which call this.
// Non-finite logits count as -inf (and are flagged); each staged logit is overwritten by
// exp(logit - max of its token). NB: see body_sync (the body threads are 0 .. NB - 1).
template <int K, int TPT, bool VAR, int NB = 0>
__device__ __forceinline__ void topk_chunk(const RouteArgs& a, float* s_log, int c, int t0, int nt,
                                           float u_tok) {
  constexpr int kT = kThreads * TPT;
  __shared__ float s_inv[kThreads], s_pp[kT];
  __shared__ uint8_t s_id[kThreads * kMaxK];
  __shared__ uint8_t s_cand[kThreads];
  __shared__ uint8_t s_rk[kThreads * kMaxK];  // rank within the warp of each candidate
  __shared__ int s_route[kMaxE];
  __shared__ float s_z[kT / 32];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, ld = E + TPT;
  // The persistent router's body (NB != 0) with k <= 3 and at most 16 experts a lane (TPT
  // 2 or 4): the lane's logits stay in registers through the selection, the exponentials
  // and the sum, and the row then receives the probabilities themselves. (With one chunk a
  // CTA, where the body does not overlap the loads, that form measured slower: 63 -> 76 us
  // for the routing of 65536 tokens over 64 experts.)
  constexpr bool kRegs = NB != 0 && K < 4 && TPT <= 4;
  constexpr int NPL = kRegs ? 16 : 1;
  if (c == 0 && tid == 0) *a.done = 0u;  // ticket counter of route_scan_kernel
  for (int e = tid; e < E; e += kT) s_route[e] = 0;
  body_sync<NB>();

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
    // group-limited routing: the groups this token may take experts from
    const unsigned gmask = (VAR && a.ng > 1) ? group_mask<TPT>(rowp, tok, sub, tmask, a.ng, a.tg, a.gsz)
                                             : 0xffffffffu;
    // an expert's group e / gsz as (e * gm24) >> 24 with gm24 = ceil(2^24 / gsz): exact for
    // e, gsz <= 256 (the error term e * (gm24 * gsz - 2^24) stays below 2^24); 0 (group 0,
    // whose bit is set) when the routing is not group-limited
    const unsigned gm24 = (VAR && a.ng > 1) ? ((1u << 24) + unsigned(a.gsz) - 1u) / unsigned(a.gsz) : 0u;
    float m = -INFINITY;
    bool bad = false;
    // may this token select expert e (group-limited routing)
    auto selectable = [&](int e) { return !VAR || ((gmask >> ((unsigned(e) * gm24) >> 24)) & 1u); };
    // local sorted list; experts arrive in increasing index, so an equal logit ranks after
    // the ones already held. Once placed, the rest shift down one slot.
    auto insert = [&](float v, int e) {
      if (!ranks_before(v, e, top[K - 1], id[K - 1])) return;
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
    };
    float lreg[NPL];
    if constexpr (K >= 4) {
      // pass 1: the token's maximum (non-finite logits flagged and set to -inf) and this
      // lane's RL = ceil(K / TPT) largest selectable logits
      constexpr int RL = (K + TPT - 1) / TPT;
      float lv[RL];
#pragma unroll
      for (int j = 0; j < RL; ++j) lv[j] = -INFINITY;
      if (tok) {
        for (int e = sub; e < E; e += TPT) {
          float v = rowp[e];
          if (!isfinite(v)) {
            bad = true;
            v = -INFINITY;
            rowp[e] = v;
          }
          m = fmaxf(m, v);
          if (selectable(e) && v > lv[RL - 1]) {
#pragma unroll
            for (int j = RL - 1; j > 0; --j) lv[j] = v > lv[j - 1] ? lv[j - 1] : (v > lv[j] ? v : lv[j]);
            lv[0] = fmaxf(lv[0], v);
          }
        }
        if (bad) atomicOr(a.status, kStatusNonfinite);
      }
      // every lane holds RL selectable logits >= its lv[RL - 1], RL * TPT >= K of them in
      // all, so the token's K-th largest selectable logit is at least the smallest of the
      // lanes' lv[RL - 1], tau: no logit below tau is selected
      float tau = lv[RL - 1];
#pragma unroll
      for (int off = TPT >> 1; off > 0; off >>= 1) tau = fminf(tau, __shfl_xor_sync(tmask, tau, off, TPT));
      // pass 2: the lane's selectable logits >= tau as a bit mask (bit q: expert sub + q TPT;
      // E / TPT <= 32 for every TPT the launch picks), inserted in increasing expert index
      // -- a few per lane instead of all
      unsigned cmask = 0u;
      if (tok) {
        int q = 0;
        for (int e = sub; e < E; e += TPT, ++q)
          if (selectable(e) && rowp[e] >= tau) cmask |= 1u << q;
      }
      while (cmask) {
        const int q = __ffs(cmask) - 1;
        cmask &= cmask - 1u;
        const int e = sub + q * TPT;
        insert(rowp[e], e);
      }
    } else if constexpr (kRegs) {
      // the lane's experts arrive in increasing index, so a held logit equal to v already
      // ranks first and a strict comparison keeps the order: the insertion is a fixed
      // sequence of selects (a branch per element diverged across the warp's lanes)
#pragma unroll
      for (int q = 0; q < NPL; ++q) {
        if (q * TPT >= E) break;  // no lane of the warp has an expert left
        const int e = sub + q * TPT;
        const bool own = tok && e < E;
        float v = own ? rowp[e] : -INFINITY;
        const bool fin = isfinite(v);
        bad |= own && !fin;
        v = fin ? v : -INFINITY;
        lreg[q] = v;
        m = fmaxf(m, v);
        if (own && selectable(e)) {
          // the new list, slot by slot from the old one: slot j takes the old slot j - 1
          // when v ranks above it, else v when v ranks above the old slot j (written into
          // temporaries: the same selects updating the list in place, from the last slot
          // down, gave lists holding one expert twice when built for the GPU, while the
          // host build of the same code was right)
          float nt[K];
          int ni[K];
#pragma unroll
          for (int j = 0; j < K; ++j) {
            const bool above = v > top[j];
            const bool above_prev = j > 0 && v > top[j > 0 ? j - 1 : 0];
            nt[j] = above_prev ? top[j > 0 ? j - 1 : 0] : (above ? v : top[j]);
            ni[j] = above_prev ? id[j > 0 ? j - 1 : 0] : (above ? e : id[j]);
          }
#pragma unroll
          for (int j = 0; j < K; ++j) {
            top[j] = nt[j];
            id[j] = ni[j];
          }
        }
      }
      if (tok && bad) atomicOr(a.status, kStatusNonfinite);
    } else {
      if (tok) {
        for (int e = sub; e < E; e += TPT) {
          float v = rowp[e];
          if (!isfinite(v)) {
            bad = true;
            v = -INFINITY;
            rowp[e] = v;
          }
          m = fmaxf(m, v);
          if (selectable(e)) insert(v, e);
        }
        if (bad) atomicOr(a.status, kStatusNonfinite);
      }
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
    // sums below reuse it; the top-k logits are held in registers). In the register form
    // the default routing takes the fast exponential here: these terms feed only the
    // softmax sum (the z-loss's logsumexp) and the probabilities of the aux loss, each
    // term within a few ulp (the gates are computed apart, with expf); the variants keep
    // expf, as their un-normalised gates are these probabilities.
    float s = 0.f;
    if constexpr (kRegs) {
#pragma unroll
      for (int q = 0; q < NPL; ++q) {
        if (q * TPT >= E) break;
        const int e = sub + q * TPT;
        float v = 0.f;
        if (tok && e < E) v = VAR ? expf(lreg[q] - m) : __expf(lreg[q] - m);
        lreg[q] = v;
        s += v;
      }
    } else if (tok) {
      for (int e = sub; e < E; e += TPT) {
        const float v = expf(rowp[e] - m);
        rowp[e] = v;
        s += v;
      }
    }
#pragma unroll
    for (int off = TPT >> 1; off > 0; off >>= 1) s += __shfl_xor_sync(tmask, s, off, TPT);
    if constexpr (kRegs) {
      // the probabilities, the products the sums below would otherwise form
      const float inv = s > 0.f ? 1.f / s : 0.f;
#pragma unroll
      for (int q = 0; q < NPL; ++q) {
        if (q * TPT >= E) break;
        const int e = sub + q * TPT;
        if (tok && e < E) rowp[e] = lreg[q] * inv;
      }
    }

    if (tok && sub == 0) {
      const int t = t0 + i;
      s_inv[i] = s > 0.f ? 1.f / s : 0.f;
      const float lse = m + logf(s);
      zacc = lse * lse;
      // an id can only stay out of range when every logit was non-finite (flagged)
#pragma unroll
      for (int j = 0; j < K; ++j)
        if (besti[j] < 0 || besti[j] >= E) besti[j] = j;
      // gates: softmax over the K selected logits (MOE_GATE_SOFTMAX_TOPK); the full-softmax
      // probabilities (MOE_GATE_NONE); or those over their gate_p-norm (MOE_GATE_PNORM,
      // scale-free, so computed from exp(l_j - l_1))
      float gw[K], ginv = 1.f;
      if (!VAR || a.gate_norm == MOE_GATE_SOFTMAX_TOPK) {
        float gsum = 0.f;
#pragma unroll
        for (int j = 0; j < K; ++j) {
          gw[j] = (bestv[0] > -INFINITY) ? expf(bestv[j] - bestv[0]) : (j == 0 ? 1.f : 0.f);
          gsum += gw[j];
        }
        ginv = 1.f / gsum;
      } else {
        variant_gates<K>(bestv, m, s_inv[i], a.gate_norm, a.gate_p, gw);
      }
      unsigned cand = 0xffu;
      if (K == 2 && a.rr && !rr_keep(bestv[0], bestv[1], u_tok)) cand &= ~2u;
      s_cand[i] = uint8_t(cand);
      if (VAR && a.uniform) {  // benchmark assignment: the ids only change, not the gates
#pragma unroll
        for (int j = 0; j < K; ++j) besti[j] = int((int64_t(t) * K + j) % E);
      }
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
  body_sync<NB>();

  // per-expert softmax-probability sums over the chunk: tpe threads per expert, each a
  // strided subset of tokens, partials added in a fixed order
  {
    int tpe = kT / E;
    if (tpe < 1) tpe = 1;
    for (int base = 0; base < E * tpe; base += kT) {
      const int x = base + tid;
      const int e = x / tpe, sb = x % tpe;
      float acc = 0.f;
      if (e < E) {
        if constexpr (kRegs) {  // the row holds the probabilities
          for (int t = sb; t < nt; t += tpe) acc += s_log[t * ld + e];
        } else {
          for (int t = sb; t < nt; t += tpe) acc += s_log[t * ld + e] * s_inv[t];
        }
      }
      s_pp[tid] = acc;
      body_sync<NB>();
      if (e < E && sb == 0) {
        float sum = 0.f;
        for (int q = 0; q < tpe; ++q) sum += s_pp[tid + q];
        a.ppart[size_t(c) * E + e] = sum;
        a.hroute[size_t(c) * E + e] = s_route[e];
      }
      body_sync<NB>();
    }
  }
  if (tid == 0) {
    float sz = 0.f;
    for (int w = 0; w < kT / 32; ++w) sz += s_z[w];
    a.zpart[c] = sz;
  }

  // rank of each candidate among the chunk's earlier candidates of the same (j, e); the
  // first kThreads threads hold one token each. All K choice ranks at once: per (j, warp,
  // e) counts in shared memory (over the staged logits, which nothing reads any more), one
  // scan over the warps per (j, e), then each token's K ranks -- three barriers for any K.
  int* s_cnt = reinterpret_cast<int*>(s_log);  // [K][kWarps][E] (16 K E <= 512 (E + TPT) bytes)
  for (int x = tid; x < K * kWarps * E; x += kT) s_cnt[x] = 0;
  body_sync<NB>();
  const bool valid = tid < nt;
  const unsigned lt_mask = (1u << lane) - 1u;
  if (tid < kThreads) {
#pragma unroll
    for (int j = 0; j < K; ++j) {
      const bool cnd = valid && ((s_cand[tid] >> j) & 1u);
      const int e = cnd ? int(s_id[tid * kMaxK + j]) : -1;
      const int key = cnd ? e : (1024 + lane);
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      const int rk = __popc(peers & lt_mask);
      s_rk[tid * kMaxK + j] = uint8_t(rk);  // < 32
      if (cnd && rk == 0) s_cnt[(j * kWarps + warp) * E + e] = __popc(peers);
    }
  }
  body_sync<NB>();
  for (int x = tid; x < K * E; x += kT) {
    const int j = x / E, e2 = x - j * E;
    int run = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      int* cw = s_cnt + (j * kWarps + w) * E + e2;
      const int v = *cw;
      *cw = run;
      run += v;
    }
    a.hist[(size_t(c) * K + j) * E + e2] = run;
  }
  body_sync<NB>();
  if (valid) {
#pragma unroll
    for (int j = 0; j < K; ++j) {
      const bool cnd = (s_cand[tid] >> j) & 1u;
      const int e = int(s_id[tid * kMaxK + j]);
      a.rank[size_t(t0 + tid) * K + j] =
          cnd ? s_cnt[(j * kWarps + warp) * E + e] + int(s_rk[tid * kMaxK + j]) : -1;
    }
  }
}

// One CTA per chunk: stage the chunk's logits (contiguous rows t0..t0+nt-1, coalesced) into
// padded shared memory, then topk_chunk. With 8 lanes a token and k <= 3 two CTAs share an
// SM (32 registers a thread).
template <int K, int TPT, bool VAR>
__global__ void __launch_bounds__(kThreads * TPT, (TPT == 8 && K <= 3) ? 2 : 1) route_topk_kernel(RouteArgs a) {
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
  topk_chunk<K, TPT, VAR>(a, s_log, c, t0, nt, u_tok);  // its first barrier orders the staging
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
template <int K, int TPT, bool VAR>
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
  const uint64_t wlimit = wait_limit_ns(a.status);
  const float u_tok = token_u<K, TPT>(a, t0, nt);

  // what each role has in flight, for the drain after an abort (see the end of the roles)
  uint32_t issued = 0, issued_par = 0;
  bool mma_any = false, mma_waited = false;
  if (warp == 0) {
    // ---------------- TMA producer
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int j = 0; j < kblocks; ++j) {
      ok = __all_sync(0xffffffffu, wait_bounded(empty0 + 8 * stage, phase ^ 1u, &s_abort, a.status, wlimit));
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
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer: one 128 x BN tile
    const uint32_t idesc = idesc_bf16(128, BN);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int j = 0; j < kblocks; ++j) {
      ok = __all_sync(0xffffffffu, wait_bounded(full0 + 8 * stage, phase, &s_abort, a.status, wlimit));
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
      mma_any = true;
      if (++stage == NS) {
        stage = 0;
        phase ^= 1u;
      }
    }
    // done_bar completes once every MMA issued has finished (also after an abort, so that
    // shared and tensor memory are reused or freed only once nothing writes them)
    if (lane == 0 && mma_any) mma_commit(done_bar);
    if (!ok && mma_any && lane == 0) wait_drain(done_bar, 0u);
    mma_waited = !ok && mma_any;
    __syncwarp();
  } else if (warp >= 4 && warp < 8) {
    // ---------------- drain: token i = 32 q + lane owns TMEM lane i
    const int q = warp & 3, i = q * 32 + lane;
    const uint32_t trow = tmem + (uint32_t(q * 32) << 16);
    const bool ok = __all_sync(0xffffffffu, wait_bounded(done_bar, 0u, &s_abort, a.status, wlimit));
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
  if (s_abort) {
    // A role may have finished its own loop before another gave up, with loads or MMAs still
    // in flight: every load issued lands and every MMA issued finishes before the ring is
    // reused and tensor memory freed (the flag is read after the barrier: CTA-uniform).
    if (warp == 0 && lane == 0)
      for (int s = 0; s < NS; ++s)
        if ((issued >> s) & 1u) wait_drain(full0 + 8 * s, (issued_par >> s) & 1u);
    if (warp == 1 && lane == 0 && mma_any && !mma_waited) wait_drain(done_bar, 0u);
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
  }
  // after a timeout (flagged in the status word) the routing below runs, in bounds, on
  // whatever the buffer holds rather than leaving its outputs unset
  topk_chunk<K, TPT, VAR>(a, s_log, c, t0, nt, u_tok);
}

// ------------------------------------------------------------------ persistent fused router
// router_topk_kernel's work for layers with more chunks than SMs: one CTA per SM walks the
// chunks blockIdx.x, blockIdx.x + gridDim.x, ... Warps 0 .. kBody / 32 - 1 run the routing
// body, warp kBody / 32 streams the chunks' x rows and W_g through a TMA ring that does not
// drain between chunks, and warp kBody / 32 + 1 issues each chunk's MMAs into one of two
// TMEM accumulators. So the next chunk's loads and MMAs run while the body routes the
// current one; router_topk_kernel, one chunk a CTA, runs its body only after its own loads,
// in waves that leave DRAM idle meanwhile. The MMA sequence (64-wide k-blocks in order,
// four K = 16 steps each) and the bias addition are router_topk_kernel's, so the logits
// equal moe_router's bit for bit. Lec16 Systems for MoE Models, "MoE Kernel 优化": the
// gating function as one fused kernel.
template <int K, int TPT, bool VAR>
__global__ void __launch_bounds__(kThreads * TPT + 64, 1)
    router_topk_persistent_kernel(const __grid_constant__ CUtensorMap tmX,
                                  const __grid_constant__ CUtensorMap tmW, RouteArgs a,
                                  FusedRouterArgs f) {
  using namespace sm100;
  constexpr int kBody = kThreads * TPT;             // the routing body's threads
  constexpr int kPW = kBody / 32, kMW = kPW + 1;    // producer and MMA warps
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[2 * 8 + 5];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int BN = f.BN, NS = f.stages;
  const int A_BYTES = 128 * 64 * 2, B_BYTES = BN * 64 * 2;
  uint8_t* sA = smem;
  uint8_t* sB = smem + NS * A_BYTES;
  float* s_log = reinterpret_cast<float*>(sB + NS * B_BYTES);  // its own buffer
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * 8, tfull0 = empty0 + 8 * 8;
  const uint32_t tempty0 = tfull0 + 16, drain_bar = tempty0 + 16;
  const int tcols = 2 * BN < 32 ? 32 : 2 * BN;  // two accumulators (BN a power of 2)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E, ld = E + TPT;
  const int kblocks = f.Mdim / 64;
  const int n_chunks = a.G * a.n_cpg;
  const int nch = blockIdx.x < unsigned(n_chunks)
                      ? (n_chunks - int(blockIdx.x) + int(gridDim.x) - 1) / int(gridDim.x) : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(tfull0 + 8 * q, 1);
      mbar_init(tempty0 + 8 * q, 1);
    }
    mbar_init(drain_bar, 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_map(&tmX);
    tma_prefetch_map(&tmW);
  }
  if (warp == kMW) tmem_alloc(smem_u32(&s_tmem), tcols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_wait();
  pdl_trigger();
  const uint64_t wlimit = wait_limit_ns(a.status);

  // chunk i of this CTA: its group, first token and token count
  auto chunk = [&](int i, int& c, int& t0, int& nt) {
    c = int(blockIdx.x) + i * int(gridDim.x);
    const int g = c / a.n_cpg, cc = c % a.n_cpg;
    t0 = g * a.Sg + cc * kThreads;
    nt = min(kThreads, a.Sg - cc * kThreads);
  };
  // what each role has in flight, for the drain after an abort
  uint32_t issued = 0, issued_par = 0;
  bool mma_any = false, mma_drained = false;

  if (warp == kPW) {
    // ---------------- TMA producer: every k-block of every chunk, the ring never drains
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int i = 0; i < nch && ok; ++i) {
      int c, t0, nt;
      chunk(i, c, t0, nt);
      for (int kb = 0; kb < kblocks; ++kb) {
        ok = __all_sync(0xffffffffu, wait_bounded(empty0 + 8 * stage, phase ^ 1u, &s_abort, a.status, wlimit));
        if (!ok) break;
        if (lane == 0) {
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
    }
  } else if (warp == kMW) {
    // ---------------- MMA issuer: one 128 x BN tile a chunk, accumulators alternating
    const uint32_t idesc = idesc_bf16(128, BN);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int i = 0; i < nch && ok; ++i) {
      const int acc = i & 1;
      const uint32_t use = uint32_t(i >> 1) & 1u;
      ok = __all_sync(0xffffffffu, wait_bounded(tempty0 + 8 * acc, use ^ 1u, &s_abort, a.status, wlimit));
      if (!ok) break;
      tc_fence_after();
      const uint32_t d = tmem + uint32_t(acc * BN);
      for (int kb = 0; kb < kblocks; ++kb) {
        ok = __all_sync(0xffffffffu, wait_bounded(full0 + 8 * stage, phase, &s_abort, a.status, wlimit));
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a0 = smem_u32(sA + stage * A_BYTES), b0 = smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(d, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32), idesc,
                     (kb | kk) != 0 ? 1u : 0u);
          mma_commit(empty0 + 8 * stage);
        }
        __syncwarp();
        mma_any = true;
        if (++stage == NS) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok && lane == 0) mma_commit(tfull0 + 8 * acc);
      __syncwarp();
    }
    if (!ok && mma_any && lane == 0) {  // every MMA issued finishes before TMEM is freed
      mma_commit(drain_bar);
      wait_drain(drain_bar, 0u);
    }
    mma_drained = !ok && mma_any;
    __syncwarp();
  } else {
    // ---------------- the routing body, chunk after chunk
    // drain: warp w reads TMEM lanes 32 (w % 4) .. (its 32 tokens) and the 16-column blocks
    // part, part + TPT, ... of the accumulator (part = w / 4), adding the bias
    const int q = warp & 3, part = warp >> 2, r = q * 32 + lane;
    for (int i = 0; i < nch; ++i) {
      int c, t0, nt;
      chunk(i, c, t0, nt);
      const int acc = i & 1;
      const uint32_t use = uint32_t(i >> 1) & 1u;
      const float u_tok = token_u<K, TPT>(a, t0, nt);
      const bool ok = __all_sync(0xffffffffu, wait_bounded(tfull0 + 8 * acc, use, &s_abort, a.status, wlimit));
      if (ok) {  // after a timeout the body below runs, in bounds, on the stale buffer
        tc_fence_after();
        const uint32_t trow = tmem + (uint32_t(q * 32) << 16) + uint32_t(acc * BN);
        const bool store = f.logits_out != nullptr && r < nt;
        float* dst = store ? f.logits_out + size_t(t0 + r) * E : nullptr;
        float* row = s_log + r * ld;
        for (int c0 = part * 16; c0 < BN; c0 += TPT * 16) {
          uint32_t v[16];
          tmem_ld16(trow + c0, v);
          tmem_ld_wait();
          float l[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            l[jj] = __uint_as_float(v[jj]) + ((f.bias && c0 + jj < E) ? f.bias[c0 + jj] : 0.f);
          if ((ld & 3) == 0 && c0 + 16 <= E) {
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
      tc_fence_before();
      body_sync<kBody>();  // the chunk's logits are staged; its accumulator is free again
      if (threadIdx.x == 0 && ok) mbar_arrive(tempty0 + 8 * acc);
      topk_chunk<K, TPT, VAR, kBody>(a, s_log, c, t0, nt, u_tok);
      body_sync<kBody>();  // the body's last reads of s_log are done before the next drain
    }
  }
  tc_fence_before();
  __syncthreads();
  if (s_abort) {
    // as in the expert GEMM: whichever role gave up, every load issued lands and every MMA
    // issued finishes before shared and tensor memory are released
    if (warp == kPW && lane == 0)
      for (int s = 0; s < NS; ++s)
        if ((issued >> s) & 1u) wait_drain(full0 + 8 * s, (issued_par >> s) & 1u);
    if (warp == kMW && lane == 0 && mma_any && !mma_drained) {
      mma_commit(drain_bar);
      wait_drain(drain_bar, 0u);
    }
    tc_fence_before();
    __syncthreads();
  }
  if (warp == kMW) {
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
  }
}

template <bool VAR, int K, int TPT>
int launch_topk_t(const RouteArgs& a, int n_chunks, cudaStream_t st) {
  const size_t smem = size_t(kThreads) * (a.E + TPT) * sizeof(float);
  MOE_CUDA_CHECK(cudaFuncSetAttribute(route_topk_kernel<K, TPT, VAR>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
  return launch_kernel(route_topk_kernel<K, TPT, VAR>, dim3(n_chunks), dim3(kThreads * TPT), smem, st, a);
}

// threads per token: enough lanes that each holds at most 16 experts
template <bool VAR, int K>
int launch_topk(const RouteArgs& a, int n_chunks, cudaStream_t st) {
  if (a.E <= 16) return launch_topk_t<VAR, K, 1>(a, n_chunks, st);
  if (a.E <= 32) return launch_topk_t<VAR, K, 2>(a, n_chunks, st);
  if (a.E <= 64) return launch_topk_t<VAR, K, 4>(a, n_chunks, st);
  return launch_topk_t<VAR, K, 8>(a, n_chunks, st);
}

template <bool VAR, int K, int TPT>
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
  MOE_CUDA_CHECK(cudaFuncSetAttribute(router_topk_kernel<K, TPT, VAR>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
  return launch_kernel(router_topk_kernel<K, TPT, VAR>, dim3(n_chunks), dim3(kThreads * TPT), smem, st,
                       tx, tw, a, f);
}

// The persistent form: one CTA per SM (at most one per chunk), a ring of up to 8 stages in
// what shared memory the staged logits leave. Returns MOE_ERR_UNSUPPORTED when it does
// not fit, so that the caller falls back to router_topk_kernel.
template <bool VAR, int K, int TPT>
int launch_router_topk_persistent_t(const CUtensorMap& tx, const CUtensorMap& tw,
                                    const RouteArgs& a, FusedRouterArgs f, int n_chunks,
                                    cudaStream_t st) {
  auto kern = router_topk_persistent_kernel<K, TPT, VAR>;
  static const int64_t static_smem = [&] {
    cudaFuncAttributes fa;
    return cudaFuncGetAttributes(&fa, kern) == cudaSuccess ? int64_t(fa.sharedSizeBytes)
                                                           : int64_t(1) << 30;
  }();
  const int stage_bytes = 128 * 64 * 2 + f.BN * 64 * 2;
  const int64_t stage_log = int64_t(kThreads) * (a.E + TPT) * int64_t(sizeof(float));
  const int64_t budget = int64_t(227 * 1024) - static_smem - 1024 - stage_log;
  int stages = budget > 0 ? int(budget / stage_bytes) : 0;
  if (stages > 8) stages = 8;
  if (stages > f.Mdim / 64) stages = f.Mdim / 64;
  if (stages < 2) return MOE_ERR_UNSUPPORTED;
  f.stages = stages;
  const size_t smem = size_t(stages) * stage_bytes + stage_log + 1024;
  MOE_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
  int per_sm = 0;
  MOE_CUDA_CHECK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads * TPT + 64, smem));
  if (per_sm < 1) return MOE_ERR_UNSUPPORTED;
  const int grid = n_chunks < num_sms() ? n_chunks : num_sms();
  return launch_kernel(kern, dim3(grid), dim3(kThreads * TPT + 64), smem, st, tx, tw, a, f);
}

// as launch_topk, with at least two threads per token (the roles need eight warps); with
// more chunks than SMs and at most 64 experts (a body of at most 512 threads, beside which
// the persistent form's two role warps fit) the persistent form
template <bool VAR, int K>
int launch_router_topk(const CUtensorMap& tx, const CUtensorMap& tw, const RouteArgs& a,
                       const FusedRouterArgs& f, int n_chunks, cudaStream_t st) {
  if constexpr (!VAR) {
    if (n_chunks > num_sms() && a.E <= 64) {
      const int rc = a.E <= 32
                         ? launch_router_topk_persistent_t<VAR, K, 2>(tx, tw, a, f, n_chunks, st)
                         : launch_router_topk_persistent_t<VAR, K, 4>(tx, tw, a, f, n_chunks, st);
      if (rc != MOE_ERR_UNSUPPORTED) return rc;
    }
  }
  if (a.E <= 32) return launch_router_topk_t<VAR, K, 2>(tx, tw, a, f, n_chunks, st);
  if (a.E <= 64) return launch_router_topk_t<VAR, K, 4>(tx, tw, a, f, n_chunks, st);
  return launch_router_topk_t<VAR, K, 8>(tx, tw, a, f, n_chunks, st);
}

// one launch of the per-chunk kernel for any k (1..8)
template <bool VAR>
int launch_topk_any_k(const RouteArgs& a, int n_chunks, cudaStream_t st) {
  switch (a.k) {
    case 1: return launch_topk<VAR, 1>(a, n_chunks, st);
    case 2: return launch_topk<VAR, 2>(a, n_chunks, st);
    case 3: return launch_topk<VAR, 3>(a, n_chunks, st);
    case 4: return launch_topk<VAR, 4>(a, n_chunks, st);
    case 5: return launch_topk<VAR, 5>(a, n_chunks, st);
    case 6: return launch_topk<VAR, 6>(a, n_chunks, st);
    case 7: return launch_topk<VAR, 7>(a, n_chunks, st);
    default: return launch_topk<VAR, 8>(a, n_chunks, st);
  }
}

template <bool VAR>
int launch_router_topk_any_k(const CUtensorMap& tx, const CUtensorMap& tw, const RouteArgs& a,
                             const FusedRouterArgs& f, int n_chunks, cudaStream_t st) {
  switch (a.k) {
    case 1: return launch_router_topk<VAR, 1>(tx, tw, a, f, n_chunks, st);
    case 2: return launch_router_topk<VAR, 2>(tx, tw, a, f, n_chunks, st);
    case 3: return launch_router_topk<VAR, 3>(tx, tw, a, f, n_chunks, st);
    case 4: return launch_router_topk<VAR, 4>(tx, tw, a, f, n_chunks, st);
    case 5: return launch_router_topk<VAR, 5>(tx, tw, a, f, n_chunks, st);
    case 6: return launch_router_topk<VAR, 6>(tx, tw, a, f, n_chunks, st);
    case 7: return launch_router_topk<VAR, 7>(tx, tw, a, f, n_chunks, st);
    default: return launch_router_topk<VAR, 8>(tx, tw, a, f, n_chunks, st);
  }
}

}  // namespace
}  // namespace moe
