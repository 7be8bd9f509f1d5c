// The layer's backward pass: layout kernels for the weight gradients and the router's
// backward (the expert GEMMs of the backward run on the tcgen05 grouped GEMM).
//
// The loss is L = sum(dy * y) + aux_coef * aux + z_coef * z. MegaBlocks router chapter §3:
// the load-balancing loss is a differentiable proxy, its gradient reaching the router only
// through the expert scores (the counts are constants); §2: the z-loss mean(lse^2). Routing
// decisions are held fixed (piecewise constant in the logits). GShard summary page, "MoE
// Transformer": each expert a two-layer FFN; Lec16 Systems for MoE Models, "DeepSeek V3 MoE":
// SwiGLU experts.
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kPad = 64;  // K-block of the grouped GEMM: weight-gradient segments start on it

// poff[g] = sum over g' < g of the rows of g' rounded up to 64 (g = 0..groups); with
// offsets null, one group of dense_rows rows.
__global__ void pad_offsets_kernel(const int32_t* __restrict__ offsets, int groups, int dense_rows,
                                   int32_t* __restrict__ poff) {
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  int run = 0;
  poff[0] = 0;
  for (int g = 0; g < groups; ++g) {
    int n = offsets ? offsets[g + 1] - offsets[g] : dense_rows;
    if (n < 0) n = 0;
    run += (n + kPad - 1) / kPad * kPad;
    poff[g + 1] = run;
  }
}

// out [C][ld_out] (bf16): column p of group g's padded range is row i = p - poff[g] of the
// group (rows off[g] + i, or i when dense), zero for i past its rows; the value is
// scale[r] * in[src(r)][c] with src(r) = gather[r] (or r). A 64 (p) x 64 (c) tile per block:
// each warp reads 8 rows as 128-byte segments, packs row pairs into 32-bit words
// T[c][p / 2] (row stride 33 words: conflict-free both ways), and writes 128-byte segments
// of 64 consecutive p of one output row.
__global__ void __launch_bounds__(256)
    seg_transpose_kernel(const __nv_bfloat16* __restrict__ in, int64_t ld_in,
                         const int32_t* __restrict__ offsets, int groups, int dense_rows,
                         const int32_t* __restrict__ poff, const int32_t* __restrict__ gather,
                         int src_rows, const float* __restrict__ scale, int C,
                         __nv_bfloat16* __restrict__ out, int64_t ld_out, unsigned* status) {
  __shared__ uint32_t T[64][33];
  __shared__ int s_g;
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int p0 = blockIdx.y * 64, c0 = blockIdx.x * 64;
  if (p0 >= poff[groups]) return;  // past the last padded segment (uniform in the block)
  if (tid == 0) {
    int lo = 0, hi = groups;  // the group whose padded range holds p0
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (poff[mid] <= p0) lo = mid;
      else hi = mid;
    }
    s_g = lo;
  }
  __syncthreads();
  const int g = s_g;
  const int base = offsets ? offsets[g] : 0;
  const int n = offsets ? offsets[g + 1] - base : dense_rows;
  const int i0 = p0 - poff[g];
  // load: row pair pp (rows 2 pp, 2 pp + 1 of the tile), 8 columns cc*8 .. +7
  const int pp = warp * 4 + (lane >> 3), cc = lane & 7;
  uint32_t lo16[4], hi16[4];  // rows 2pp and 2pp+1, as 4 bf16 pairs each
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const int i = i0 + 2 * pp + h;
    if (i < n && c0 + cc * 8 < C) {
      const int r = base + i;
      int src = gather ? gather[r] : r;
      if (src < 0 || src >= src_rows) {
        atomicOr(status, kStatusDeviceData);
        src = -1;
      }
      if (src >= 0) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(in + int64_t(src) * ld_in + c0 + cc * 8));
        const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
        const float sc = scale ? scale[r] : 1.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f = __bfloat1622float2(b[q]);
          v[2 * q] = f.x * sc;
          v[2 * q + 1] = f.y * sc;
        }
      }
    }
    uint32_t* dst = h ? hi16 : lo16;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
      dst[q] = *reinterpret_cast<const uint32_t*>(&b2);
    }
  }
  // word (c, pp) = (row 2pp, row 2pp+1) at column c: low half from row 2pp
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    T[cc * 8 + 2 * q][pp] = __byte_perm(lo16[q], hi16[q], 0x5410);
    T[cc * 8 + 2 * q + 1][pp] = __byte_perm(lo16[q], hi16[q], 0x7632);
  }
  __syncthreads();
  // store: output row c = c0 + warp * 4 + lane / 8 (+ 32), 16 bytes = 8 p (4 words) a lane
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int cr = h * 32 + warp * 4 + (lane >> 3), wi = (lane & 7) * 4;
    if (c0 + cr >= C) continue;
    const uint4 o = make_uint4(T[cr][wi], T[cr][wi + 1], T[cr][wi + 2], T[cr][wi + 3]);
    *reinterpret_cast<uint4*>(out + int64_t(c0 + cr) * ld_out + p0 + wi * 2) = o;
  }
}

// Transposed weights for the backward's dgrad GEMMs, packed tile-major like the forward's
// ([g][N/BN][K/64][BN][64], one contiguous block per TMA box):
//   mode 0: N = Hn hidden units, K = M: element (g, n, k) = W_out[g][k][n], W_out [g][M][Hn];
//           with parts > 1 (shared experts side by side, g = 0): W_out[n / Hp][k][n % Hp].
//   mode 1: N = M, K = F: ReLU (F = Hn) element (g, n, k) = W_in[g][k][n]; SwiGLU (F = 2 Hn,
//           the forward's interleaved order) k = 256 b + c: c < 128: W_in[g][128 b + c][n],
//           else W_up[g][128 b + c - 128][n]. W_in, W_up [g][Hn][M] (shared experts: their
//           hidden units side by side, [Hn][M]).
__global__ void __launch_bounds__(256)
    pack_transposed_kernel(const __nv_bfloat16* __restrict__ W, const __nv_bfloat16* __restrict__ W2,
                           int mode, int swiglu, int groups, int N, int K, int M, int Hp, int parts,
                           int BN, __nv_bfloat16* __restrict__ dst) {
  const int64_t total = int64_t(groups) * N * (K / 8);
  for (int64_t u = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; u < total;
       u += int64_t(gridDim.x) * blockDim.x) {
    const int kq = int(u % (K / 8));
    const int64_t gn = u / (K / 8);
    const int n = int(gn % N);
    const int g = int(gn / N);
    const int k0 = kq * 8;
    __align__(16) __nv_bfloat16 v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int k = k0 + q;
      int64_t src;
      const __nv_bfloat16* base = W;
      if (mode == 0) {
        const int part = n / Hp, j = n % Hp;  // parts == 1: part 0, j = n
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
      v[q] = base[src];
    }
    const int64_t blk = (int64_t(g) * (N / BN) + n / BN) * (K / 64) + k0 / 64;
    *reinterpret_cast<uint4*>(dst + blk * BN * 64 + int64_t(n % BN) * 64 + (k0 % 64)) =
        *reinterpret_cast<const uint4*>(v);
  }
}

// dL/dlogits, one warp per token (lane l holds experts l, l + 32, ...):
//   gate term   MOE_GATE_SOFTMAX_TOPK: g = softmax over the k selected logits,
//               dl[id_j] += g_j (dg_j - sum_i g_i dg_i); MOE_GATE_NONE: g_j = p[id_j],
//               dl[id_j] += g_j dg_j and dl[e] -= p_e sum_j g_j dg_j; MOE_GATE_PNORM:
//               g_j = w_j / ||w||_p with w_j = exp(l_id_j - l_id_1) (the forward's gates),
//               dl[id_j] += g_j dg_j - g_j^p sum_i g_i dg_i;
//   aux term    aux_coef * E / (G * S_g) * p_e (f_e - sum_e' f_e' p_e'), f = counts_routed of
//               the token's group / (S_g k);
//   z term      z_coef * 2 / S * lse * p_e.
// dg_j (the gate's gradient) = sum of the n_tiles partials of gpart[row] (the GEMM's N
// tiles, two column halves each, in order) for a kept assignment, 0 for a dropped one (it
// adds nothing to y).
template <int KMAX>
__global__ void __launch_bounds__(256)
    router_bwd_kernel(const float* __restrict__ logits, const int32_t* __restrict__ expert_id,
                      const int32_t* __restrict__ row, const float* __restrict__ gpart, int n_tiles,
                      const int32_t* __restrict__ counts_routed, int S, int G, int E, int k,
                      int gate_norm, float gate_p, float aux_coef, float z_coef,
                      float* __restrict__ dlogits,
                      __nv_bfloat16* __restrict__ dlb, int Ep) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = int((int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  if (t >= S) return;
  const float* lr = logits + int64_t(t) * E;
  float l[8], p[8];
  float m = -INFINITY;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int e = lane + 32 * q;
    l[q] = e < E ? lr[e] : -INFINITY;
    m = fmaxf(m, l[q]);
  }
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float s = 0.f;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    p[q] = lane + 32 * q < E ? expf(l[q] - m) : 0.f;
    s += p[q];
  }
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  const float inv = 1.f / s, lse = m + logf(s);
#pragma unroll
  for (int q = 0; q < 8; ++q) p[q] *= inv;
  // the k choices: ids, selected logits, gate gradients (lane j < k gathers dg_j)
  int id[KMAX];
  float dg[KMAX], gsel[KMAX];
  float dgl = 0.f;
  if (lane < k) {
    const int r = row[int64_t(t) * k + lane];
    if (r >= 0)
      for (int nt = 0; nt < n_tiles; ++nt) dgl += gpart[int64_t(r) * n_tiles + nt];
  }
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    id[j] = j < k ? expert_id[int64_t(t) * k + j] : 0;
    dg[j] = __shfl_sync(0xffffffffu, dgl, j);
    gsel[j] = j < k ? lr[id[j]] : -INFINITY;
  }
  float dl[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (gate_norm == MOE_GATE_SOFTMAX_TOPK) {
    const float top = gsel[0];  // the largest selected logit
    float gs = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      gsel[j] = j < k ? expf(gsel[j] - top) : 0.f;
      gs += gsel[j];
    }
    float inner = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      gsel[j] /= gs;
      inner += gsel[j] * dg[j];
    }
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (j < k && id[j] == lane + 32 * q) dl[q] += gsel[j] * (dg[j] - inner);
  } else if (gate_norm == MOE_GATE_PNORM) {
    // g_j^p = w_j^p / sum_i w_i^p: kept as w_j^p in wp[] and divided once
    const float top = gsel[0];
    float wp[KMAX], sp = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      gsel[j] = j >= k ? 0.f : (top > -INFINITY ? expf(gsel[j] - top) : (j == 0 ? 1.f : 0.f));
      wp[j] = j < k ? powf(gsel[j], gate_p) : 0.f;
      sp += wp[j];
    }
    const float ginv = 1.f / powf(sp, 1.f / gate_p), spinv = 1.f / sp;
    float inner = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      gsel[j] *= ginv;
      inner += gsel[j] * dg[j];
    }
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (j < k && id[j] == lane + 32 * q) dl[q] += gsel[j] * dg[j] - wp[j] * spinv * inner;
  } else {  // MOE_GATE_NONE
    float inner = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      gsel[j] = j < k ? expf(gsel[j] - m) * inv : 0.f;
      inner += gsel[j] * dg[j];
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) dl[q] -= p[q] * inner;
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (j < k && id[j] == lane + 32 * q) dl[q] += gsel[j] * dg[j];
  }
  const int Sg = S / G;
  if (aux_coef != 0.f) {
    const int32_t* cr = counts_routed + int64_t(t / Sg) * E;
    const float fs = 1.f / (float(Sg) * float(k));
    float f[8], fp = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = lane + 32 * q;
      f[q] = e < E ? float(cr[e]) * fs : 0.f;
      fp += f[q] * p[q];
    }
    for (int off = 16; off > 0; off >>= 1) fp += __shfl_xor_sync(0xffffffffu, fp, off);
    const float c = aux_coef * float(E) / (float(G) * float(Sg));
#pragma unroll
    for (int q = 0; q < 8; ++q) dl[q] += c * p[q] * (f[q] - fp);
  }
  if (z_coef != 0.f) {
    const float c = z_coef * 2.f / float(S) * lse;
#pragma unroll
    for (int q = 0; q < 8; ++q) dl[q] += c * p[q];
  }
  float* out = dlogits + int64_t(t) * E;
  __nv_bfloat16* outb = dlb + int64_t(t) * Ep;  // bf16, zero-padded to Ep: the GEMMs' operand
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int e = lane + 32 * q;
    if (e < E) out[e] = dl[q];
    if (e < Ep) outb[e] = __float2bfloat16_rn(e < E ? dl[q] : 0.f);
  }
}

// dbias: part[ch][e] = sum over chunk ch's 256 tokens of dl[t][e] (thread e, tokens in order),
// then out[e] = sum over chunks in order (sum_partials_kernel).
__global__ void __launch_bounds__(256)
    colsum_partial_kernel(const float* __restrict__ dl, int S, int E, float* __restrict__ part) {
  pdl_wait();
  pdl_trigger();
  const int e = threadIdx.x, ch = blockIdx.x;
  if (e >= E) return;
  const int t1 = min(S, (ch + 1) * 256);
  float acc = 0.f;
  for (int t = ch * 256; t < t1; ++t) acc += dl[int64_t(t) * E + e];
  part[int64_t(ch) * E + e] = acc;
}

// Gather into per-expert 64-padded segments (the row-major A or B operand of the weight-
// gradient GEMM): padded row p of expert e (poff[e] <= p < poff[e+1]) is
// scale[r] * src[token_of[r]] with r = offsets[e] + p - poff[e] while p - poff[e] is below
// e's row count, and zeros after it. One warp per padded row, 16-byte units (bf16, rounded
// to nearest even after an fp32 multiply). With tail, the 64 rows of tail from row
// offsets[E] on (tail_units a row) are zeroed too: the GEMM reads them past the last
// segment.
__global__ void __launch_bounds__(256)
    pad_gather_kernel(const uint4* __restrict__ src, int units, const int32_t* __restrict__ token_of,
                      const float* __restrict__ scale, const int32_t* __restrict__ offsets,
                      const int32_t* __restrict__ poff, int E, int S, int64_t rows_bound,
                      uint4* __restrict__ out, uint4* __restrict__ tail, int tail_units,
                      unsigned* __restrict__ status) {
  __shared__ int s_poff[257], s_off[257];
  pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i <= E; i += blockDim.x) {
    s_poff[i] = poff[i];
    s_off[i] = offsets[i];
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t w0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const int64_t P = min(int64_t(s_poff[E]), rows_bound);
  for (int64_t p = w0; p < P; p += nw) {
    int lo = 0, hi = E;  // the expert e with poff[e] <= p < poff[e + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_poff[mid] <= p) lo = mid;
      else hi = mid;
    }
    const int64_t local = p - s_poff[lo];
    uint4* dst = out + p * units;
    int t = -1;
    float sc = 1.f;
    if (local < s_off[lo + 1] - s_off[lo]) {
      const int64_t r = s_off[lo] + local;
      t = token_of[r];
      if (scale) sc = scale[r];
      if (unsigned(t) >= unsigned(S)) {
        if (lane == 0) atomicOr(status, kStatusDeviceData);
        t = -1;
      }
    }
    if (t < 0) {
      for (int q = lane; q < units; q += 32) dst[q] = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    const uint4* row = src + int64_t(t) * units;
    for (int q = lane; q < units; q += 32) {
      uint4 v = __ldg(row + q);
      if (scale) {
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __bfloat1622float2(h[i]);
          h[i] = __floats2bfloat162_rn(f.x * sc, f.y * sc);
        }
      }
      dst[q] = v;
    }
  }
  if (tail && w0 < 64) {
    uint4* trow = tail + (int64_t(s_off[E]) + w0) * tail_units;
    for (int q = lane; q < tail_units; q += 32) trow[q] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// koffs[i] = min(total, i * chunk) for i = 0..n: split-K ranges of one K-ragged GEMM.
__global__ void split_offsets_kernel(int n, int chunk, int total, int32_t* __restrict__ koffs) {
  pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i <= n; i += blockDim.x) koffs[i] = min(total, i * chunk);
}

// out[i] = sum over s = 0..n-1, in order, of part[s * stride + i], i < len (split-K
// partials).
__global__ void __launch_bounds__(256)
    sum_partials_kernel(const float* __restrict__ part, int n, int64_t len, int64_t stride,
                        float* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= len) return;
  float acc = 0.f;
  for (int s = 0; s < n; ++s) acc += part[int64_t(s) * stride + i];
  out[i] = acc;
}

}  // namespace

int launch_pad_gather(const void* src, int cols, const int32_t* token_of, const float* scale,
                      const int32_t* offsets, const int32_t* poff, int E, int S, int64_t rows_bound,
                      void* out, void* tail, int tail_cols, unsigned* status, cudaStream_t st) {
  if (E > 256 || cols % 8 || tail_cols % 8) return MOE_ERR_UNSUPPORTED;
  int64_t blocks = (rows_bound * 32 + 255) / 256;
  const int64_t cap = int64_t(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 8) blocks = 8;  // the first 64 warps zero the tail
  return launch_kernel(pad_gather_kernel, dim3(unsigned(blocks)), dim3(256), 0, st,
                       static_cast<const uint4*>(src), cols / 8, token_of, scale, offsets, poff, E,
                       S, rows_bound, static_cast<uint4*>(out), static_cast<uint4*>(tail),
                       tail_cols / 8, status);
}

int launch_pad_offsets(const int32_t* offsets, int groups, int dense_rows, int32_t* poff,
                       cudaStream_t st) {
  return launch_kernel(pad_offsets_kernel, dim3(1), dim3(32), 0, st, offsets, groups, dense_rows,
                       poff);
}

int launch_seg_transpose(const void* in, int64_t ld_in, const int32_t* offsets, int groups,
                         int dense_rows, const int32_t* poff, int64_t rows_pad_max,
                         const int32_t* gather, int src_rows, const float* scale, int C, void* out,
                         int64_t ld_out, unsigned* status, cudaStream_t st) {
  if (C % 8 || ld_in % 8 || ld_out % 8 || rows_pad_max % 64) return MOE_ERR_UNSUPPORTED;
  const dim3 grid(unsigned((C + 63) / 64), unsigned(rows_pad_max / 64));
  if (grid.y == 0) return MOE_OK;
  return launch_kernel(seg_transpose_kernel, grid, dim3(256), 0, st,
                       static_cast<const __nv_bfloat16*>(in), ld_in, offsets, groups, dense_rows,
                       poff, gather, src_rows, scale, C, static_cast<__nv_bfloat16*>(out), ld_out,
                       status);
}

int launch_pack_transposed(int mode, int swiglu, int groups, int N, int K, int M, int Hp, int parts,
                           const void* W, const void* W2, void* dst, cudaStream_t st) {
  const int BN = mode == 0 ? gemm_bn(N, EPI_DGRAD2) : gemm_bn(N, EPI_SCALE);
  if (BN <= 0 || N % BN || K % 64) return MOE_ERR_UNSUPPORTED;
  const int64_t total = int64_t(groups) * N * (K / 8);
  const unsigned grid = unsigned((total + 255) / 256 < 65535 * 8 ? (total + 255) / 256 : 65535 * 8);
  pack_transposed_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(W),
                                               static_cast<const __nv_bfloat16*>(W2), mode, swiglu,
                                               groups, N, K, M, Hp, parts, BN,
                                               static_cast<__nv_bfloat16*>(dst));
  MOE_CUDA_CHECK(cudaGetLastError());
  return MOE_OK;
}

// dbias = the column sums of dlogits, in a fixed order (the partials reuse the dW_g partial
// buffer); nothing without dbias
int router_dbias(const moe_config_t& c, const RouterBwdBufs& b, float* dbias, cudaStream_t st) {
  if (!dbias) return MOE_OK;
  const int nch = (c.S + 255) / 256;
  int rc;
  if ((rc = launch_kernel(colsum_partial_kernel, dim3(unsigned(nch)), dim3(256), 0, st,
                          static_cast<const float*>(b.dlogits), c.S, c.E, b.dwg_part)) != MOE_OK)
    return rc;
  return launch_kernel(sum_partials_kernel, dim3(unsigned((c.E + 255) / 256)), dim3(256), 0, st,
                       static_cast<const float*>(b.dwg_part), nch, int64_t(c.E), int64_t(c.E), dbias);
}

int launch_router_backward(const moe_config_t& c, const float* logits, const moe_route_out_t& r,
                           const float* gpart, int n_tiles, float aux_coef, float z_coef,
                           const RouterBwdBufs& b, const void* x, const void* W_g, float* dW_g,
                           float* dbias, unsigned* status, cudaStream_t st) {
  if (c.E > 256) return MOE_ERR_UNSUPPORTED;
  const int Ep = (c.E + 63) / 64 * 64;
  const unsigned blocks = unsigned((int64_t(c.S) * 32 + 255) / 256);
  int rc;
  if (c.k <= 2)
    rc = launch_kernel(router_bwd_kernel<2>, dim3(blocks), dim3(256), 0, st, logits, r.expert_id, r.row,
                       gpart, n_tiles, r.counts_routed, c.S, c.G, c.E, c.k, c.gate_norm, c.gate_p, aux_coef,
                       z_coef, b.dlogits, static_cast<__nv_bfloat16*>(b.dlb), Ep);
  else
    rc = launch_kernel(router_bwd_kernel<8>, dim3(blocks), dim3(256), 0, st, logits, r.expert_id, r.row,
                       gpart, n_tiles, r.counts_routed, c.S, c.G, c.E, c.k, c.gate_norm, c.gate_p, aux_coef,
                       z_coef, b.dlogits, static_cast<__nv_bfloat16*>(b.dlb), Ep);
  if (rc != MOE_OK) return rc;
  if (c.dtype == MOE_F32) {  // the fp32 path: dx_r and dW_g on plain FMA (backward_f32.cu)
    if ((rc = router_grads_f32(c, b.dlogits, x, W_g, b.dx_r, dW_g, st)) != MOE_OK) return rc;
    return router_dbias(c, b, dbias, st);
  }
  // K ranges of the two router GEMMs: [0, Ep) and [0, Sp)
  if ((rc = launch_pad_offsets(nullptr, 1, c.E, b.koff_e, st)) != MOE_OK) return rc;
  if ((rc = launch_pad_offsets(nullptr, 1, c.S, b.koff_s, st)) != MOE_OK) return rc;
  // W_g^T [M][Ep] (zero-padded), the B operand of dx_r
  if ((rc = launch_seg_transpose(W_g, c.M, nullptr, 1, c.E, b.koff_e, Ep, nullptr, c.E, nullptr, c.M,
                                 b.wgT, Ep, status, st)) != MOE_OK)
    return rc;

  // dx_r [S][M] = dl . W_g (one group of S rows, K = Ep); dW_g [E][M] = dl^T . x (K = Sp)
  GemmDesc d;
  d.epi = EPI_F32_BIAS;
  d.A = b.dlb; d.a_rows = c.S; d.K = Ep;
  d.B = b.wgT; d.N = c.M; d.b_rows = c.M; d.b_tiled = false;
  d.koffs = b.koff_e; d.c1 = c.S; d.groups = 1;
  d.out = b.dx_r; d.ldo = c.M; d.n_valid = c.M; d.status = status;
  if ((rc = launch_gemm_bf16(d, st)) != MOE_OK) return rc;
  // dW_g: K = Sp split into nsplit ranges (one output tile per 128 experts x 256 columns
  // would otherwise leave most SMs idle over a long K), partials summed in order
  const int64_t kblk = b.Sp / 64;
  const int tiles = ((c.E + 127) / 128) * ((c.M + 255) / 256);
  int nsplit = (2 * num_sms() + tiles - 1) / tiles;
  if (nsplit > b.max_split) nsplit = b.max_split;
  if (nsplit > kblk) nsplit = int(kblk);
  if (nsplit < 1) nsplit = 1;
  const int chunk = int((kblk + nsplit - 1) / nsplit) * 64;
  if ((rc = launch_kernel(split_offsets_kernel, dim3(1), dim3(64), 0, st, nsplit, chunk, int(b.Sp),
                          b.koff_split)) != MOE_OK)
    return rc;
  // MN-major operands read in place: A = dl [S][Ep] (bf16), B = x [S][M]; rows past S read
  // as zeros. Split s writes rows s * Ep .. of the partials (rows E .. Ep - 1 are zeros).
  GemmDesc w;
  w.epi = EPI_F32_BIAS;
  w.mn = true;
  w.A = b.dlb; w.a_krows = c.S; w.a_rows = Ep; w.K = int(b.Sp);
  w.B = x; w.b_krows = c.S; w.N = c.M; w.b_rows = c.M; w.b_tiled = false;
  w.koffs = b.koff_split; w.c1 = Ep; w.groups = nsplit;
  w.out = b.dwg_part; w.ldo = c.M; w.n_valid = c.M; w.status = status;
  if ((rc = launch_gemm_bf16(w, st)) != MOE_OK) return rc;
  const int64_t len = int64_t(c.E) * c.M;
  if ((rc = launch_kernel(sum_partials_kernel, dim3(unsigned((len + 255) / 256)), dim3(256), 0, st,
                          static_cast<const float*>(b.dwg_part), nsplit, len, int64_t(Ep) * c.M,
                          dW_g)) != MOE_OK)
    return rc;
  return router_dbias(c, b, dbias, st);
}

}  // namespace moe
