// Grouped bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM), fed by TMA.
//
//   D[r, n] = sum_k A[r, k] * B[g * N + n, k]   for the rows r of group g,
//
// A [rows, K] row-major and B [groups * N, K] (row-major, or packed tile-major by
// launch_pack_in / launch_pack_out), both K-major like the [out, in] weights of a linear
// layer, fp32 accumulation in tensor memory, a fused epilogue:
//   EPI_F32_BIAS  fp32 out (+ per-column bias)          -- router logits
//   EPI_RELU      bf16 out = relu(D)                    -- expert GEMM 1, ReLU expert
//   EPI_SWIGLU    bf16 out = silu(D_gate) * D_up        -- expert GEMM 1, SwiGLU expert
//   EPI_SCALE     bf16 out = row_scale[r] * D           -- expert GEMM 2 (gate weighting)
//
// GShard summary page, "MoE Transformer": each expert is a two-layer FFN of the dense
// FFN's shape, weighted by its gate in the combination. Lec16 Systems for MoE Models,
// "DeepSeek V3 MoE": SwiGLU experts. MegaBlocks router chapter §4: the experts' rows come
// in expert-contiguous segments of uneven length (here read from device offsets, so the
// host never synchronises to size the grid).
//
// Structure (persistent: one CTA per SM, looping over output tiles):
//   warp 0      one lane issues TMA loads of its A rows (128 x 64) and B rows (x 64) into a
//               ring of shared-memory stages (128-byte swizzle), signalling `full` barriers;
//   warp 1      owns tensor memory; one lane issues tcgen05.mma (K = 16 per instruction)
//               into one of two TMEM accumulators, committing each stage to its `empty`
//               barrier and each tile to the accumulator's `tfull` barrier;
//   warps 2..5  epilogue: tcgen05.ld the accumulator (warp w reads TMEM lanes 32*(w%4)..),
//               apply the fused epilogue, store, then arrive on the accumulator's `tempty`
//               barrier, so the next tile's MMAs overlap this tile's epilogue.
// PAIR = false: one CTA computes a 128 x BN tile (cta_group::1).
// PAIR = true:  a cluster of two CTAs computes a 256 x BN tile with cta_group::2 MMAs: each
//               CTA stages its 128 rows of A and BN/2 rows of B (half the weight bytes per
//               SM per output of the single-CTA tile); the even CTA issues the MMAs, which
//               read both CTAs' shared memory and write each CTA's 128 accumulator rows into
//               its own TMEM; both CTAs' loads complete on the even CTA's `full` barrier, its
//               commits arrive on both CTAs' `empty` / `tfull` barriers, and both epilogues
//               arrive on its `tempty` barrier.
// Tiles are ordered group by group, then by N tile, then by M tile, so the CTAs that run
// at the same time share each weight tile through L2.
//
// Every wait is bounded: after the wait limit (2 s unless set in the workspace header) a
// waiting thread sets the status word's timeout bit and a CTA-wide abort flag; every role
// then stops and, after a CTA barrier, the producer waits for its loads in flight and the
// MMA thread for its MMAs, whichever role gave up; TMEM is freed before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // bf16 elements per 128-byte swizzled row
constexpr int kMaxGroups = 256;

// The bf16 epilogues whose output goes out through shared memory and TMA stores (see
// epilogue_bf16_tma): activation (GEMM 1) and gate scaling (GEMM 2).
template <int EPI, bool KRAG>
constexpr bool tma_epilogue() {
  return !KRAG && (EPI == EPI_RELU || EPI == EPI_SWIGLU || EPI == EPI_SCALE || EPI == EPI_DGRAD2 ||
                   EPI == EPI_SWIGLU_BWD);
}
// its boxes: 32 rows x 64 bf16 (128-byte swizzle, 4 KB) for the four-warp epilogues, 32 rows
// x 32 bf16 (64-byte swizzle, 2 KB) for the eight-warp data-gradient epilogues: 16 KB a CTA
template <int EPI>
constexpr bool tma_box32() {
  return EPI == EPI_DGRAD2 || EPI == EPI_SWIGLU_BWD;
}

template <int BN, bool PAIR, bool KRAG = false, bool TEPI = false>
struct Cfg {
  static constexpr int CTAS = PAIR ? 2 : 1;
  static constexpr int TILE_M = BM * CTAS;  // rows of one output tile
  static constexpr int B_ROWS = BN / CTAS;  // B rows each CTA stages
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = B_ROWS * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // K-ragged mode: each epilogue warp stages fp32 outputs in boxes of 32 rows x F32_BOX
  // columns that TMA stores to global memory: 32 columns (128-byte rows, 4 KB, two buffers a
  // warp) for single-CTA tiles; 16 columns (64-byte rows, 2 KB, three buffers) for CTA pairs,
  // whose 32 KB k-blocks then get a sixth ring stage. (Single-CTA 256-wide tiles would get a
  // fourth 48 KB stage the same way, but there the twice as many, half-size stores cost more
  // than the stage gains.) The bf16 TMA epilogue: 16 KB (one box a warp, see tma_box32).
  static constexpr int F32_BOX = PAIR ? 16 : 32;
  static constexpr int F32_BUFS = PAIR ? 3 : 2;
  static constexpr int STG_BYTES = KRAG ? 4 * F32_BUFS * 32 * F32_BOX * 4 : (TEPI ? 4 * 4096 : 0);
  // shared memory a CTA may take (227 KB) less the alignment slack, the barriers (for up to
  // 8 stages), the TMEM address and flags, and the group tables
  static constexpr int FIXED = 1024 + (2 * 8 + 5) * 8 + 16 + 3 * (kMaxGroups + 1) * 4;
  static constexpr int RING = 232448 - FIXED - STG_BYTES;
  static constexpr int STAGES = (RING / STAGE_BYTES) > 8 ? 8 : (RING / STAGE_BYTES);
  static constexpr int TMEM_COLS = 2 * BN < 32 ? 32 : 2 * BN;
  static constexpr int BAR_BYTES = (2 * STAGES + 5) * 8;
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + STG_BYTES + BAR_BYTES + 16 +
                              3 * (kMaxGroups + 1) * 4;
};

// Epilogue warps: four, one per 32 TMEM lanes. The data-gradient epilogues, whose
// per-element work (the stored h or dh read back, the mask or the SwiGLU derivative, the
// gate partials) can outlast a tile's MMAs, have eight: two per 32 lanes, each taking half
// of the tile's columns.
template <int EPI, bool KRAG>
constexpr int epi_warps() {
  return (!KRAG && (EPI == EPI_DGRAD2 || EPI == EPI_SWIGLU_BWD)) ? 8 : 4;
}

struct KParams {
  const int32_t* offsets;
  int b_tiled;  // B packed tile-major: box (g, nt, kb) is block (g * n_tiles + nt) * kblocks + kb
  int groups;
  int rows_dense;
  int64_t rows_cap;
  int N, K, n_tiles;
  void* out;
  int64_t ldo;
  const float* row_scale;
  const float* bias;
  int n_valid;
  unsigned* status;
  const void* aux;  // EPI_DGRAD2: h; EPI_SWIGLU_BWD: dh (bf16)
  int64_t ld_aux;
  float* gpart;     // EPI_DGRAD2: [rows][n_tiles][2] sums of D * h over each half of a
                    // tile's columns, nullable
  int relu;
  const int32_t* koffs;  // K-ragged mode: per-group K range
  int c1;                // K-ragged mode: output rows per group
  void* out2;            // interleaved SwiGLU rows: the second 128-row block of each pair
  const char* pfB;       // tile-major B, nullable: prefetch the start of the first tile
  int64_t pf_bytes;      // bytes of that tile to prefetch into L2
  // K-ragged MN-major mode: A [.., c1] and B [.., N] row-major (K = rows); group g's K rows
  // start at aoffs[g] in A and boffs[g] in B (null: koffs[g]), koffs giving the lengths
  const int32_t* aoffs;
  const int32_t* boffs;
  int reverse;  // walk the tile schedule from its last tile (grouped rows only)
  int out_keep; // bf16 output read by the next kernel: stores marked evict-last in L2
};

using namespace sm100;

// ------------------------------------------------------------------ the epilogue
// One warp drains 32 accumulator rows (TMEM lanes) x BN columns at `tbase`; the thread
// holding tile row `grow` stores it if `valid`. nt: the tile's N index. With eight
// epilogue warps (the data-gradient epilogues) the warp takes half `part` of the columns.
template <int BN, int EPI>
__device__ __forceinline__ void epilogue_rows(const KParams& p, uint32_t tbase, bool valid,
                                              int64_t grow, int nt, bool zero = false, int part = 0) {
  if constexpr (EPI == EPI_F32_BIAS) {
    float* out = static_cast<float*>(p.out) + grow * p.ldo;
    if (p.out2) {  // row j of group g in the interleaved SwiGLU order (128 gate, 128 up rows)
      const int64_t g = grow / p.c1, j = grow % p.c1, c = j & 255;
      out = static_cast<float*>(c < 128 ? p.out : p.out2) +
            (g * (p.c1 / 2) + (j >> 8) * 128 + (c & 127)) * p.ldo;
    }
    const bool vec = (p.ldo & 3) == 0;
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 16) {
      uint32_t v[16];
      tmem_ld16(tbase + c0, v);
      tmem_ld_wait();
      if (valid) {
        const int nb = nt * BN + c0;
        float f[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          f[j] = zero ? 0.f  // a K-ragged group with no rows: its gradient is 0
                      : __uint_as_float(v[j]) + ((p.bias && nb + j < p.n_valid) ? p.bias[nb + j] : 0.f);
        if (vec && nb + 16 <= p.n_valid) {
          float4* d = reinterpret_cast<float4*>(out + nb);
#pragma unroll
          for (int j = 0; j < 4; ++j) d[j] = make_float4(f[4 * j], f[4 * j + 1], f[4 * j + 2], f[4 * j + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (nb + j < p.n_valid) out[nb + j] = f[j];
        }
      }
    }
  } else if constexpr (EPI == EPI_DGRAD2) {
    // D = dy_perm . W_out (unscaled); out = w_r * D (ReLU: where h > 0), gate partial
    // sum_c D * h over this tile's columns (h as the forward stored it, bf16)
    // columns cb .. ce - 1 of the tile: half `part`
    constexpr int kHalf = BN / 2;
    const int cb = part * kHalf, ce = cb + kHalf;
    const float scale = (valid && p.row_scale) ? p.row_scale[grow] : 1.f;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + grow * p.ldo + nt * BN;
    const __nv_bfloat16* hrow = static_cast<const __nv_bfloat16*>(p.aux) + grow * p.ld_aux + nt * BN;
    float gsum = 0.f;
    // h of 32 columns per step, the next step's loads issued before this step's math
    uint4 hn[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      hn[q] = valid ? __ldg(reinterpret_cast<const uint4*>(hrow + cb) + q) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 1
    for (int c0 = cb; c0 < ce; c0 += 32) {
      uint4 hc[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) hc[q] = hn[q];
      if (valid && c0 + 32 < ce) {
#pragma unroll
        for (int q = 0; q < 4; ++q) hn[q] = __ldg(reinterpret_cast<const uint4*>(hrow + c0 + 32) + q);
      }
      uint32_t v[32];
      tmem_ld16(tbase + c0, *reinterpret_cast<uint32_t(*)[16]>(v));
      tmem_ld16(tbase + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
      tmem_ld_wait();
      if (valid) {
        const uint32_t* hw = reinterpret_cast<const uint32_t*>(hc);
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float2 hv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hw[j]));
          const float d0 = __uint_as_float(v[2 * j]), d1 = __uint_as_float(v[2 * j + 1]);
          gsum += d0 * hv.x + d1 * hv.y;
          float o0 = d0 * scale, o1 = d1 * scale;
          if (p.relu) {
            o0 = hv.x > 0.f ? o0 : 0.f;
            o1 = hv.y > 0.f ? o1 : 0.f;
          }
          pk[j] = pack_bf16x2(o0, o1);
        }
        if (p.out_keep) {
          const uint64_t pol = policy_evict_last();
          store_bf16x16_hint(out + c0, *reinterpret_cast<const uint32_t(*)[8]>(pk), pol);
          store_bf16x16_hint(out + c0 + 16, *reinterpret_cast<const uint32_t(*)[8]>(pk + 8), pol);
        } else {
          store_bf16x16(out + c0, *reinterpret_cast<const uint32_t(*)[8]>(pk));
          store_bf16x16(out + c0 + 16, *reinterpret_cast<const uint32_t(*)[8]>(pk + 8));
        }
      }
    }
    if (valid && p.gpart) p.gpart[(grow * p.n_tiles + nt) * 2 + part] = gsum;
  } else if constexpr (EPI == EPI_SWIGLU_BWD) {
    // D = (a | b): the tile's 128 gate and 128 up pre-activations of hidden units
    // 128 nt ..; with dh: da = dh * b * silu'(a), db = dh * silu(a), written to the same
    // interleaved column positions (out [rows, 2H])
    // hidden units cb .. ce - 1 of the tile's BN / 2: half `part`
    constexpr int kQuarter = BN / 4;
    const int cb = part * kQuarter, ce = cb + kQuarter;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + grow * p.ldo + nt * BN;
    const __nv_bfloat16* dhrow = static_cast<const __nv_bfloat16*>(p.aux) + grow * p.ld_aux + nt * (BN / 2);
    uint4 dn[2];  // the next step's dh, loaded before this step's math
#pragma unroll
    for (int q = 0; q < 2; ++q)
      dn[q] = valid ? __ldg(reinterpret_cast<const uint4*>(dhrow + cb) + q) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 1
    for (int c0 = cb; c0 < ce; c0 += 16) {
      const uint4 d0 = dn[0], d1 = dn[1];
      if (valid && c0 + 16 < ce) {
        dn[0] = __ldg(reinterpret_cast<const uint4*>(dhrow + c0 + 16));
        dn[1] = __ldg(reinterpret_cast<const uint4*>(dhrow + c0 + 16) + 1);
      }
      uint32_t av[16], bv[16];
      tmem_ld16(tbase + c0, av);
      tmem_ld16(tbase + BN / 2 + c0, bv);
      tmem_ld_wait();
      if (valid) {
        const uint32_t dw[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
        uint32_t pa[8], pb[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float2 dh = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&dw[j]));
          float da[2], db[2];
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const float a = __uint_as_float(av[2 * j + q]), b = __uint_as_float(bv[2 * j + q]);
            const float sg = 1.f / (1.f + __expf(-a));
            const float d = q ? dh.y : dh.x;
            da[q] = d * b * sg * (1.f + a * (1.f - sg));
            db[q] = d * a * sg;
          }
          pa[j] = pack_bf16x2(da[0], da[1]);
          pb[j] = pack_bf16x2(db[0], db[1]);
        }
        store_bf16x16(out + c0, pa);
        store_bf16x16(out + BN / 2 + c0, pb);
      }
    }
  } else if constexpr (EPI == EPI_SWIGLU) {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + grow * p.ldo + nt * (BN / 2);
#pragma unroll 1
    for (int c0 = 0; c0 < BN / 2; c0 += 16) {
      uint32_t gv[16], uv[16];
      tmem_ld16(tbase + c0, gv);
      tmem_ld16(tbase + BN / 2 + c0, uv);
      tmem_ld_wait();
      if (valid) {
        uint32_t pk[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float g0 = __uint_as_float(gv[2 * j]), g1 = __uint_as_float(gv[2 * j + 1]);
          const float h0 = g0 / (1.f + __expf(-g0)) * __uint_as_float(uv[2 * j]);
          const float h1 = g1 / (1.f + __expf(-g1)) * __uint_as_float(uv[2 * j + 1]);
          pk[j] = pack_bf16x2(h0, h1);
        }
        store_bf16x16(out + c0, pk);
      }
    }
  } else {
    float scale = 1.f;
    if (EPI == EPI_SCALE && valid && p.row_scale) scale = p.row_scale[grow];
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + grow * p.ldo + nt * BN;
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
      uint32_t v0[16], v1[16];
      tmem_ld16(tbase + c0, v0);
      tmem_ld16(tbase + c0 + 16, v1);
      tmem_ld_wait();
      if (valid) {
        uint32_t pk0[8], pk1[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float a0 = __uint_as_float(v0[2 * j]), a1 = __uint_as_float(v0[2 * j + 1]);
          float b0 = __uint_as_float(v1[2 * j]), b1 = __uint_as_float(v1[2 * j + 1]);
          if (EPI == EPI_RELU) {
            a0 = fmaxf(a0, 0.f); a1 = fmaxf(a1, 0.f); b0 = fmaxf(b0, 0.f); b1 = fmaxf(b1, 0.f);
          } else {
            a0 *= scale; a1 *= scale; b0 *= scale; b1 *= scale;
          }
          pk0[j] = pack_bf16x2(a0, a1);
          pk1[j] = pack_bf16x2(b0, b1);
        }
        if (p.out_keep) {
          const uint64_t q = policy_evict_last();
          store_bf16x16_hint(out + c0, pk0, q);
          store_bf16x16_hint(out + c0 + 16, pk1, q);
        } else {
          store_bf16x16(out + c0, pk0);
          store_bf16x16(out + c0 + 16, pk1);
        }
      }
    }
  }
}

// The bf16 epilogues (activation, gate scale) of one warp through shared memory: rows
// grow0 .. grow0 + 31 of the output (the first nvr valid), 64 output columns at a time. The
// warp reads its accumulator rows from TMEM, applies the epilogue, and, when all 32 rows
// are valid, writes them as bf16 into a 128-byte-swizzled 32 x 64 box in shared memory
// (conflict-free) that lane 0 stores with one TMA tensor store; the box is rewritten once
// that store has read it, a wait that the next columns' TMEM loads and math overlap. A
// warp whose rows end inside it (the last rows of an expert's segment) stores its valid
// rows from registers instead, so that no row of the next segment is written. Storing each
// lane's row directly made every warp store touch 32 lines: with a wide output (GEMM 1's h,
// d_ff wide) that kept L1 at 70 % of its throughput and the tensor pipe at 77 %.
template <int BN, int EPI>
__device__ __forceinline__ void epilogue_bf16_tma(const KParams& p, const CUtensorMap* tmO,
                                                  uint32_t tbase, int64_t grow0, int nvr, int nt,
                                                  uint8_t* buf, int lane) {
  constexpr int OUT_COLS = EPI == EPI_SWIGLU ? BN / 2 : BN;  // output columns of a tile
  const int64_t ocol0 = int64_t(nt) * OUT_COLS;
  float scale = 1.f;
  if (EPI == EPI_SCALE && lane < nvr && p.row_scale) scale = p.row_scale[grow0 + lane];
  const bool full = nvr == 32;
  const uint64_t pol = p.out_keep ? policy_evict_last() : 0ull;
#pragma unroll 1
  for (int c0 = 0; c0 < OUT_COLS; c0 += 64) {
    uint32_t pk[32];  // this lane's row: 64 bf16 of the chunk
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // 32 output columns at a time
      const int c = c0 + 32 * h;
      if constexpr (EPI == EPI_SWIGLU) {
        uint32_t g0[16], g1[16], u0[16], u1[16];
        tmem_ld16(tbase + c, g0);
        tmem_ld16(tbase + c + 16, g1);
        tmem_ld16(tbase + BN / 2 + c, u0);
        tmem_ld16(tbase + BN / 2 + c + 16, u1);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t* gv = j < 8 ? g0 : g1;
          const uint32_t* uv = j < 8 ? u0 : u1;
          const int jj = 2 * (j & 7);
          const float a0 = __uint_as_float(gv[jj]), a1 = __uint_as_float(gv[jj + 1]);
          const float h0 = a0 / (1.f + __expf(-a0)) * __uint_as_float(uv[jj]);
          const float h1 = a1 / (1.f + __expf(-a1)) * __uint_as_float(uv[jj + 1]);
          pk[16 * h + j] = pack_bf16x2(h0, h1);
        }
      } else {
        uint32_t v0[16], v1[16];
        tmem_ld16(tbase + c, v0);
        tmem_ld16(tbase + c + 16, v1);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t* v = j < 8 ? v0 : v1;
          const int jj = 2 * (j & 7);
          float a0 = __uint_as_float(v[jj]), a1 = __uint_as_float(v[jj + 1]);
          if (EPI == EPI_RELU) {
            a0 = fmaxf(a0, 0.f);
            a1 = fmaxf(a1, 0.f);
          } else {
            a0 *= scale;
            a1 *= scale;
          }
          pk[16 * h + j] = pack_bf16x2(a0, a1);
        }
      }
    }
    if (full) {
      if (lane == 0) bulk_wait_read<0>();  // the previous box's store has read the buffer
      __syncwarp();
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<uint4*>(buf + lane * 128 + ((q ^ (lane & 7)) << 4)) =
            make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (p.out_keep) tma_store_2d_hint(tmO, int(ocol0 + c0), int(grow0), smem_u32(buf), pol);
        else tma_store_2d(tmO, int(ocol0 + c0), int(grow0), smem_u32(buf));
        bulk_commit();
      }
    } else if (lane < nvr) {
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + (grow0 + lane) * p.ldo + ocol0 + c0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t(&pq)[8] = *reinterpret_cast<const uint32_t(*)[8]>(pk + 8 * q);
        if (p.out_keep) store_bf16x16_hint(out + 16 * q, pq, pol);
        else store_bf16x16(out + 16 * q, pq);
      }
    }
  }
}

// A warp's 32 rows x 32 bf16 columns (pk: this lane's row) at output column col: with all
// 32 rows valid, through a 64-byte-swizzled 2 KB box in shared memory (16-byte chunk q of
// row r at r * 64 + ((q ^ ((r >> 1) & 3)) << 4), conflict-free) and one TMA store, once the
// box's previous store has read it; else each valid row directly.
__device__ __forceinline__ void store_box32(const KParams& p, const CUtensorMap* tmO, uint8_t* buf,
                                            const uint32_t (&pk)[16], int64_t col, int64_t grow0,
                                            int nvr, int lane, uint64_t pol) {
  if (nvr == 32) {
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4*>(buf + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4)) =
          make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (p.out_keep) tma_store_2d_hint(tmO, int(col), int(grow0), smem_u32(buf), pol);
      else tma_store_2d(tmO, int(col), int(grow0), smem_u32(buf));
      bulk_commit();
    }
  } else if (lane < nvr) {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + (grow0 + lane) * p.ldo + col;
    const uint32_t(&p0)[8] = *reinterpret_cast<const uint32_t(*)[8]>(pk);
    const uint32_t(&p1)[8] = *reinterpret_cast<const uint32_t(*)[8]>(pk + 8);
    if (p.out_keep) {
      store_bf16x16_hint(out, p0, pol);
      store_bf16x16_hint(out + 16, p1, pol);
    } else {
      store_bf16x16(out, p0);
      store_bf16x16(out + 16, p1);
    }
  }
}

// The data-gradient epilogues of one warp (rows grow0 .., the first nvr valid; half or
// quarter `part` of the tile's columns), as epilogue_rows computes them, their bf16 output
// stored 32 columns at a time with store_box32.
//   EPI_DGRAD2: D = dy_perm . W_out (unscaled); out = w_r * D (ReLU: where h > 0), and the
//     gate partial sum_c D * h over the half (h as the forward stored it).
//   EPI_SWIGLU_BWD: D = (a | b), the tile's 128 gate and 128 up pre-activations; with dh:
//     da = dh * b * silu'(a), db = dh * silu(a), at the same interleaved columns.
template <int BN, int EPI>
__device__ __forceinline__ void epilogue_dgrad_tma(const KParams& p, const CUtensorMap* tmO,
                                                   uint32_t tbase, int64_t grow0, int nvr, int nt,
                                                   int part, uint8_t* buf, int lane) {
  const bool valid = lane < nvr;
  const int64_t grow = grow0 + lane;
  const uint64_t pol = p.out_keep ? policy_evict_last() : 0ull;
  if constexpr (EPI == EPI_DGRAD2) {
    constexpr int kHalf = BN / 2;
    const int cb = part * kHalf, ce = cb + kHalf;
    const float scale = (valid && p.row_scale) ? p.row_scale[grow] : 1.f;
    const __nv_bfloat16* hrow = static_cast<const __nv_bfloat16*>(p.aux) + grow * p.ld_aux + nt * BN;
    float gsum = 0.f;
    uint4 hn[4];  // h of the next 32 columns, loaded before this step's math
#pragma unroll
    for (int q = 0; q < 4; ++q)
      hn[q] = valid ? __ldg(reinterpret_cast<const uint4*>(hrow + cb) + q) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 1
    for (int c0 = cb; c0 < ce; c0 += 32) {
      uint4 hc[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) hc[q] = hn[q];
      if (valid && c0 + 32 < ce) {
#pragma unroll
        for (int q = 0; q < 4; ++q) hn[q] = __ldg(reinterpret_cast<const uint4*>(hrow + c0 + 32) + q);
      }
      uint32_t v[32];
      tmem_ld16(tbase + c0, *reinterpret_cast<uint32_t(*)[16]>(v));
      tmem_ld16(tbase + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
      tmem_ld_wait();
      const uint32_t* hw = reinterpret_cast<const uint32_t*>(hc);
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float2 hv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hw[j]));
        const float d0 = __uint_as_float(v[2 * j]), d1 = __uint_as_float(v[2 * j + 1]);
        gsum += d0 * hv.x + d1 * hv.y;
        float o0 = d0 * scale, o1 = d1 * scale;
        if (p.relu) {
          o0 = hv.x > 0.f ? o0 : 0.f;
          o1 = hv.y > 0.f ? o1 : 0.f;
        }
        pk[j] = pack_bf16x2(o0, o1);
      }
      store_box32(p, tmO, buf, pk, int64_t(nt) * BN + c0, grow0, nvr, lane, pol);
    }
    if (valid && p.gpart) p.gpart[(grow * p.n_tiles + nt) * 2 + part] = gsum;
  } else {
    constexpr int kQuarter = BN / 4;
    const int cb = part * kQuarter, ce = cb + kQuarter;
    const __nv_bfloat16* dhrow =
        static_cast<const __nv_bfloat16*>(p.aux) + grow * p.ld_aux + nt * (BN / 2);
    uint4 dn[4];  // the next 32 hidden units' dh, loaded before this step's math
#pragma unroll
    for (int q = 0; q < 4; ++q)
      dn[q] = valid ? __ldg(reinterpret_cast<const uint4*>(dhrow + cb) + q) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 1
    for (int c0 = cb; c0 < ce; c0 += 32) {
      uint4 dc[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) dc[q] = dn[q];
      if (valid && c0 + 32 < ce) {
#pragma unroll
        for (int q = 0; q < 4; ++q) dn[q] = __ldg(reinterpret_cast<const uint4*>(dhrow + c0 + 32) + q);
      }
      uint32_t av[32], bv[32];
      tmem_ld16(tbase + c0, *reinterpret_cast<uint32_t(*)[16]>(av));
      tmem_ld16(tbase + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(av + 16));
      tmem_ld16(tbase + BN / 2 + c0, *reinterpret_cast<uint32_t(*)[16]>(bv));
      tmem_ld16(tbase + BN / 2 + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(bv + 16));
      tmem_ld_wait();
      const uint32_t* dw = reinterpret_cast<const uint32_t*>(dc);
      uint32_t pa[16], pb[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float2 dh = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&dw[j]));
        float da[2], db[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float a = __uint_as_float(av[2 * j + q]), b = __uint_as_float(bv[2 * j + q]);
          const float sg = 1.f / (1.f + __expf(-a));
          const float d = q ? dh.y : dh.x;
          da[q] = d * b * sg * (1.f + a * (1.f - sg));
          db[q] = d * a * sg;
        }
        pa[j] = pack_bf16x2(da[0], da[1]);
        pb[j] = pack_bf16x2(db[0], db[1]);
      }
      store_box32(p, tmO, buf, pa, int64_t(nt) * BN + c0, grow0, nvr, lane, pol);
      store_box32(p, tmO, buf, pb, int64_t(nt) * BN + BN / 2 + c0, grow0, nvr, lane, pol);
    }
  }
}

// K-ragged mode's fp32 epilogue for one warp: rows grow0 .. grow0 + 31 (the first nvr valid),
// BOX (32 or 16) columns at a time: lanes write their row into a swizzled 32 x BOX staging
// buffer (128- or 64-byte swizzle, conflict-free), fence it for the async proxy, and lane 0
// stores it with one TMA tensor store (NBUF buffers in turn; a buffer is rewritten once the
// store that last read it has finished reading). A warp whose rows end inside it (the last
// rows of a one-group output) stores its valid rows from the buffer with plain stores
// instead.
template <int BN, int BOX, int NBUF>
__device__ __forceinline__ void epilogue_f32_tma(const KParams& p, const CUtensorMap* tmO,
                                                 const CUtensorMap* tmO2, uint32_t tbase,
                                                 int64_t grow0, int nvr, int nt, bool zero,
                                                 uint8_t* bufs, int lane, int& nb) {
  static_assert(BOX == 32 || BOX == 16, "fp32 staging boxes are 32 or 16 columns");
  constexpr int kRowBytes = BOX * 4;           // one staged row
  constexpr int kBufBytes = 32 * kRowBytes;
  constexpr int kLanesPerRow = BOX / 4;        // plain-store path: 16 bytes a lane
  // the 16-byte chunk c of row r sits at chunk c ^ (r & 7) (128-byte swizzle) or
  // c ^ ((r >> 1) & 3) (64-byte swizzle)
  auto chunk = [](int c, int r) { return BOX == 32 ? (c ^ (r & 7)) : (c ^ ((r >> 1) & 3)); };
  const CUtensorMap* map = tmO;
  int64_t orow = grow0;
  float* out0 = static_cast<float*>(p.out);
  if (p.out2) {  // interleaved SwiGLU rows: 128 to out, the next 128 to out2 (32-row aligned)
    const int64_t g = grow0 / p.c1, j = grow0 % p.c1, c = j & 255;
    orow = g * (p.c1 / 2) + (j >> 8) * 128 + (c & 127);
    if (c >= 128) {
      map = tmO2;
      out0 = static_cast<float*>(p.out2);
    }
  }
#pragma unroll 1
  for (int c0 = 0; c0 < BN; c0 += BOX) {
    uint32_t v[BOX];
    tmem_ld16(tbase + c0, *reinterpret_cast<uint32_t(*)[16]>(v));
    if constexpr (BOX == 32) tmem_ld16(tbase + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
    tmem_ld_wait();
    uint8_t* buf = bufs + nb * kBufBytes;
    if (lane == 0) bulk_wait_read<NBUF - 1>();
    __syncwarp();
#pragma unroll
    for (int c = 0; c < BOX / 4; ++c) {
      const float4 f = zero ? make_float4(0.f, 0.f, 0.f, 0.f)
                            : make_float4(__uint_as_float(v[4 * c]), __uint_as_float(v[4 * c + 1]),
                                          __uint_as_float(v[4 * c + 2]), __uint_as_float(v[4 * c + 3]));
      *reinterpret_cast<float4*>(buf + lane * kRowBytes + (chunk(c, lane) << 4)) = f;
    }
    fence_proxy_async_smem();
    __syncwarp();
    const int col = nt * BN + c0;
    if (lane == 0) {
      if (nvr == 32 && col < p.n_valid)  // weight gradients: not read back by this step
        tma_store_2d_hint(map, col, int(orow), smem_u32(buf), policy_evict_first());
      // one bulk group per box, empty when nothing was stored: the wait above counts
      // groups, so a buffer is rewritten only once the store that read it has (a chunk past
      // N or a warp of plain stores that committed nothing would let it overwrite a buffer
      // a TMA store is still reading)
      bulk_commit();
    }
    if (nvr < 32 && nvr > 0) {
      const int cl = (lane % kLanesPerRow) * 4;
#pragma unroll 1
      for (int pass = 0; pass < kLanesPerRow; ++pass) {
        const int rr = pass * (32 / kLanesPerRow) + lane / kLanesPerRow;
        if (rr < nvr && col + cl < p.n_valid) {
          const float* sv = reinterpret_cast<const float*>(buf + rr * kRowBytes + (chunk(cl >> 2, rr) << 4));
          float* out = out0 + (orow + rr) * p.ldo + col + cl;
          for (int i = 0; i < 4 && col + cl + i < p.n_valid; ++i) out[i] = sv[i];
        }
      }
    }
    __syncwarp();
    nb = nb + 1 == NBUF ? 0 : nb + 1;
  }
}

// Shared-memory descriptor of an MN-major operand staged as 64-column TMA boxes (128-byte
// rows, one K index a row, 128-byte swizzle): the swizzle atom is 8 K rows of 64 MN
// elements; atoms follow each other along K every 1024 bytes (stride offset) and along MN
// every 8 KB, the next box (leading offset).
__device__ __forceinline__ uint64_t mn_sw128_desc(uint32_t saddr) {
  uint64_t d = uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t(8192 >> 4) << 16;  // leading-dimension offset: next 64 MN elements
  d |= uint64_t(1024 >> 4) << 32;  // stride-dimension offset: next 8 K rows
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}

// ------------------------------------------------------------------ the kernel
template <int BN, int EPI, bool PAIR, bool KRAG, bool MN = false>
__global__ void __launch_bounds__(64 + 32 * epi_warps<EPI, KRAG>(), 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmO,   // K-ragged: fp32 output
                        const __grid_constant__ CUtensorMap tmO2,  // K-ragged: second output
                        const KParams p) {
  constexpr bool TEPI = tma_epilogue<EPI, KRAG>();
  using C = Cfg<BN, PAIR, KRAG, TEPI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::STAGES * C::A_BYTES;
  // output staging: K-ragged [4 warps][2][32 rows][128 B]; bf16 TMA epilogue [4 warps][32][128 B]
  uint8_t* sStg = sB + C::STAGES * C::B_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + C::STG_BYTES);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 2 * C::STAGES + 5);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  int* s_total = reinterpret_cast<int*>(s_tmem + 2);
  int* s_tstart = reinterpret_cast<int*>(s_tmem + 4);  // [groups+1] first m-tile of each group
  int* s_off = s_tstart + (kMaxGroups + 1);            // [groups+1] first row of each group
  int* s_koff = s_off + (kMaxGroups + 1);              // K-ragged: [groups+1] K offsets

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * C::STAGES;
  const uint32_t tfull0 = empty0 + 8 * C::STAGES;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain_bar = tempty0 + 16;
  const int G = (p.offsets || KRAG) ? p.groups : 1;
  const uint32_t rank = PAIR ? cluster_rank() : 0u;
  const bool leader = rank == 0;
  const int unit = PAIR ? int(blockIdx.x >> 1) : int(blockIdx.x);  // this CTA's tile stream
  const int units = PAIR ? int(gridDim.x >> 1) : int(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, epi_warps<EPI, KRAG>() * C::CTAS);
    }
    mbar_init(drain_bar, 1);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
  }
  if (warp == 1) {
    if constexpr (PAIR) tmem_alloc_pair(smem_u32(s_tmem), C::TMEM_COLS);
    else tmem_alloc(smem_u32(s_tmem), C::TMEM_COLS);
  }
  if (p.pfB && threadIdx.x == 0 && leader) {
    // The weights do not depend on the previous kernel: bring the first k-blocks of this
    // unit's first B tile into L2 while that kernel finishes. The tile is a guess (one
    // m-tile per group when the rows are grouped), so it may be the wrong one, never one
    // outside B.
    const int mt = p.offsets ? 1 : (p.rows_dense + C::TILE_M - 1) / C::TILE_M;
    const int ut = (p.offsets && p.reverse) ? G * p.n_tiles - 1 - unit : unit;
    const int g = p.offsets ? ut / p.n_tiles : 0;
    const int nt = p.offsets ? ut % p.n_tiles : unit / (mt > 0 ? mt : 1);
    if (ut >= 0 && g < G && nt < p.n_tiles) {  // (reversed: no guess past the first tile)
      const int64_t kb_bytes = int64_t(BN) * BK * 2;
      const int64_t tile_bytes = int64_t(p.K / BK) * kb_bytes;
      const char* base = p.pfB + (int64_t(g) * p.n_tiles + nt) * tile_bytes;
      const int64_t n = p.pf_bytes < tile_bytes ? p.pf_bytes : tile_bytes;
      for (int64_t o = 0; o + 16 <= n; o += 65536)
        prefetch_l2_bulk(base + o, uint32_t(n - o < 65536 ? (n - o) & ~int64_t(15) : 65536));
    }
  }
  pdl_wait();  // everything above is local setup; below, the first reads of the inputs
  pdl_trigger();
  const uint64_t wlimit = wait_limit_ns(p.status);
  if (warp == 2) {
    // m-tile prefix over the groups, from the device row offsets
    bool bad = false;
    int run = 0;
    for (int base = 0; base < G; base += 32) {
      const int g = base + lane;
      int cnt = 0;
      if (g < G) {
        int lo, hi;
        if constexpr (KRAG) {  // c1 output rows per group; K range from koffs
          lo = g * p.c1;
          hi = lo + p.c1;
          const int k0 = p.koffs[g], k1 = p.koffs[g + 1];
          if (k0 < 0 || k1 < k0 || k1 > p.K || (k0 | k1) % BK) bad = true;
          s_koff[g] = k0;
          if (g == G - 1) s_koff[G] = k1;
        } else {
          lo = p.offsets ? p.offsets[g] : 0;
          hi = p.offsets ? p.offsets[g + 1] : p.rows_dense;
        }
        if (lo < 0 || hi < lo || int64_t(hi) > p.rows_cap) bad = true;
        else cnt = (hi - lo + C::TILE_M - 1) / C::TILE_M;
        s_off[g] = lo;
        if (g == G - 1) s_off[G] = hi;
      }
      int v = cnt;
      for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += n;
      }
      if (g < G) s_tstart[g + 1] = run + v;
      run += __shfl_sync(0xffffffffu, v, 31);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      s_tstart[0] = 0;
      *s_total = bad ? 0 : run * p.n_tiles;
      if (bad && leader) atomicOr(p.status, kStatusDeviceData);
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync_all();  // barriers initialised in both CTAs
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int total = *s_total;
  const int kblocks = p.K / BK;

  // tile t -> group g, first row m0, valid rows, n tile
  auto decode = [&](int t, int& g, int& m0, int& rows, int& nt) {
    if (p.reverse) t = total - 1 - t;
    int lo = 0, hi = G;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_tstart[mid] * p.n_tiles <= t) lo = mid;
      else hi = mid;
    }
    g = lo;
    const int local = t - s_tstart[g] * p.n_tiles;
    const int mt = s_tstart[g + 1] - s_tstart[g];
    nt = local / mt;
    const int m_t = local % mt;
    m0 = s_off[g] + m_t * C::TILE_M;
    rows = min(C::TILE_M, s_off[g + 1] - m0);
  };

  // what each role has in flight, for the drain after an abort: the stages whose last load
  // the producer issued (and that load's phase), whether the MMA thread issued MMAs and
  // has already waited for them
  uint32_t issued = 0, issued_par = 0;
  bool mma_any = false, mma_drained = false;
  if (warp == 0) {
    // ---------------- TMA producer: the whole warp walks the schedule, lane 0 issues
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = unit; t < total && ok; t += units) {
      int g, m0, rows, nt;
      decode(t, g, m0, rows, nt);
      const int arow = m0 - (KRAG ? g * p.c1 : 0) + int(rank) * BM;
      const int brow = (KRAG ? 0 : g * p.N) + nt * BN + int(rank) * C::B_ROWS;
      const int bblk = (g * p.n_tiles + nt) * kblocks;
      const int kb0 = KRAG ? s_koff[g] / BK : 0;
      const int nkb = KRAG ? s_koff[g + 1] / BK - kb0 : kblocks;
      const int abase = MN ? (p.aoffs ? __ldg(p.aoffs + g) : s_koff[g]) : 0;  // K rows of A
      const int bbase = MN ? (p.boffs ? __ldg(p.boffs + g) : s_koff[g]) : 0;  // K rows of B
      for (int kb = 0; kb < nkb; ++kb) {
        ok = __all_sync(0xffffffffu, wait_bounded(empty0 + 8 * stage, phase ^ 1u, s_abort, p.status, wlimit));
        if (!ok) break;
        if (lane == 0) {
          const uint32_t fb = full0 + 8 * stage;
          const uint32_t dA = smem_u32(sA + stage * C::A_BYTES);
          const uint32_t dB = smem_u32(sB + stage * C::B_BYTES);
          if (leader) mbar_expect_tx(fb, C::CTAS * C::STAGE_BYTES);
          if constexpr (MN) {
            // 64 K rows x 64 columns a box: A's columns arow .. (this CTA's output rows), B's
            // columns brow .. ; the boxes of a stage sit 8 KB apart
            const int ya = abase + kb * BK, yb = bbase + kb * BK;
            const uint32_t bar = PAIR ? cluster_addr(fb, 0) : fb;
#pragma unroll
            for (int i = 0; i < BM / 64; ++i) {
              if constexpr (PAIR) tma_load_2d_pair(dA + i * 8192, &tmA, arow + 64 * i, ya, bar);
              else tma_load_2d(dA + i * 8192, &tmA, arow + 64 * i, ya, bar);
            }
#pragma unroll
            for (int i = 0; i < C::B_ROWS / 64; ++i) {
              if constexpr (PAIR) tma_load_2d_pair(dB + i * 8192, &tmB, brow + 64 * i, yb, bar);
              else tma_load_2d(dB + i * 8192, &tmB, brow + 64 * i, yb, bar);
            }
          } else if constexpr (PAIR) {
            const uint32_t lfb = cluster_addr(fb, 0);  // the even CTA's full barrier
            tma_load_2d_pair(dA, &tmA, (kb0 + kb) * BK, arow, lfb);
            if (p.b_tiled) tma_load_3d_pair(dB, &tmB, 0, int(rank) * C::B_ROWS, bblk + kb, lfb);
            else tma_load_2d_pair(dB, &tmB, (kb0 + kb) * BK, brow, lfb);
          } else {
            tma_load_2d(dA, &tmA, (kb0 + kb) * BK, arow, fb);
            if (p.b_tiled) tma_load_3d(dB, &tmB, 0, 0, bblk + kb, fb);
            else tma_load_2d(dB, &tmB, (kb0 + kb) * BK, brow, fb);
          }
        }
        __syncwarp();
        issued |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer (the even CTA of a pair): the warp waits, lane 0 issues
    if (leader) {
      // MN-major operands: bits 15 and 16 of the instruction descriptor
      constexpr uint32_t kIdesc = idesc_bf16(C::TILE_M, BN) | (MN ? (3u << 15) : 0u);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int i = 0;
      for (int t = unit; t < total && ok; t += units, ++i) {
        const int acc = i & 1;
        const uint32_t use = uint32_t(i >> 1) & 1u;
        ok = __all_sync(0xffffffffu, wait_bounded(tempty0 + 8 * acc, use ^ 1u, s_abort, p.status, wlimit));
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem_base + uint32_t(acc * BN);
        int nkb = kblocks;
        if constexpr (KRAG) {
          int g, m0, rows, nt;
          decode(t, g, m0, rows, nt);
          nkb = (s_koff[g + 1] - s_koff[g]) / BK;
        }
        for (int kb = 0; kb < nkb; ++kb) {
          ok = __all_sync(0xffffffffu, wait_bounded(full0 + 8 * stage, phase, s_abort, p.status, wlimit));
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t a0 = smem_u32(sA + stage * C::A_BYTES);
            const uint32_t b0 = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              // K-major: a K step of 16 is 32 bytes along the swizzled row; MN-major: 16
              // K rows of 128 bytes
              const uint64_t ad = MN ? mn_sw128_desc(a0 + kk * 2048) : sw128_desc(a0 + kk * 32);
              const uint64_t bd = MN ? mn_sw128_desc(b0 + kk * 2048) : sw128_desc(b0 + kk * 32);
              if constexpr (PAIR) mma_bf16_pair(d, ad, bd, kIdesc, (kb | kk) != 0 ? 1u : 0u);
              else mma_bf16(d, ad, bd, kIdesc, (kb | kk) != 0 ? 1u : 0u);
            }
            if constexpr (PAIR) mma_commit_pair(empty0 + 8 * stage, uint16_t(3));
            else mma_commit(empty0 + 8 * stage);
          }
          __syncwarp();
          mma_any = true;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok && lane == 0) {
          if constexpr (PAIR) mma_commit_pair(tfull0 + 8 * acc, uint16_t(3));
          else mma_commit(tfull0 + 8 * acc);
        }
        __syncwarp();
      }
      if (!ok && mma_any && lane == 0) {  // every MMA issued must finish before TMEM is freed
        if constexpr (PAIR) mma_commit_pair(drain_bar, uint16_t(1));
        else mma_commit(drain_bar);
        wait_drain(drain_bar, 0u);
      }
      mma_drained = !ok && mma_any;
      __syncwarp();
    }
  } else {
    // ---------------- epilogue warps 2 .. 1 + epi_warps
    const int q = warp & 3;  // TMEM lanes 32q..32q+31 = this CTA's tile rows
    const int part = (warp - 2) >> 2;  // eight epilogue warps: the half of the columns
    const uint32_t tempty_leader = PAIR ? cluster_addr(tempty0, 0) : tempty0;
    int stg_buf = 0;  // K-ragged: the staging buffer the next 32 columns go to
    int i = 0;
    for (int t = unit; t < total; t += units, ++i) {
      const int acc = i & 1;
      const uint32_t use = uint32_t(i >> 1) & 1u;
      int g, m0, rows, nt;
      decode(t, g, m0, rows, nt);
      if constexpr (EPI == EPI_DGRAD2 || EPI == EPI_SWIGLU_BWD) {
        // the tile's h (dh) row segment of this lane: into L2 while the MMAs run
        const int r = int(rank) * BM + q * 32 + lane;
        constexpr int kAuxCols = EPI == EPI_DGRAD2 ? BN : BN / 2;
        if (r < rows)
          prefetch_l2_bulk(static_cast<const __nv_bfloat16*>(p.aux) + (int64_t(m0) + r) * p.ld_aux +
                               int64_t(nt) * kAuxCols,
                           uint32_t(kAuxCols * 2));
      }
      const bool ok = __all_sync(0xffffffffu, wait_bounded(tfull0 + 8 * acc, use, s_abort, p.status, wlimit));
      if (!ok) break;
      tc_fence_after();
      const int r = int(rank) * BM + q * 32 + lane;  // row within the tile
      const uint32_t tbase = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(acc * BN);
      const bool zero = KRAG && s_koff[g + 1] == s_koff[g];  // no MMA ran for this tile
      if constexpr (KRAG && EPI == EPI_F32_BIAS) {
        const int r0 = int(rank) * BM + q * 32;  // this warp's first row in the tile
        const int nvr = rows - r0 < 0 ? 0 : (rows - r0 > 32 ? 32 : rows - r0);
        epilogue_f32_tma<BN, C::F32_BOX, C::F32_BUFS>(p, &tmO, &tmO2, tbase, int64_t(m0) + r0, nvr,
                                                      nt, zero, sStg + q * (C::STG_BYTES / 4),
                                                      lane, stg_buf);
      } else if constexpr (TEPI && tma_box32<EPI>()) {
        const int r0 = int(rank) * BM + q * 32;
        const int nvr = rows - r0 < 0 ? 0 : (rows - r0 > 32 ? 32 : rows - r0);
        epilogue_dgrad_tma<BN, EPI>(p, &tmO, tbase, int64_t(m0) + r0, nvr, nt, part,
                                    sStg + (warp - 2) * 2048, lane);
      } else if constexpr (TEPI) {
        const int r0 = int(rank) * BM + q * 32;
        const int nvr = rows - r0 < 0 ? 0 : (rows - r0 > 32 ? 32 : rows - r0);
        epilogue_bf16_tma<BN, EPI>(p, &tmO, tbase, int64_t(m0) + r0, nvr, nt, sStg + q * 4096,
                                   lane);
      } else {
        epilogue_rows<BN, EPI>(p, tbase, r < rows, int64_t(m0) + r, nt, zero, part);
      }
      // the accumulator is free: every lane has waited for its tensor-memory loads
      // (tcgen05.wait::ld); a relaxed arrive, as nothing of the stores needs ordering here
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (PAIR) mbar_arrive_cluster_relaxed(tempty_leader + 8 * acc);
        else mbar_arrive_relaxed(tempty0 + 8 * acc);
      }
    }
    // every TMA store has finished before the CTA's shared memory goes away
    if constexpr ((KRAG && EPI == EPI_F32_BIAS) || TEPI)
      if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (*s_abort) {
    // A role may have finished its own loop before another gave up, with loads or MMAs still
    // in flight: every load issued lands (the even CTA's full barriers also count the odd
    // CTA's bytes) and every MMA issued finishes before shared and tensor memory go away.
    // The flag is read after the barrier, so every thread of the CTA takes this branch.
    if (warp == 0 && leader && lane == 0) {
      for (int s = 0; s < C::STAGES; ++s)
        if ((issued >> s) & 1u) wait_drain(full0 + 8 * s, (issued_par >> s) & 1u);
    }
    if (warp == 1 && leader && lane == 0 && mma_any && !mma_drained) {
      if constexpr (PAIR) mma_commit_pair(drain_bar, uint16_t(1));
      else mma_commit(drain_bar);
      wait_drain(drain_bar, 0u);
    }
    tc_fence_before();
    __syncthreads();
  }
  if constexpr (PAIR) cluster_sync_all();  // both CTAs done with TMEM and each other's smem
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ short-K weight gradients
// K-ragged, MN-major weight gradients (dW[g] = A_g^T . B_g over group g's K rows) when every
// group's K range is at most kResKB k-blocks: the GShard grouped layer's experts, whose rows
// are at most (groups x capacity) = 256. A tile (128 output rows x 256 columns) then takes
// only 4 k-blocks, and the tiles of one (group, N tile) all read the same 256 columns of B.
// The work goes in runs: (group, chunk of kRunM m-tiles, N tile), N tile innermost, the CTAs
// taking runs grid-strided, so that the runs in flight at one time share their A rows and
// the B of their group through L2. A CTA keeps its run's B k-blocks resident in kResKB fixed
// slots (32 KB each), loaded once per run, while A streams through its own ring. Such a
// GEMM is bound by its fp32 epilogue, which stores at about the rate HBM absorbs writes
// from every SM; what the B reuse buys is an MMA that keeps the accumulators ready.
// Measured on the GShard grouped layer's backward (two such GEMMs, 2.15 GB of fp32 each):
// runs of 2 m-tiles 1.387 ms, of 1, 3, 4 or 8: 1.474, 1.437, 1.437, 1.437 ms, against
// 1.428 ms for the streamed-B kernel (longer runs leave the CTAs' last runs uneven). Roles as in grouped_gemm_kernel: warp 0 the
// TMA producer, warp 1 the MMA issuer (two TMEM accumulators), warps 2..5 the fp32 TMA-store
// epilogue. Slot kb's barriers: b_full completes once per run that loads it, b_empty once
// per run that used it (the MMA thread commits it after the run's last tile), so neither
// can run two phases ahead of its waiter.
constexpr int kResKB = 4;
constexpr int kRunM = 2;  // m-tiles a run (the group's last may hold one)

struct ResCfg {
  static constexpr int BN = 256;
  static constexpr int A_BYTES = BM * BK * 2;  // 64 K rows x 128 output rows: two 64-column boxes
  static constexpr int B_BYTES = BN * BK * 2;  // 64 K rows x 256 columns: four boxes
  static constexpr int STG_BYTES = 4 * 2 * 4096;                  // fp32 staging, 32 x 32 boxes
  static constexpr int NBARS = 2 * 8 + 2 * kResKB + 5;            // A ring, B slots, TMEM, drain
  static constexpr int TABLE_BYTES = (kMaxGroups + 1) * 4;        // K offsets
  static constexpr int FIXED = 1024 + NBARS * 8 + 16 + TABLE_BYTES;
  static constexpr int A_RAW = (232448 - FIXED - kResKB * B_BYTES - STG_BYTES) / A_BYTES;
  static constexpr int A_STAGES = A_RAW > 8 ? 8 : A_RAW;
  static constexpr int SMEM = FIXED + kResKB * B_BYTES + A_STAGES * A_BYTES + STG_BYTES;
};
static_assert(ResCfg::A_STAGES >= 2, "the A ring needs two stages");

__global__ void __launch_bounds__(192, 1)
    wgrad_resident_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmO,
                          const __grid_constant__ CUtensorMap tmO2, const KParams p) {
  using R = ResCfg;
  constexpr int BN = R::BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sB = smem;                             // [kResKB] resident B k-blocks
  uint8_t* sA = sB + kResKB * R::B_BYTES;         // [A_STAGES] A ring
  uint8_t* sStg = sA + R::A_STAGES * R::A_BYTES;  // [4 warps][2][32 rows][128 B]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + R::STG_BYTES);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + R::NBARS);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  int* s_total = reinterpret_cast<int*>(s_tmem + 2);
  int* s_koff = reinterpret_cast<int*>(s_tmem + 4);  // [groups + 1]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t afull0 = smem_u32(bars), aempty0 = afull0 + 8 * 8;
  const uint32_t bfull0 = aempty0 + 8 * 8, bempty0 = bfull0 + 8 * kResKB;
  const uint32_t tfull0 = bempty0 + 8 * kResKB, tempty0 = tfull0 + 16, drain_bar = tempty0 + 16;
  const int G = p.groups;

  if (threadIdx.x == 0) {
    for (int s = 0; s < R::A_STAGES; ++s) {
      mbar_init(afull0 + 8 * s, 1);
      mbar_init(aempty0 + 8 * s, 1);
    }
    for (int kb = 0; kb < kResKB; ++kb) {
      mbar_init(bfull0 + 8 * kb, 1);
      mbar_init(bempty0 + 8 * kb, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 4);
    }
    mbar_init(drain_bar, 1);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
  }
  if (warp == 1) tmem_alloc(smem_u32(s_tmem), 2 * BN);
  pdl_wait();  // everything above is local setup; below, the first reads of the inputs
  pdl_trigger();
  const uint64_t wlimit = wait_limit_ns(p.status);
  const int mt = (p.c1 + BM - 1) / BM;  // m tiles a group
  const int n_mc = (mt + kRunM - 1) / kRunM;  // m-tile chunks a group
  if (warp == 2) {
    // the groups' K offsets: multiples of 64, in order, each range at most kResKB k-blocks
    bool bad = false;
    for (int g = lane; g <= G; g += 32) {
      const int k = p.koffs[g];
      s_koff[g] = k;
      if (k < 0 || k > p.K || k % BK) bad = true;
      if (g > 0) {
        const int kp = p.koffs[g - 1];
        if (k < kp || k - kp > kResKB * BK) bad = true;
      }
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      *s_total = bad ? 0 : G * n_mc * p.n_tiles;  // runs
      if (bad) atomicOr(p.status, kStatusDeviceData);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int n_runs = *s_total;
  // run r -> group g, N tile nt, m-tiles mb .. me - 1 of the group
  auto run_of = [&](int r, int& g, int& nt, int& mb, int& me) {
    const int per_g = n_mc * p.n_tiles;
    g = r / per_g;
    const int local = r - g * per_g;
    const int mc = local / p.n_tiles;
    nt = local - mc * p.n_tiles;
    mb = mc * kRunM;
    me = min(mt, mb + kRunM);
  };

  // in flight, for the drain after an abort: the producer's last load into each A stage and
  // each B slot (and the phase it completes); whether the MMA thread issued MMAs
  uint32_t a_issued = 0, a_par = 0, b_issued = 0, b_par = 0;
  bool mma_any = false, mma_drained = false;
  if (warp == 0) {
    // ---------------- TMA producer
    int stage = 0;
    uint32_t phase = 0;
    int uses[kResKB] = {};  // runs that have loaded slot kb
    bool ok = true;
    for (int r = blockIdx.x; r < n_runs && ok; r += gridDim.x) {
      int g, nt, mb, me;
      run_of(r, g, nt, mb, me);
      const int k0 = s_koff[g], nkb = (s_koff[g + 1] - k0) / BK;
      const int abase = p.aoffs ? __ldg(p.aoffs + g) : k0;  // K rows of A
      const int bbase = p.boffs ? __ldg(p.boffs + g) : k0;  // K rows of B
      {  // the run's B k-blocks into the slots
#pragma unroll
        for (int kb = 0; kb < kResKB; ++kb) {
          if (kb >= nkb || !ok) break;
          if (uses[kb] > 0)  // the slot's last run has finished its MMAs
            ok = __all_sync(0xffffffffu, wait_bounded(bempty0 + 8 * kb, uint32_t(uses[kb] - 1) & 1u,
                                                      s_abort, p.status, wlimit));
          if (!ok) break;
          if (lane == 0) {
            const uint32_t fb = bfull0 + 8 * kb;
            const uint32_t dB = smem_u32(sB + kb * R::B_BYTES);
            mbar_expect_tx(fb, R::B_BYTES);
#pragma unroll
            for (int i = 0; i < BN / 64; ++i)
              tma_load_2d(dB + i * 8192, &tmB, nt * BN + 64 * i, bbase + kb * BK, fb);
          }
          __syncwarp();
          b_issued |= 1u << kb;
          b_par = (b_par & ~(1u << kb)) | ((uint32_t(uses[kb]) & 1u) << kb);
          ++uses[kb];
        }
      }
      for (int mi = mb; mi < me && ok; ++mi) {
        const int acol = mi * BM;  // A's columns: the tile's output rows within the group
        for (int kb = 0; kb < nkb && ok; ++kb) {
          ok = __all_sync(0xffffffffu, wait_bounded(aempty0 + 8 * stage, phase ^ 1u, s_abort, p.status, wlimit));
          if (!ok) break;
          if (lane == 0) {
            const uint32_t fb = afull0 + 8 * stage;
            const uint32_t dA = smem_u32(sA + stage * R::A_BYTES);
            mbar_expect_tx(fb, R::A_BYTES);
#pragma unroll
            for (int i = 0; i < BM / 64; ++i)
              tma_load_2d(dA + i * 8192, &tmA, acol + 64 * i, abase + kb * BK, fb);
          }
          __syncwarp();
          a_issued |= 1u << stage;
          a_par = (a_par & ~(1u << stage)) | (phase << stage);
          if (++stage == R::A_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer
    constexpr uint32_t kIdesc = idesc_bf16(BM, BN) | (3u << 15);  // MN-major A and B
    int stage = 0;
    uint32_t phase = 0;
    int uses[kResKB] = {};  // runs whose B this thread has waited for, per slot
    bool ok = true;
    int i = 0;
    for (int r = blockIdx.x; r < n_runs && ok; r += gridDim.x) {
      int g, nt, mb, me;
      run_of(r, g, nt, mb, me);
      const int nkb = (s_koff[g + 1] - s_koff[g]) / BK;
      for (int mi = mb; mi < me && ok; ++mi, ++i) {
        const bool first = mi == mb;     // the run's first tile: wait for its B
        const bool last = mi == me - 1;  // the run's last tile: release its B slots after the MMAs
        const int acc = i & 1;
        const uint32_t use = uint32_t(i >> 1) & 1u;
        ok = __all_sync(0xffffffffu, wait_bounded(tempty0 + 8 * acc, use ^ 1u, s_abort, p.status, wlimit));
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem_base + uint32_t(acc * BN);
#pragma unroll
        for (int kb = 0; kb < kResKB; ++kb) {
          if (kb >= nkb) break;
          if (first) {
            ok = __all_sync(0xffffffffu, wait_bounded(bfull0 + 8 * kb, uint32_t(uses[kb]) & 1u, s_abort,
                                                      p.status, wlimit));
            if (!ok) break;
            ++uses[kb];
          }
          ok = __all_sync(0xffffffffu, wait_bounded(afull0 + 8 * stage, phase, s_abort, p.status, wlimit));
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t a0 = smem_u32(sA + stage * R::A_BYTES);
            const uint32_t b0 = smem_u32(sB + kb * R::B_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              mma_bf16(d, mn_sw128_desc(a0 + kk * 2048), mn_sw128_desc(b0 + kk * 2048), kIdesc,
                       (kb | kk) != 0 ? 1u : 0u);
            mma_commit(aempty0 + 8 * stage);
            if (last) mma_commit(bempty0 + 8 * kb);
          }
          __syncwarp();
          mma_any = true;
          if (++stage == R::A_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok && lane == 0) mma_commit(tfull0 + 8 * acc);
        __syncwarp();
      }
    }
    if (!ok && mma_any && lane == 0) {  // every MMA issued must finish before TMEM is freed
      mma_commit(drain_bar);
      wait_drain(drain_bar, 0u);
    }
    mma_drained = !ok && mma_any;
    __syncwarp();
  } else {
    // ---------------- epilogue warps 2 .. 5: TMEM lanes 32q .. 32q + 31
    const int q = warp & 3;
    int stg_buf = 0;
    int i = 0;
    bool ok = true;
    for (int r = blockIdx.x; r < n_runs && ok; r += gridDim.x) {
      int g, nt, mb, me;
      run_of(r, g, nt, mb, me);
      for (int mi = mb; mi < me; ++mi, ++i) {
        const int m0 = g * p.c1 + mi * BM;
        const int rows = min(BM, p.c1 - mi * BM);
        const int acc = i & 1;
        const uint32_t use = uint32_t(i >> 1) & 1u;
        ok = __all_sync(0xffffffffu, wait_bounded(tfull0 + 8 * acc, use, s_abort, p.status, wlimit));
        if (!ok) break;
        tc_fence_after();
        const uint32_t tbase = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(acc * BN);
        const bool zero = s_koff[g + 1] == s_koff[g];  // no MMA ran for this tile
        const int r0 = q * 32;
        const int nvr = rows - r0 < 0 ? 0 : (rows - r0 > 32 ? 32 : rows - r0);
        epilogue_f32_tma<BN, 32, 2>(p, &tmO, &tmO2, tbase, int64_t(m0) + r0, nvr, nt, zero,
                                    sStg + q * 2 * 4096, lane, stg_buf);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_relaxed(tempty0 + 8 * acc);
      }
    }
    if (lane == 0) bulk_wait_all();  // every TMA store has read its staging buffer
  }

  tc_fence_before();
  __syncthreads();
  if (*s_abort) {
    // whichever role gave up, every load issued lands and every MMA issued finishes before
    // shared and tensor memory are released
    if (warp == 0 && lane == 0) {
      for (int s = 0; s < R::A_STAGES; ++s)
        if ((a_issued >> s) & 1u) wait_drain(afull0 + 8 * s, (a_par >> s) & 1u);
      for (int kb = 0; kb < kResKB; ++kb)
        if ((b_issued >> kb) & 1u) wait_drain(bfull0 + 8 * kb, (b_par >> kb) & 1u);
    }
    if (warp == 1 && lane == 0 && mma_any && !mma_drained) {
      mma_commit(drain_bar);
      wait_drain(drain_bar, 0u);
    }
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * BN);
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D bf16 tensor map over a row-major [rows, K] matrix; box = 64 columns x box_rows rows.
int make_map(CUtensorMap* m, const void* base, int64_t rows, int K, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return MOE_ERR_CUDA;
  if (reinterpret_cast<uintptr_t>(base) % 16 != 0) return MOE_ERR_INVALID_ARG;
  cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(K) * 2};
  cuuint32_t box[2] = {cuuint32_t(BK), cuuint32_t(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// 2-D fp32 tensor map over a row-major [rows, N] output, boxes of 32 rows x box_cols columns:
// 32 with the 128-byte swizzle, 16 with the 64-byte one (the K-ragged epilogue's TMA stores).
int make_map_f32_out(CUtensorMap* m, void* base, int64_t rows, int N, int box_cols) {
  auto fn = encode_fn();
  if (!fn) return MOE_ERR_CUDA;
  if (reinterpret_cast<uintptr_t>(base) % 16 != 0 || (int64_t(N) * 4) % 16 != 0) return MOE_ERR_INVALID_ARG;
  cuuint64_t dims[2] = {cuuint64_t(N), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(N) * 4};
  cuuint32_t box[2] = {cuuint32_t(box_cols), 32};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// 2-D bf16 tensor map over a row-major [rows, cols] output with row stride ld elements,
// boxes of 32 rows x box_cols columns: 64 with the 128-byte swizzle, 32 with the 64-byte
// swizzle (the bf16 TMA epilogues' stores).
int make_map_bf16_out(CUtensorMap* m, void* base, int64_t rows, int cols, int64_t ld, int box_cols) {
  auto fn = encode_fn();
  if (!fn) return MOE_ERR_CUDA;
  if (reinterpret_cast<uintptr_t>(base) % 16 != 0 || (ld * 2) % 16 != 0 || cols < box_cols ||
      ld < cols || rows < 1 || (box_cols != 64 && box_cols != 32))
    return MOE_ERR_INVALID_ARG;
  cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(ld) * 2};
  cuuint32_t box[2] = {cuuint32_t(box_cols), 32};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// 3-D bf16 tensor map over a tile-major packed matrix: `blocks` contiguous [block_rows][64]
// blocks; a box is box_rows rows (all of a block, or half of it for a CTA pair).
int make_map_tiled(CUtensorMap* m, const void* base, int64_t blocks, int block_rows, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return MOE_ERR_CUDA;
  if (reinterpret_cast<uintptr_t>(base) % 16 != 0) return MOE_ERR_INVALID_ARG;
  cuuint64_t dims[3] = {cuuint64_t(BK), cuuint64_t(block_rows), cuuint64_t(blocks)};
  cuuint64_t strides[2] = {cuuint64_t(BK) * 2, cuuint64_t(BK) * 2 * block_rows};
  cuuint32_t box[3] = {cuuint32_t(BK), cuuint32_t(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

template <int BN, int EPI, bool PAIR, bool KRAG = false, bool MN = false>
int run_gemm(const GemmDesc& d, cudaStream_t st) {
  constexpr bool TEPI = tma_epilogue<EPI, KRAG>();
  using C = Cfg<BN, PAIR, KRAG, TEPI>;
  CUtensorMap ta, tb;
  if (KRAG && (!d.koffs || d.c1 < 1 || d.b_tiled || d.groups < 1)) return MOE_ERR_INVALID_ARG;
  int rc;
  if constexpr (MN) {  // row-major [K rows, c1] and [K rows, N]; 64 x 64 boxes
    if (d.c1 % 64 || d.N % 8 || d.a_krows < 1 || d.b_krows < 1) return MOE_ERR_UNSUPPORTED;
    if ((rc = make_map(&ta, d.A, d.a_krows, d.c1, 64)) != MOE_OK) return rc;
    rc = make_map(&tb, d.B, d.b_krows, d.N, 64);
  } else {
    rc = make_map(&ta, d.A, KRAG ? d.c1 : d.a_rows, d.K, BM);
    if (rc != MOE_OK) return rc;
    if (d.b_tiled) {
    if (d.N % BN != 0 || d.b_rows % d.N != 0) return MOE_ERR_UNSUPPORTED;
    rc = make_map_tiled(&tb, d.B, d.b_rows / BN * (d.K / BK), BN, C::B_ROWS);
    } else {  // row-major B: a pair's CTAs each load their half of the BN rows
      if (PAIR && !KRAG) return MOE_ERR_UNSUPPORTED;
      rc = make_map(&tb, d.B, d.b_rows, d.K, C::B_ROWS);
    }
  }
  if (rc != MOE_OK) return rc;
  CUtensorMap to, to2;  // K-ragged: the fp32 outputs, 32 x 32 boxes, 128-byte swizzle
  memset(&to, 0, sizeof(to));
  memset(&to2, 0, sizeof(to2));
  if constexpr (KRAG) {
    if (d.epi != EPI_F32_BIAS || d.ldo != d.N) return MOE_ERR_UNSUPPORTED;
    const int64_t out_rows = int64_t(d.groups) * d.c1 / (d.out2 ? 2 : 1);
    if ((rc = make_map_f32_out(&to, d.out, out_rows, d.N, C::F32_BOX)) != MOE_OK) return rc;
    if (d.out2 && (rc = make_map_f32_out(&to2, d.out2, out_rows, d.N, C::F32_BOX)) != MOE_OK)
      return rc;
  }
  if constexpr (TEPI) {  // the bf16 output [rows, columns] (row stride ldo)
    const int64_t out_rows = d.offsets ? d.a_rows : int64_t(d.rows_dense);
    const int out_cols = EPI == EPI_SWIGLU ? d.N / 2 : d.N;
    if ((rc = make_map_bf16_out(&to, d.out, out_rows, out_cols, d.ldo, tma_box32<EPI>() ? 32 : 64)) !=
        MOE_OK)
      return rc;
  }
  KParams p;
  p.b_tiled = d.b_tiled ? 1 : 0;
  p.offsets = d.offsets;
  p.groups = d.groups;
  p.rows_dense = d.rows_dense;
  p.rows_cap = KRAG ? int64_t(d.groups) * d.c1 : d.a_rows;
  p.N = d.N;
  p.K = d.K;
  p.n_tiles = (d.N + BN - 1) / BN;
  p.out = d.out;
  p.ldo = d.ldo;
  p.row_scale = d.row_scale;
  p.bias = d.bias;
  p.n_valid = d.n_valid;
  p.status = d.status;
  p.aux = d.aux;
  p.ld_aux = d.ld_aux;
  p.gpart = d.gpart;
  p.relu = d.relu;
  p.koffs = d.koffs;
  p.c1 = d.c1;
  p.out2 = d.out2;
  p.pfB = (!KRAG && d.b_tiled) ? static_cast<const char*>(d.B) : nullptr;
  p.pf_bytes = int64_t(512) << 10;
  p.aoffs = d.aoffs;
  p.boffs = d.boffs;
  p.reverse = (d.reverse && d.offsets && !KRAG) ? 1 : 0;
  p.out_keep = (d.out_keep && d.offsets && !KRAG && d.a_rows <= int64_t(d.groups) * C::TILE_M) ? 1 : 0;
  auto kern = grouped_gemm_kernel<BN, EPI, PAIR, KRAG, MN>;
  MOE_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM));
  const int64_t m_tiles =
      KRAG ? int64_t(d.groups) * ((d.c1 + C::TILE_M - 1) / C::TILE_M)
           : d.offsets ? (d.a_rows + C::TILE_M - 1) / C::TILE_M + d.groups
                       : (int64_t(d.rows_dense) + C::TILE_M - 1) / C::TILE_M;
  const int64_t tiles = m_tiles * p.n_tiles;
  cudaLaunchConfig_t lc = {};
  lc.blockDim = dim3(64 + 32 * epi_warps<EPI, KRAG>());
  lc.dynamicSmemBytes = C::SMEM;
  lc.stream = st;
  cudaLaunchAttribute attr[2];
  int64_t units = num_sms();
  if constexpr (PAIR) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    lc.gridDim = dim3(2);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &lc) != cudaSuccess || clusters < 1)
      clusters = num_sms() / 2;
    units = clusters;
  }
  if (units > tiles) units = tiles;
  if (units < 1) units = 1;
  lc.gridDim = dim3(unsigned(units * C::CTAS));
  if (pdl_enabled()) {  // see launch_kernel
    attr[lc.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[lc.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs += 1;
  }
  MOE_CUDA_CHECK(cudaLaunchKernelEx(&lc, kern, ta, tb, to, to2, p));
  return MOE_OK;
}

// wgrad_resident_kernel's launch: the K-ragged MN-major operands as run_gemm maps them,
// fp32 outputs in 32 x 32 boxes, one CTA per SM (at most one per tile).
int run_wgrad_resident(const GemmDesc& d, cudaStream_t st) {
  using R = ResCfg;
  if (!d.koffs || d.c1 < 1 || d.groups < 1 || d.groups > kMaxGroups || d.b_tiled)
    return MOE_ERR_INVALID_ARG;
  if (d.c1 % 64 || d.N % 8 || d.a_krows < 1 || d.b_krows < 1) return MOE_ERR_UNSUPPORTED;
  if (d.epi != EPI_F32_BIAS || d.ldo != d.N) return MOE_ERR_UNSUPPORTED;
  CUtensorMap ta, tb, to, to2;
  int rc;
  if ((rc = make_map(&ta, d.A, d.a_krows, d.c1, 64)) != MOE_OK) return rc;
  if ((rc = make_map(&tb, d.B, d.b_krows, d.N, 64)) != MOE_OK) return rc;
  memset(&to, 0, sizeof(to));
  memset(&to2, 0, sizeof(to2));
  const int64_t out_rows = int64_t(d.groups) * d.c1 / (d.out2 ? 2 : 1);
  if ((rc = make_map_f32_out(&to, d.out, out_rows, d.N, 32)) != MOE_OK) return rc;
  if (d.out2 && (rc = make_map_f32_out(&to2, d.out2, out_rows, d.N, 32)) != MOE_OK) return rc;
  KParams p;
  memset(&p, 0, sizeof(p));
  p.groups = d.groups;
  p.rows_cap = int64_t(d.groups) * d.c1;
  p.N = d.N;
  p.K = d.K;
  p.n_tiles = (d.N + R::BN - 1) / R::BN;
  p.out = d.out;
  p.ldo = d.ldo;
  p.n_valid = d.n_valid;
  p.status = d.status;
  p.koffs = d.koffs;
  p.c1 = d.c1;
  p.out2 = d.out2;
  p.aoffs = d.aoffs;
  p.boffs = d.boffs;
  MOE_CUDA_CHECK(cudaFuncSetAttribute(wgrad_resident_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, R::SMEM));
  const int64_t runs =
      int64_t(d.groups) * (((d.c1 + BM - 1) / BM + kRunM - 1) / kRunM) * p.n_tiles;
  if (runs * kRunM > INT32_MAX) return MOE_ERR_UNSUPPORTED;
  int64_t units = num_sms();
  if (units > runs) units = runs;
  if (units < 1) units = 1;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(unsigned(units));
  lc.blockDim = dim3(192);
  lc.dynamicSmemBytes = R::SMEM;
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  if (pdl_enabled()) {  // see launch_kernel
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
  }
  MOE_CUDA_CHECK(cudaLaunchKernelEx(&lc, wgrad_resident_kernel, ta, tb, to, to2, p));
  return MOE_OK;
}

}  // namespace

int make_tma_map_rows(CUtensorMap* m, const void* base, int64_t rows, int K, int box_rows) {
  return make_map(m, base, rows, K, box_rows);
}

int launch_gemm_bf16(const GemmDesc& d, cudaStream_t st) {
  if (d.K < BK || d.K % BK != 0 || d.N < 1) return MOE_ERR_UNSUPPORTED;
  if (d.offsets && (d.groups < 1 || d.groups > kMaxGroups)) return MOE_ERR_UNSUPPORTED;
  if (d.a_rows < 1 || d.a_rows > INT32_MAX || d.b_rows < 1) return MOE_ERR_INVALID_ARG;
  const int bn = gemm_bn(d.N, d.epi);
  // 256-wide tiles of packed weights run on CTA pairs (cta_group::2, 256 x 256 tiles)
  const bool pair = d.b_tiled && bn == 256;
  if (d.koffs) {  // weight gradients: K ragged per group, fp32 out
    if (d.epi != EPI_F32_BIAS || d.groups > kMaxGroups) return MOE_ERR_UNSUPPORTED;
    // the fp32 epilogue masks columns past N, so any N takes the widest tile up to 256.
    // With long K ranges (>= 768 a group on average) and outputs of 256 rows or more a group
    // the tiles run on CTA pairs (256 x 256: each SM pulls 32 KB a k-block for 128 x 256
    // outputs instead of 48 KB); short K ranges are bound by the fp32 stores, where the
    // pair's shared accumulator hand-off only costs (measured: preset 5 backward 3.81 ->
    // 3.53 ms with pairs, preset 2 1.75 -> 2.03 ms)
    const bool pair = d.N > 128 && d.c1 >= 256 && int64_t(d.K) >= 768 * int64_t(d.groups);
    if (d.mn) {  // MN-major operands (row-major activations read in place)
      // short K ranges known to the caller and at least two m-tiles a group: the tiles of a
      // (group, N tile) share their B, which then stays resident (wgrad_resident_kernel)
      if (!pair && d.N > 128 && d.k_max > 0 && d.k_max <= kResKB * BK && d.c1 >= 2 * BM)
        return run_wgrad_resident(d, st);
      if (d.N > 128) return pair ? run_gemm<256, EPI_F32_BIAS, true, true, true>(d, st)
                                 : run_gemm<256, EPI_F32_BIAS, false, true, true>(d, st);
      if (d.N > 64) return run_gemm<128, EPI_F32_BIAS, false, true, true>(d, st);
      return run_gemm<64, EPI_F32_BIAS, false, true, true>(d, st);
    }
    if (pair) return run_gemm<256, EPI_F32_BIAS, true, true>(d, st);
    if (d.N > 128) return run_gemm<256, EPI_F32_BIAS, false, true>(d, st);
    if (d.N > 64) return run_gemm<128, EPI_F32_BIAS, false, true>(d, st);
    return run_gemm<64, EPI_F32_BIAS, false, true>(d, st);
  }
  switch (d.epi) {
    case EPI_DGRAD2:
      if (bn == 256) return pair ? run_gemm<256, EPI_DGRAD2, true>(d, st)
                                 : run_gemm<256, EPI_DGRAD2, false>(d, st);
      if (bn == 128) return run_gemm<128, EPI_DGRAD2, false>(d, st);
      if (bn == 64) return run_gemm<64, EPI_DGRAD2, false>(d, st);
      return MOE_ERR_UNSUPPORTED;
    case EPI_SWIGLU_BWD:
      if (bn == 256) return pair ? run_gemm<256, EPI_SWIGLU_BWD, true>(d, st)
                                 : run_gemm<256, EPI_SWIGLU_BWD, false>(d, st);
      return MOE_ERR_UNSUPPORTED;
    case EPI_F32_BIAS:
      switch (bn) {
        case 16: return run_gemm<16, EPI_F32_BIAS, false>(d, st);
        case 32: return run_gemm<32, EPI_F32_BIAS, false>(d, st);
        case 64: return run_gemm<64, EPI_F32_BIAS, false>(d, st);
        case 128: return run_gemm<128, EPI_F32_BIAS, false>(d, st);
        case 256: return run_gemm<256, EPI_F32_BIAS, false>(d, st);
      }
      return MOE_ERR_UNSUPPORTED;
    case EPI_SWIGLU:
      if (bn == 256) return pair ? run_gemm<256, EPI_SWIGLU, true>(d, st)
                                 : run_gemm<256, EPI_SWIGLU, false>(d, st);
      return MOE_ERR_UNSUPPORTED;
    case EPI_RELU:
      if (bn == 256) return pair ? run_gemm<256, EPI_RELU, true>(d, st)
                                 : run_gemm<256, EPI_RELU, false>(d, st);
      if (bn == 128) return run_gemm<128, EPI_RELU, false>(d, st);
      if (bn == 64) return run_gemm<64, EPI_RELU, false>(d, st);
      return MOE_ERR_UNSUPPORTED;
    case EPI_SCALE:
      if (bn == 256) return pair ? run_gemm<256, EPI_SCALE, true>(d, st)
                                 : run_gemm<256, EPI_SCALE, false>(d, st);
      if (bn == 128) return run_gemm<128, EPI_SCALE, false>(d, st);
      if (bn == 64) return run_gemm<64, EPI_SCALE, false>(d, st);
      return MOE_ERR_UNSUPPORTED;
  }
  return MOE_ERR_INVALID_ARG;
}

}  // namespace moe
