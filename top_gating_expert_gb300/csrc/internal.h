// Internal declarations shared by the CUDA translation units of the MoE library.
// Not part of the public ABI (that is include/moe.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Bits of the device status word (first 4 bytes of every workspace).
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned kStatusNonfinite = 2u;
constexpr unsigned kStatusDeviceData = 4u;

// Byte offset, in every workspace header, of the wait limit in ns (uint64; 0 = 2 s) that
// the kernels' bounded waits apply (moe_set_wait_limit).
constexpr size_t kWaitLimitOffset = 8;

// Tokens per routing chunk (one CTA of the routing kernels, one thread per token).
constexpr int kRouteChunk = 128;

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Byte offsets of every region carved from a workspace.
struct WsLayout {
  int n_cpg = 0;     // routing chunks per group
  int n_chunks = 0;  // G * n_cpg
  size_t status = 0, done = 0, hist = 0, hroute = 0, ppart = 0, zpart = 0, rank = 0,
         gbase = 0, gaux = 0, gz = 0;
  size_t step_bytes = 0;
  size_t logits = 0, x_perm = 0, h_perm = 0, y_perm = 0, h_shared = 0, s_out = 0;
  size_t layer_bytes = 0;
};

inline int64_t rows_max(const moe_config_t& c, int C) {
  int64_t sk = int64_t(c.S) * c.k;
  if (C < 0) return sk;
  int64_t cap = int64_t(c.G) * c.E * C;
  return cap < sk ? cap : sk;
}

inline size_t elem_bytes(const moe_config_t& c) { return c.dtype == MOE_BF16 ? 2 : 4; }

inline WsLayout ws_layout(const moe_config_t& c, int C) {
  WsLayout L;
  const int Sg = c.S / c.G;
  L.n_cpg = (Sg + kRouteChunk - 1) / kRouteChunk;
  L.n_chunks = c.G * L.n_cpg;
  size_t o = 0;
  L.status = o; L.done = o + 4; o += 256;
  L.hist = o;   o = align256(o + size_t(L.n_chunks) * c.k * c.E * 4);
  L.hroute = o; o = align256(o + size_t(L.n_chunks) * c.E * 4);
  L.ppart = o;  o = align256(o + size_t(L.n_chunks) * c.E * 4);
  L.zpart = o;  o = align256(o + size_t(L.n_chunks) * 4);
  L.rank = o;   o = align256(o + size_t(c.S) * c.k * 4);
  L.gbase = o;  o = align256(o + size_t(c.G) * c.E * 4);
  L.gaux = o;   o = align256(o + size_t(c.G) * c.E * 4);  // [G][<= E slices]
  L.gz = o;     o = align256(o + size_t(c.G) * 4);
  L.step_bytes = o;
  const int64_t R = rows_max(c, C);
  const size_t eb = elem_bytes(c);
  const size_t Hs = size_t(c.n_shared) * c.H_shared;
  L.logits = o; o = align256(o + size_t(c.S) * c.E * 4);
  L.x_perm = o; o = align256(o + size_t(R) * c.M * eb);
  // h has 64 more rows, zeroed by every layer forward: the backward's weight-gradient GEMM
  // reads h row-major in 64-row blocks from each expert's first row
  L.h_perm = o; o = align256(o + size_t(R + 64) * c.H * eb);
  L.y_perm = o; o = align256(o + size_t(R) * c.M * eb);
  L.h_shared = o; o = align256(o + size_t(c.S) * Hs * eb);
  L.s_out = o;  o = align256(o + (Hs ? size_t(c.S) * c.M * eb : 0));
  L.layer_bytes = o;
  return L;
}

// Byte offsets of the backward workspace (moe_layer_backward): R rows of the routed
// experts; Rp = R_max + 64 E rows of the per-expert 64-padded segments (gate-scaled dy and
// x gathered into them, zero rows between segments).
struct WsLayoutBwd {
  int64_t Rp = 0, Sp = 0;
  int n_tiles2 = 0;  // gate partials a row of the backward GEMM 2: two per N tile
  size_t status = 0, dy_perm = 0, dh = 0, dab = 0, gpart = 0, dx_perm = 0, poff = 0, poff_s = 0,
         wdyP = 0, xP = 0, dlogits = 0, dx_r = 0, dlb = 0, wgT = 0, koff_e = 0, koff_split = 0,
         dwg_part = 0, dhs = 0, dabs = 0, dxs = 0;
  static constexpr int kMaxSplit = 64;  // split-K ranges of the router's dW_g
  size_t bytes = 0;
};

// ------------------------------------------------------------------ GEMM tiling
// Epilogues of the bf16 tcgen05 GEMM (gemm_tcgen05.cu).
enum GemmEpilogue {
  EPI_F32_BIAS = 0,    // fp32 out (+ per-column bias); in K-ragged mode the weight gradients
  EPI_RELU = 1,        // bf16 relu(D)
  EPI_SWIGLU = 2,      // bf16 silu(D_gate) * D_up
  EPI_SCALE = 3,       // bf16 row_scale[r] * D
  EPI_DGRAD2 = 4,      // backward of GEMM 2: bf16 w_r * D (ReLU: masked by h > 0), gate partials
  EPI_SWIGLU_BWD = 5,  // backward of the SwiGLU: from D = (a | b) and dh, bf16 (da | db)
};

// N-tile width of the bf16 GEMM for N output columns per group (0 = unsupported). The
// packed weight layout depends on it, so packing and launching both take it from here.
inline int gemm_bn(int N, int epi) {
  if (epi == EPI_F32_BIAS) {
    for (int bn = 16; bn <= 256; bn *= 2)
      if (N <= bn) return bn;
    return 0;
  }
  if (epi == EPI_SWIGLU || epi == EPI_SWIGLU_BWD) return N % 256 == 0 ? 256 : 0;
  if (N % 256 == 0) return 256;
  if (N % 128 == 0) return 128;
  if (N % 64 == 0) return 64;
  return 0;
}

inline WsLayoutBwd ws_layout_bwd(const moe_config_t& c, int C) {
  WsLayoutBwd B;
  const int64_t R = rows_max(c, C);
  const bool sw = c.act == MOE_ACT_SWIGLU;
  const int64_t F = sw ? 2 * int64_t(c.H) : c.H;
  const int64_t Hc = int64_t(c.n_shared) * c.H_shared, Fs = sw ? 2 * Hc : Hc;
  B.Rp = (R + 64 * int64_t(c.E) + 63) / 64 * 64;
  B.Sp = (int64_t(c.S) + 63) / 64 * 64;
  const int bn2 = gemm_bn(c.H, EPI_DGRAD2);
  B.n_tiles2 = bn2 > 0 ? 2 * (c.H / bn2) : 1;  // two column halves a tile
  const size_t eb = c.dtype == MOE_BF16 ? 2 : 4;  // the row buffers' element size
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o = align256(o + bytes); return at; };
  B.status = take(256);
  B.dy_perm = take(size_t(R) * c.M * eb);
  B.dh = take(sw ? size_t(R) * c.H * eb : 0);
  B.dab = take(size_t(R + 64) * F * eb);  // + 64 zeroed rows (read past the last segment)
  B.gpart = take(size_t(R) * B.n_tiles2 * 4);
  B.dx_perm = take(size_t(R) * c.M * eb);
  B.poff = take(size_t(c.E + 1) * 4);
  B.poff_s = take(2 * 4);
  B.wdyP = take(size_t(B.Rp) * c.M * eb);
  B.xP = take(size_t(B.Rp) * c.M * eb);
  B.dlogits = take(size_t(c.S) * c.E * 4);
  B.dx_r = take(size_t(c.S) * c.M * 4);
  const size_t Ep = (size_t(c.E) + 63) / 64 * 64;
  B.dlb = take(size_t(c.S) * Ep * 2);
  B.wgT = take(size_t(c.M) * Ep * 2);
  B.koff_e = take(2 * 4);
  B.koff_split = take((WsLayoutBwd::kMaxSplit + 1) * 4);
  // dW_g's split-K partials ([splits][Ep][M]), later the bias partials ([S/256 chunks][E])
  const size_t nch = (size_t(c.S) + 255) / 256;
  const size_t part_floats = size_t(WsLayoutBwd::kMaxSplit) * Ep * c.M;
  B.dwg_part = take((part_floats > nch * c.E ? part_floats : nch * c.E) * 4);
  B.dhs = take(sw ? size_t(c.S) * Hc * eb : 0);
  B.dabs = take(size_t(c.S) * Fs * eb);
  B.dxs = take(Hc ? size_t(c.S) * c.M * eb : 0);
  B.bytes = o;
  return B;
}

// ------------------------------------------------------------------ launchers
// route.cu. With a DispatchFuse, the last routing kernel also writes x_perm (the dispatch
// gather, x_perm[row[t, j]] = x[t] for every kept choice); the routing outputs are the same.
struct DispatchFuse {
  const void* x;             // [S, M], 16-byte aligned
  void* x_perm;              // [R_max, M], 16-byte aligned
  const void* prefetch;      // nullable: bytes to bring into L2 while the routing finishes
  int64_t prefetch_bytes;    // (the first expert GEMM's first weight tiles), multiple of 16
  void* h_tail;              // nullable: h [R_max + 64, h_cols] bf16, rows R .. R + 63 zeroed
  int h_cols;                //   (R = the kept rows; h_cols % 8 == 0)
};
int launch_route(const moe_config_t& c, int C, const float* logits, const float* u,
                 const moe_route_out_t& out, char* ws, const WsLayout& L, cudaStream_t st,
                 const DispatchFuse* d = nullptr);
// bf16 router projection fused with the first routing kernel (logits_out nullable), then the
// same scan and finalize kernels as launch_route.
int launch_router_route(const moe_config_t& c, int C, const void* x, const void* W_g,
                        const float* bias, const float* u, float* logits_out,
                        const moe_route_out_t& out, char* ws, const WsLayout& L, cudaStream_t st,
                        const DispatchFuse* d = nullptr);

// permute.cu
int launch_dispatch(const moe_config_t& c, int64_t R_max, const void* x, const int32_t* token_of,
                    const int32_t* offsets, void* x_perm, cudaStream_t st);
int launch_combine(const moe_config_t& c, const void* y_perm, const int32_t* row,
                   const void* shared_out, const void* residual, void* y, int64_t R_max,
                   cudaStream_t st, const float* add32 = nullptr);  // + fp32 [S, M] term
// Weight packing. bf16: tile-major [groups][N/BN][K/64][BN][64] (one contiguous 32 KB block
// per TMA box of the GEMM, BN = gemm_bn); fp32: row-major [groups][N][K].
//   first layer: N = H (ReLU) or 2H (SwiGLU: blocks of 256 rows = 128 W_in rows, then the
//                same 128 W_up rows), K = M;
//   second layer: N = M, K = H (W_out [groups][M][H], or n_shared experts side by side).
int launch_pack_in(const moe_config_t& c, int groups, int H, const void* W_in, const void* W_up,
                   void* packed, cudaStream_t st);
int launch_pack_out(const moe_config_t& c, int groups, int H, int n_parts, const void* W_out,
                    void* packed, cudaStream_t st);

// gemm_tcgen05.cu : bf16 GEMM D = A . B^T over ragged row groups, tcgen05 + TMA.
struct GemmDesc {
  int epi = EPI_RELU;
  const void* A = nullptr; int64_t a_rows = 0; int K = 0;  // A [a_rows, K] bf16, row-major
  const void* B = nullptr; int64_t b_rows = 0;             // B [b_rows, K] bf16
  bool b_tiled = false;            // B packed tile-major (see launch_pack_in), else row-major
  int N = 0;                       // B rows per group = GEMM N of each group
  const int32_t* offsets = nullptr;  // device [groups+1] row offsets into A; null = dense
  int groups = 1;
  int rows_dense = 0;              // rows of the single group when offsets is null
  void* out = nullptr; int64_t ldo = 0;  // output element stride between rows
  const float* row_scale = nullptr;      // EPI_SCALE: per-row factor (null = 1)
  const float* bias = nullptr;           // EPI_F32_BIAS: per-column bias (nullable)
  int n_valid = 0;                       // EPI_F32_BIAS: columns stored
  unsigned* status = nullptr;
  // EPI_DGRAD2: aux = h [rows, N] bf16 (ld_aux elements a row), gpart = per-(row, N tile,
  // column half) sums of D * h, [rows][N / BN][2] (nullable), relu = mask by h > 0.
  // EPI_SWIGLU_BWD: aux = dh [rows, N/2].
  const void* aux = nullptr; int64_t ld_aux = 0;
  float* gpart = nullptr;
  int relu = 0;
  // K-ragged mode (weight gradients, EPI_F32_BIAS): group g = rows g*c1 .. g*c1 + c1 - 1 of
  // the output, its K range [koffs[g], koffs[g+1]) (multiples of 64) of A [c1, K] and
  // B [N, K] (both row-major; A and B are shared by all groups, K = koffs[groups]).
  const int32_t* koffs = nullptr;
  int c1 = 0;
  // with out2: output rows are pairs of 128-row blocks (the interleaved SwiGLU order) that go
  // to out (first block) and out2 (second), each [groups * c1 / 2, N]
  void* out2 = nullptr;
  // MN-major K-ragged mode: A [a_krows, c1] and B [b_krows, N] row-major, K along the rows;
  // group g takes koffs[g+1] - koffs[g] rows from row aoffs[g] of A and boffs[g] of B (null:
  // koffs[g]); rows past a tensor's end read as zeros
  // grouped rows: walk the tiles from the last group's (GEMM 2 then starts on the rows of h
  // that GEMM 1 wrote last, still in L2)
  bool reverse = false;
  // the output is read by the next kernel (GEMM 1's h by GEMM 2): with about one m-tile a
  // group, its stores are marked evict-last in L2
  bool out_keep = false;
  bool mn = false;
  int64_t a_krows = 0, b_krows = 0;
  const int32_t* aoffs = nullptr;
  const int32_t* boffs = nullptr;
  // K-ragged mode: a bound the caller knows on every group's K range (0: none known). With
  // at most 256 a group, MN-major 256-wide outputs run the resident-B kernel
  int k_max = 0;
};
int launch_gemm_bf16(const GemmDesc& d, cudaStream_t st);
// 2-D tensor map over a row-major bf16 [rows, K] matrix, boxes of 64 columns x box_rows rows,
// 128-byte swizzle (the operand layout of the tcgen05 kernels).
int make_tma_map_rows(CUtensorMap* m, const void* base, int64_t rows, int K, int box_rows);

// simt_f32.cu : plain-FMA fp32 path for small layers.
int launch_router_f32(const moe_config_t& c, const float* x, const float* W_g, const float* bias,
                      float* logits, cudaStream_t st);
int launch_ffn_up_f32(const moe_config_t& c, int H, const float* A, const int32_t* offsets,
                      int groups, int rows_dense, int64_t rows_cap, const float* W_packed,
                      float* h, unsigned* status, cudaStream_t st);
int launch_ffn_down_f32(const moe_config_t& c, int H, const float* h, const int32_t* offsets,
                        int groups, int rows_dense, int64_t rows_cap, const float* row_scale,
                        const float* W_out, float* y, unsigned* status, cudaStream_t st);

// backward.cu
int launch_pad_offsets(const int32_t* offsets, int groups, int dense_rows, int32_t* poff,
                       cudaStream_t st);
// dst[p] = scale[r] * src[token_of[r]] over per-expert 64-padded segments (poff), zeros
// in the padding; with tail, 64 rows of tail from row offsets[E] zeroed (bf16, cols % 8 == 0)
int launch_pad_gather(const void* src, int cols, const int32_t* token_of, const float* scale,
                      const int32_t* offsets, const int32_t* poff, int E, int S, int64_t rows_bound,
                      void* out, void* tail, int tail_cols, unsigned* status, cudaStream_t st);
int launch_seg_transpose(const void* in, int64_t ld_in, const int32_t* offsets, int groups,
                         int dense_rows, const int32_t* poff, int64_t rows_pad_max,
                         const int32_t* gather, int src_rows, const float* scale, int C, void* out,
                         int64_t ld_out, unsigned* status, cudaStream_t st);
int launch_pack_transposed(int mode, int swiglu, int groups, int N, int K, int M, int Hp, int parts,
                           const void* W, const void* W2, void* dst, cudaStream_t st);
// the router backward's scratch (all in the backward workspace)
struct RouterBwdBufs {
  float* dlogits;  // [S][E] fp32
  void* dlb;       // [S][Ep] bf16, Ep = E rounded up to 64
  void* wgT;       // [M][Ep] bf16
  float* dx_r;     // [S][M] fp32
  int32_t* koff_e; int32_t* koff_s;  // [2] each
  int64_t Sp;
  int32_t* koff_split;  // [max_split + 1]: split-K ranges of dW_g
  float* dwg_part;      // [max_split][Ep][M] partials of dW_g
  int max_split;
};
int launch_router_backward(const moe_config_t& c, const float* logits, const moe_route_out_t& r,
                           const float* gpart, int n_tiles, float aux_coef, float z_coef,
                           const RouterBwdBufs& b, const void* x, const void* W_g, float* dW_g,
                           float* dbias, unsigned* status, cudaStream_t st);

// backward_f32.cu: the fp32 path's backward on plain FMA.
// One expert FFN's data gradients on (ragged or dense) row segments, fp32 row-major: D =
// dy_rows . W_out into dab, the gate partials (gpart[r][0], the other n_tiles - 1 entries 0),
// da (ReLU: masked by h > 0) or dh then (da | db) in the forward pack's column order
// (SwiGLU), dx_rows = (da | db) . W_in.
struct FfnBwdF32 {
  const void* x_rows; int64_t rows_cap; const int32_t* offsets; int groups; int dense_rows;
  int M, Hn, swiglu;
  const void* W_in_packed;  // the forward's fp32 pack [groups][F][M] (SwiGLU recompute)
  const void* Wt_in;        // [groups][M][F]
  const void* Wt_out;       // [groups][Hn][M]
  const void* dy_rows;      // [rows_cap][M]
  const float* w;           // per-row gate (null: 1)
  const void* h;            // the forward's hidden rows [rows_cap][Hn]
  void* dh;                 // SwiGLU scratch [rows_cap][Hn]
  void* dab;                // [rows_cap][F]
  float* gpart; int n_tiles;
  void* dx_rows;            // [rows_cap][M]
};
int ffn_backward_data_f32(const FfnBwdF32& f, cudaStream_t st);
// out[g][a][b] = sum over group g's rows r, in order, of s_r P[r][pc(a)] Q[r][b]; pmode 0:
// pc(a) = a; 1 / 2: the SwiGLU gate / up column of unit a in the forward pack's order
int weight_grad_f32(const void* P, int ldP, const float* scale, int pmode, const void* Q, int ldQ,
                    const int32_t* offsets, int groups, int dense_rows, int A, int Bn, float* out,
                    cudaStream_t st);
// the router's dx_r = dlogits . W_g and dW_g = dlogits^T x
int router_grads_f32(const moe_config_t& c, const float* dlogits, const void* x, const void* W_g,
                     float* dx_r, float* dW_g, cudaStream_t st);
// the backward's transposed weights for fp32, row-major [groups][N][K] (the index rules of
// launch_pack_transposed)
int launch_pack_transposed_f32(int mode, int swiglu, int groups, int N, int K, int M, int Hp,
                               int parts, const void* W, const void* W2, void* dst,
                               cudaStream_t st);

int num_sms();

// Programmatic dependent launch: every kernel of the library is launched with programmatic
// stream serialisation (unless the environment sets MOE_PDL=0), so that it may start while
// its predecessor in the stream drains. Each kernel therefore calls pdl_wait() before its
// first global-memory access (it returns once the preceding kernel has completed and its
// writes are visible; without the attribute it returns at once), then pdl_trigger() to let
// its own successor be scheduled.
bool pdl_enabled();

template <typename... Params, typename... Args>
int launch_kernel(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                  Args&&... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  if (pdl_enabled()) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
  }
  if (cudaLaunchKernelEx(&lc, kernel, static_cast<Args&&>(args)...) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

#ifdef __CUDACC__
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// 16-byte row copies: a read-only load that skips L1, and a plain store (the copy's
// destination is read again soon, by the next kernel)
__device__ __forceinline__ uint4 ld_nc_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
// L2 prefetch of [p, p + bytes): p 16-byte aligned, bytes a multiple of 16
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void st_v4(uint4* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
#endif

}  // namespace moe

#define MOE_CUDA_CHECK(call)                       \
  do {                                             \
    cudaError_t e_ = (call);                       \
    if (e_ != cudaSuccess) return MOE_ERR_CUDA;    \
  } while (0)
