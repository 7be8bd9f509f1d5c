/*
 * moe.h -- C ABI of the GB300 (sm_103a) Mixture-of-Experts layer forward.
 *
 * One GPU computes one MoE layer forward:
 *   router projection -> softmax / top-k gates -> random 2nd-expert dispatch ->
 *   per-(group, expert) capacity slots -> expert-contiguous rows -> gather ->
 *   grouped expert FFN (GEMM1 + activation, GEMM2 + gate) -> combine back to token order,
 * plus the load-balancing (aux) loss and the router z-loss.
 *
 * Sources, by page title and section:
 *   GShard summary page ("GShard: Scaling Giant Models with Conditional Computation and
 *     Automatic Sharding"): "MoE Transformer", "Top-2 gating" (Expert capacity, Local
 *     group dispatching, Auxiliary loss, Random routing), and the dispatch path listing
 *     "token hidden states -> router scores -> top-k -> capacity / token position
 *     assignment -> dispatch -> local experts -> combine".
 *   "04 · 路由、负载均衡与专家并行" (MegaBlocks router and parallelism): §2 router
 *     (bias-free linear, softmax, top-k, z-loss), §3 load-balancing loss, §6 shared expert.
 *   "Lec16 Systems for MoE Models": "Switch Transformer" (Softmax(KeepTopK)), "共享专家
 *     vs. 路由专家", "MoE 训练中的负载均衡", "DeepSeek V3 MoE" (SwiGLU), "MoE Kernel 优化"
 *     (fused gating kernel, dense token-to-expert table).
 *
 * Conventions (every entry point):
 *   - Pointers named x, W_*, logits, y, *_perm, ws and the fields of moe_route_out_t are
 *     DEVICE pointers owned by the caller. The library allocates no device memory,
 *     frees nothing and keeps no pointer after a call returns.
 *   - moe_config_t pointers are HOST pointers, read during the call only.
 *   - Calls are asynchronous and ordered on `stream` (NULL = the legacy default stream);
 *     none synchronises except moe_get_device_status.
 *   - Row-major tensors; weights in the [out, in] (K-major) layout of a linear layer:
 *     W_g [E, M]; W_in, W_up [E, H, M]; W_out [E, M, H]; shared Ws_in, Ws_up
 *     [n_shared, H_shared, M]; Ws_out [n_shared, M, H_shared].
 *   - Element type of x, weights, x_perm, h, y_perm, y, residual: float (MOE_F32) or
 *     bf16 (MOE_BF16, raw 16-bit storage). logits, gate, w_perm, bias, u, losses: float.
 *   - Return value: MOE_OK (0) or a negative MOE_ERR_* code. Host-side checks (shapes,
 *     nulls, workspace size) fail before anything is launched. Errors found on the
 *     device (non-finite logits, a bounded wait that ran out, bad device indices) are
 *     recorded in the workspace's status word and reported by moe_get_device_status.
 *   - No C++ exception crosses this boundary.
 */
#ifndef TOP_GATING_EXPERT_GB300_MOE_H
#define TOP_GATING_EXPERT_GB300_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* a cudaStream_t */

/* element types and activations */
enum { MOE_F32 = 0, MOE_BF16 = 1 };
enum { MOE_ACT_RELU = 0, MOE_ACT_SWIGLU = 1 };

/* status codes */
enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1, /* shape, divisibility, null pointer, bad enum            */
  MOE_ERR_UNSUPPORTED = -2, /* valid but not built: dtype/act/size combination         */
  MOE_ERR_WORKSPACE = -3,   /* ws too small or misaligned                              */
  MOE_ERR_CUDA = -4,        /* a CUDA runtime call or a kernel launch failed            */
  MOE_ERR_TIMEOUT = -5,     /* device: a bounded wait ran out (kernel returned early)   */
  MOE_ERR_NONFINITE = -6,   /* device: a router logit was NaN or infinite               */
  MOE_ERR_DEVICE_DATA = -7  /* device: an index or offset read on the device was invalid */
};

/* gate normalisations (moe_config_t.gate_norm) */
enum { MOE_GATE_SOFTMAX_TOPK = 0, MOE_GATE_NONE = 1, MOE_GATE_PNORM = 2 };

/* drop_reason values */
enum { MOE_KEPT = 0, MOE_DROP_CAPACITY = 1, MOE_DROP_RANDOM = 2 };

/* workspace kinds for moe_workspace_bytes */
enum { MOE_WS_STEP = 0, MOE_WS_LAYER = 1, MOE_WS_BACKWARD = 2 };

/*
 * Layer configuration. Parameter names follow the pages' problem statement: S tokens,
 * G groups (GShard "Local group dispatching": S/G consecutive tokens per group), E routed
 * experts, M = d_model, H = d_ff, k = experts per token, capacity factor, shared experts.
 *   S >= 1, G >= 1, S % G == 0; 1 <= E <= 256; 1 <= k <= min(E, 8).
 *   capacity_factor > 0: capacity mode, C = ceil(capacity_factor * k * (S/G) / E) per
 *     (group, expert) (GShard "Local group dispatching": 2N/(G*E) at factor 1, k = 2);
 *     capacity_factor <= 0: dropless (no assignment is dropped).
 *   random_routing: 0/1; 1 needs k == 2 and a non-null u (GShard "Random routing").
 *   n_shared >= 0 always-on shared experts of hidden size H_shared, each added with
 *     weight 1 (Lec16 "共享专家 vs. 路由专家").
 *   bf16: M % 64 == 0, H % 64 == 0 (H % 128 == 0 for SwiGLU), n_shared*H_shared likewise.
 *   f32 (the plain-FMA path, meant for small layers): M % 4 == 0, H % 4 == 0 (H % 128 == 0
 *     for SwiGLU), H_shared % 4 == 0.
 * Routing variants (a zero-filled tail gives the default routing above):
 *   gate_norm: MOE_GATE_SOFTMAX_TOPK (softmax over the k selected logits), MOE_GATE_NONE
 *     (the k full-softmax probabilities as they are: Lec16 "DeepSeek V3 MoE",
 *     TopK(Softmax(h W), 8)) or MOE_GATE_PNORM (those probabilities divided by their
 *     gate_p-norm; gate_p > 0, finite: MegaBlocks router §2). The random-routing
 *     decision always uses the softmax over the two selected logits.
 *   n_expert_groups: 0 or 1 = off; else 2..16 dividing E: the experts form that many
 *     contiguous groups, each token keeps the topk_groups (1..n_expert_groups) groups
 *     of largest best logit (ties to the lower group) and takes its top-k among their
 *     experts; k <= topk_groups * E / n_expert_groups (Lec16 "DeepSeek V3 MoE": 8
 *     groups, 4 kept).
 *   uniform_assignment: 0/1; 1 replaces token t's expert ids by (t*k + j) mod E and keeps
 *     the router's gates (MegaBlocks router §2 benchmark switch); not with
 *     random_routing.
 */
typedef struct {
  int32_t S, G, E, M, H, k;
  float capacity_factor;
  int32_t random_routing;
  int32_t n_shared, H_shared;
  int32_t act;   /* MOE_ACT_* */
  int32_t dtype; /* MOE_F32 / MOE_BF16 */
  int32_t gate_norm;  /* MOE_GATE_* */
  float gate_p;
  int32_t n_expert_groups, topk_groups;
  int32_t uniform_assignment;
} moe_config_t;

/*
 * Routing outputs (all device pointers, caller-allocated). R_max = moe_rows_max().
 *   expert_id   int32 [S, k]  chosen experts, largest logit first; equal logits rank
 *                             the lower expert index first.
 *   gate        float [S, k]  Softmax over the k selected logits (= the full softmax's
 *                             top-k probabilities renormalised), or as gate_norm says;
 *                             0 where not kept.
 *   pos         int32 [S, k]  slot in the (group, expert) queue, -1 when not kept.
 *                             Queue order: all 1st choices of the group in token order,
 *                             then all 2nd choices, ...; random-skipped choices take no slot.
 *   drop_reason uint8 [S, k]  MOE_KEPT / MOE_DROP_CAPACITY / MOE_DROP_RANDOM.
 *   row         int32 [S, k]  row of the assignment in the expert-contiguous buffers,
 *                             -1 when not kept.
 *   counts      int32 [G, E]  kept assignments per (group, expert).
 *   counts_routed int32 [G, E] top-k choices per (group, expert) before random routing
 *                             and capacity (the f_e of the aux loss).
 *   expert_offsets int32 [E+1] first row of each expert; expert_offsets[E] = R rows used.
 *                             Inside an expert: group by group, each in slot order.
 *   token_of    int32 [R_max] token of each row (rows >= R untouched).
 *   w_perm      float [R_max] gate of each row.
 *   aux_loss    float [1]     E * sum_e f_e * P_e per group, mean over groups; f_e =
 *                             counts_routed / (S/G * k), P_e = mean softmax probability.
 *   z_loss      float [1]     mean over tokens of logsumexp(logits)^2.
 */
typedef struct {
  int32_t* expert_id;
  float* gate;
  int32_t* pos;
  uint8_t* drop_reason;
  int32_t* row;
  int32_t* counts;
  int32_t* counts_routed;
  int32_t* expert_offsets;
  int32_t* token_of;
  float* w_perm;
  float* aux_loss;
  float* z_loss;
} moe_route_out_t;

/* ---------------------------------------------------------------- host-only queries */

/* Human-readable name of a status code (static storage). */
const char* moe_status_string(int status);

/* ABI version of this library (major * 100 + minor): 102 (moe_config_t with the routing
 * variant fields; moe_set_wait_limit). */
int moe_abi_version(void);

/* MOE_OK if the configuration is valid and built, else the reason. Host only. */
int moe_validate_config(const moe_config_t* cfg);

/* Capacity per (group, expert); *C = -1 in dropless mode. Host only. */
int moe_capacity(const moe_config_t* cfg, int32_t* C);

/* Upper bound on kept assignments: min(S*k, G*E*C) in capacity mode, S*k dropless. */
int moe_rows_max(const moe_config_t* cfg, int64_t* R_max);

/*
 * Workspace bytes. MOE_WS_STEP: what moe_router, moe_route, moe_expert_* and
 * moe_shared_ffn need (status word + routing scratch). MOE_WS_BACKWARD: what
 * moe_layer_backward needs. MOE_WS_LAYER: what
 * moe_layer_forward needs (the step workspace plus logits, x_perm, h, y_perm and the
 * shared-expert buffers). Workspaces must be 256-byte aligned and zero-filled once
 * before first use: their first 256 bytes are a header holding the status word (bytes
 * 0..3), a ticket (4..7) and the wait limit (8..15, see moe_set_wait_limit).
 */
int moe_workspace_bytes(const moe_config_t* cfg, int kind, size_t* bytes);

/* Element counts of the packed weight buffers (see moe_pack_weights); any may be NULL. */
int moe_packed_sizes(const moe_config_t* cfg, int64_t* w_in_packed_elems,
                     int64_t* w_out_packed_elems, int64_t* ws_in_packed_elems,
                     int64_t* ws_out_packed_elems);

/* ---------------------------------------------------------------- weight packing */

/*
 * Packs the routed experts' weights once, before any forward, into the layout the grouped
 * GEMMs stream.
 *   First layer, logical [E, N1, M]: ReLU N1 = H (W_in; W_up unused, may be NULL); SwiGLU
 *   N1 = 2H in blocks of 256 rows: block b holds W_in rows 128b..128b+127 then W_up rows
 *   128b..128b+127, so one 256-wide GEMM tile sees a gate column and its up column
 *   (Lec16 "DeepSeek V3 MoE": (Swish(x W1) * (x W2)) W3, W1 = W_in, W2 = W_up, W3 = W_out).
 *   Second layer, logical [E, M, H] = W_out.
 *   bf16: each logical [groups, N, K] matrix is stored tile-major,
 *   [groups][N/BN][K/64][BN][64], so every 64-column x BN-row box the GEMM loads is one
 *   contiguous block (BN = 256, 128 or 64: the GEMM's N tile). fp32: row-major.
 * Sizes: moe_packed_sizes. Packed buffers must not alias the unpacked ones.
 */
int moe_pack_weights(const moe_config_t* cfg, const void* W_in, const void* W_up,
                     const void* W_out, void* W_in_packed, void* W_out_packed,
                     moe_stream_t stream);

/*
 * Packs the n_shared shared experts as ONE expert whose hidden units are all of theirs
 * (a sum of FFNs is one FFN over the concatenated hidden dimension), in the layouts of
 * moe_pack_weights:
 *   Ws_in_packed  logical [n_shared*H_shared (x2 for SwiGLU, interleaved as above), M]
 *   Ws_out_packed logical [M, n_shared*H_shared]
 */
int moe_pack_shared_weights(const moe_config_t* cfg, const void* Ws_in, const void* Ws_up,
                            const void* Ws_out, void* Ws_in_packed, void* Ws_out_packed,
                            moe_stream_t stream);

/* ---------------------------------------------------------------- the forward steps */

/*
 * Router projection (MegaBlocks §2: a linear layer without bias; Lec16 "Switch
 * Transformer": G(x) = Softmax(x W_g)). logits [S, E] float = x [S, M] . W_g[E, M]^T
 * accumulated in fp32, plus bias[e] when bias (float [E]) is non-null.
 */
int moe_router(const moe_config_t* cfg, const void* x, const void* W_g, const float* bias,
               float* logits, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Routing from logits [S, E] (float): softmax and logsumexp, top-k and gates, random
 * 2nd-expert dispatch (keep iff u[t] < 2 / (1 + exp(l1 - l2)) in fp64, u float [S]),
 * capacity slots, expert-contiguous rows, aux and z losses. Fills every field of *out.
 * Integer outputs are a pure function of the logits and u (bit-exact, deterministic).
 * Non-finite logits set MOE_ERR_NONFINITE in the status word.
 */
int moe_route(const moe_config_t* cfg, const float* logits, const float* u,
              const moe_route_out_t* out, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_router followed by moe_route in one pass over x: the same outputs in *out, and the
 * logits in logits_out when it is non-null (Lec16 Systems for MoE Models, "MoE Kernel
 * 优化": the gating function -- projection, softmax, top-k and the token-to-expert table --
 * fused instead of one kernel per step).
 *   bf16: one kernel per 128-token chunk computes the chunk's logits on the tensor cores
 *         and routes from them without writing them to memory (unless logits_out is
 *         given), then moe_route's scan and finalize kernels run. logits_out may be NULL.
 *   fp32: moe_router into logits_out, then moe_route; logits_out must be non-null.
 * The logits equal moe_router's bit for bit, and every output equals what moe_route
 * computes from them, bit for bit, except that with E <= 16 aux_loss and z_loss may differ
 * in the last bits (the softmax sums are split over more threads). Passing logits_out or
 * not changes no other output. ws: MOE_WS_STEP bytes. Errors: as moe_router and moe_route.
 */
int moe_router_route(const moe_config_t* cfg, const void* x, const void* W_g, const float* bias,
                     const float* u, float* logits_out, const moe_route_out_t* out, void* ws,
                     size_t ws_bytes, moe_stream_t stream);

/*
 * moe_route without a workspace, for callers that cannot allocate device memory. The
 * paper has no counterpart: this is a deployment convenience of this library.
 *
 * Who needs it: code that may not call cudaMalloc, for example a plugin running inside a
 * host framework whose own allocator owns all device memory, or a latency-critical loop
 * that must not allocate once it has started. Such a caller passes only inputs and
 * outputs; the routing scratch comes from a fixed 4 MiB array inside this library, which
 * every GPU that loads the library holds until the process exits.
 *
 *   - Same inputs, outputs and results as moe_route (bit-identical).
 *   - Configurations whose routing scratch exceeds 4 MiB (moe_workspace_bytes with
 *     MOE_WS_STEP) are rejected with MOE_ERR_WORKSPACE before anything is launched.
 *   - The first call on each device looks up the array's device address (with that device
 *     current); make that first call before any stream capture.
 *   - All calls share the one array: calls that overlap on the GPU (on different streams,
 *     or from different host threads) race and corrupt each other's results. Order them.
 *   - device_status (nullable, device int32) receives the call's device status bits:
 *     0 = ok, 2 = non-finite logits, 4 = invalid device data.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
int moe_route_noalloc(const moe_config_t* cfg, const float* logits, const float* u,
                      const moe_route_out_t* out, int32_t* device_status, moe_stream_t stream);

/* Gather: x_perm[r, :] = x[token_of[r], :] for r < expert_offsets[E]. x_perm [R_max, M]. */
int moe_dispatch(const moe_config_t* cfg, const void* x, const moe_route_out_t* r,
                 void* x_perm, moe_stream_t stream);

/*
 * Grouped GEMM 1 with the activation fused in its epilogue, over the ragged expert
 * segments given by expert_offsets (device):
 *   ReLU:   h[r, :] = relu(x_perm[r] . W_in[e]^T)                    h_perm [R_max, H]
 *   SwiGLU: h[r, :] = silu(x_perm[r] . W_in[e]^T) * (x_perm[r] . W_up[e]^T)
 * fp32 accumulation; h stored in the element type (bf16 rounds once).
 */
int moe_expert_up(const moe_config_t* cfg, const void* x_perm, const int32_t* expert_offsets,
                  const void* W_in_packed, void* h_perm, void* ws, size_t ws_bytes,
                  moe_stream_t stream);

/* Grouped GEMM 2 with the gate fused in its epilogue (W_out_packed from moe_pack_weights):
 *   y_perm[r, :] = w_perm[r] * (h_perm[r] . W_out[e]^T)                 y_perm [R_max, M] */
int moe_expert_down(const moe_config_t* cfg, const void* h_perm, const int32_t* expert_offsets,
                    const float* w_perm, const void* W_out_packed, void* y_perm, void* ws,
                    size_t ws_bytes, moe_stream_t stream);

/* moe_expert_up followed by moe_expert_down; h_perm is caller scratch [R_max, H]. */
int moe_expert_ffn(const moe_config_t* cfg, const void* x_perm, const int32_t* expert_offsets,
                   const float* w_perm, const void* W_in_packed, const void* W_out_packed,
                   void* h_perm, void* y_perm, void* ws, size_t ws_bytes, moe_stream_t stream);

/* The shared experts on every token (weight 1 each):
 *   shared_out [S, M] = FFN_shared(x) with the packed weights; h_shared [S, n_shared*H_shared]
 *   is caller scratch. */
int moe_shared_ffn(const moe_config_t* cfg, const void* x, const void* Ws_in_packed,
                   const void* Ws_out_packed, void* h_shared, void* shared_out, void* ws,
                   size_t ws_bytes, moe_stream_t stream);

/*
 * Combine (scatter back to token order): for every token t,
 *   y[t] = sum over kept choices j, in ascending j, of y_perm[row[t, j]]
 *          (+ shared_out[t] if non-null) (+ residual[t] if non-null),
 * summed in fp32 and rounded once. A token with nothing kept gets 0 (+ residual): the
 * GShard overflow token passes through the residual connection.
 */
int moe_combine(const moe_config_t* cfg, const void* y_perm, const moe_route_out_t* r,
                const void* shared_out, const void* residual, void* y, moe_stream_t stream);

/*
 * The whole layer: moe_router_route, moe_dispatch, moe_expert_ffn, moe_shared_ffn
 * (when n_shared > 0) and moe_combine, with the intermediates carved from ws
 * (MOE_WS_LAYER bytes). logits_out (float [S, E]) receives the router logits when
 * non-null. W_*_packed / Ws_*_packed come from the pack calls above; bias, u, residual
 * and the shared weights may be NULL when unused. Results are those of the separate calls
 * bit for bit; the launches differ: the routing's last kernel also does the dispatch
 * gather (and brings GEMM 1's first weight tiles into L2), and the 64 rows of h after the
 * kept ones are zeroed in ws for moe_layer_backward. Only the first 256 bytes of ws (the
 * status word and a ticket) must be zero when it is first used; nothing else in it is read
 * before it is written.
 */
int moe_layer_forward(const moe_config_t* cfg, const void* x, const void* W_g, const float* bias,
                      const void* W_in_packed, const void* W_out_packed, const void* Ws_in_packed,
                      const void* Ws_out_packed, const float* u, const void* residual, void* y,
                      float* logits_out, const moe_route_out_t* r, void* ws, size_t ws_bytes,
                      moe_stream_t stream);

/* ---------------------------------------------------------------- the backward pass */

/*
 * Transposed weights for the backward's data-gradient GEMMs (element counts as
 * moe_packed_sizes' w_in / w_out):
 *   Wt_out_packed  logical [E, H, M]: W_out[e] transposed (gradient through GEMM 2);
 *   Wt_in_packed   logical [E, M, H] (ReLU) or [E, M, 2H] (SwiGLU, the K order of the forward's
 *                  interleaved pack): W_in[e] (and W_up[e]) transposed.
 * bf16: packed tile-major like the forward's; fp32: plain row-major in the logical shape.
 */
int moe_pack_weights_backward(const moe_config_t* cfg, const void* W_in, const void* W_up,
                              const void* W_out, void* Wt_in_packed, void* Wt_out_packed,
                              moe_stream_t stream);

/* The same for the shared experts, with their hidden units side by side (counts as
 * moe_packed_sizes' ws_in / ws_out). */
int moe_pack_shared_weights_backward(const moe_config_t* cfg, const void* Ws_in, const void* Ws_up,
                                     const void* Ws_out, void* Wst_in_packed, void* Wst_out_packed,
                                     moe_stream_t stream);

/* Gradients written by moe_layer_backward (device pointers; fp32 weights' gradients). */
typedef struct {
  void* dx;       /* [S, M] in the layer's element type                                   */
  float* dW_g;    /* [E, M]                                                                */
  float* dbias;   /* [E], nullable (the gradient of a per-expert logit offset)            */
  float* dW_in;   /* [E, H, M]                                                             */
  float* dW_up;   /* [E, H, M] (SwiGLU), else NULL                                         */
  float* dW_out;  /* [E, M, H]                                                             */
  float* dWs_in;  /* [n_shared * H_shared, M] (shared experts side by side), or NULL       */
  float* dWs_up;  /* [n_shared * H_shared, M] (SwiGLU), or NULL                            */
  float* dWs_out; /* [M, n_shared * H_shared], or NULL                                     */
} moe_grads_t;

/*
 * The backward pass of moe_layer_forward: the gradients of
 *     L = sum(dy * y) + aux_coef * aux_loss + z_coef * z_loss
 * (dy [S, M] the upstream gradient of y; MegaBlocks router §3: the load-balancing loss
 * reaches the router only through the expert scores, its counts being constants; §2:
 * z-loss) with the routing decisions held fixed. A dropped assignment gives its gate no
 * gradient. Every gate normalisation (MOE_GATE_*); uniform assignment (ids that do not come
 * from the logits) gives MOE_ERR_UNSUPPORTED. bf16 and fp32 layers.
 * Inputs from the forward: logits (the forward's logits_out, [S, E]), r (its routing
 * outputs) and fwd_ws (the MOE_WS_LAYER workspace of that moe_layer_forward call,
 * unchanged since: it holds x_perm, h and the shared experts' h). residual: 1 if the
 * forward had a residual (dx then includes dy). Packs: W_in_packed / Ws_in_packed from
 * the forward pack calls (the SwiGLU pre-activations are recomputed), the transposed packs
 * from moe_pack_weights_backward / moe_pack_shared_weights_backward (shared ones NULL
 * without shared experts). ws: MOE_WS_BACKWARD bytes (its own status word).
 * Every step runs on the GPU: gather of dy, GEMM 2's data gradient with the gate's
 * gradient, the SwiGLU derivative, GEMM 1's data gradient (tcgen05); the weights'
 * gradients as K-ragged tcgen05 GEMMs over per-expert 64-padded transposed rows; the
 * router's gradient (dlogits, then dx, dW_g, dbias); dx summed in fp32 and rounded once.
 * fp32 layers (the small-layer path) take the same steps on plain FMA, one thread an
 * output element, every sum (over d_model, d_ff, an expert's rows, the experts or the
 * tokens) in a fixed order.
 */
int moe_layer_backward(const moe_config_t* cfg, const void* x, const void* dy, const void* W_g,
                       const void* W_in_packed, const void* Wt_in_packed, const void* Wt_out_packed,
                       const void* Ws_in_packed, const void* Wst_in_packed,
                       const void* Wst_out_packed, const float* logits, const moe_route_out_t* r,
                       const void* fwd_ws, size_t fwd_ws_bytes, int residual, float aux_coef,
                       float z_coef, const moe_grads_t* grads, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/*
 * Synchronises `stream`, reads the status word in ws, clears it, and returns MOE_OK or
 * the device error recorded since the last call (MOE_ERR_TIMEOUT, MOE_ERR_NONFINITE or
 * MOE_ERR_DEVICE_DATA; MOE_ERR_CUDA if the synchronisation itself failed).
 */
int moe_get_device_status(void* ws, moe_stream_t stream);

/*
 * Sets, in the header of workspace ws (DEVICE pointer, 256-byte aligned), how long a
 * kernel launched with that workspace waits for an event of its own pipeline (a TMA load
 * landing, an MMA finishing, an accumulator being freed) before it gives up: limit_ns
 * nanoseconds, or the default of 2 s when limit_ns is 0 (a zero-filled header). A kernel
 * that gives up stops issuing work, lets the loads and MMAs it already issued finish,
 * frees its tensor memory and returns early; its outputs are then undefined and
 * moe_get_device_status reports MOE_ERR_TIMEOUT. Waits for work already issued are not
 * shortened. Not from the pages: a guard that keeps a stalled pipeline from holding the GPU
 * (the 2 s default), and with a tiny limit a way to exercise that path.
 * Stream-ordered: kernels enqueued on `stream` after this call see the new limit. Returns
 * MOE_ERR_INVALID_ARG for a null or misaligned ws, MOE_ERR_CUDA if the copy fails.
 */
int moe_set_wait_limit(void* ws, uint64_t limit_ns, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* TOP_GATING_EXPERT_GB300_MOE_H */
