// The C ABI of include/moe.h: argument checks, workspace carving and the order of launches.
// Every check that can fail does so on the host, before anything is launched.
#include <algorithm>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "internal.h"

namespace moe {

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = getenv("MOE_PDL");
    return !(v && v[0] == '0');
  }();
  return on;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 1;
  return n;
}

namespace {

int validate(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->S < 1 || c->G < 1 || c->S % c->G != 0) return MOE_ERR_INVALID_ARG;
  if (c->E < 1 || c->E > 256) return MOE_ERR_INVALID_ARG;
  if (c->k < 1 || c->k > 8 || c->k > c->E) return MOE_ERR_INVALID_ARG;
  if (c->M < 1 || c->H < 1) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->act != MOE_ACT_RELU && c->act != MOE_ACT_SWIGLU) return MOE_ERR_INVALID_ARG;
  if (c->random_routing != 0 && c->random_routing != 1) return MOE_ERR_INVALID_ARG;
  if (c->random_routing && c->k != 2) return MOE_ERR_INVALID_ARG;
  if (!isfinite(c->capacity_factor)) return MOE_ERR_INVALID_ARG;
  if (c->n_shared < 0 || (c->n_shared > 0 && c->H_shared < 1)) return MOE_ERR_INVALID_ARG;
  if (c->gate_norm < MOE_GATE_SOFTMAX_TOPK || c->gate_norm > MOE_GATE_PNORM) return MOE_ERR_INVALID_ARG;
  if (c->gate_norm == MOE_GATE_PNORM && !(isfinite(c->gate_p) && c->gate_p > 0.f))
    return MOE_ERR_INVALID_ARG;
  if (c->n_expert_groups < 0 || c->n_expert_groups > 16) return MOE_ERR_INVALID_ARG;
  if (c->n_expert_groups > 1) {
    if (c->E % c->n_expert_groups) return MOE_ERR_INVALID_ARG;
    if (c->topk_groups < 1 || c->topk_groups > c->n_expert_groups) return MOE_ERR_INVALID_ARG;
    if (c->k > c->topk_groups * (c->E / c->n_expert_groups)) return MOE_ERR_INVALID_ARG;
  }
  if (c->uniform_assignment != 0 && c->uniform_assignment != 1) return MOE_ERR_INVALID_ARG;
  if (c->uniform_assignment && c->random_routing) return MOE_ERR_INVALID_ARG;
  if (int64_t(c->S) * c->k > INT32_MAX / 2) return MOE_ERR_UNSUPPORTED;
  const int64_t Hs = int64_t(c->n_shared) * c->H_shared;
  const bool swiglu = c->act == MOE_ACT_SWIGLU;
  if (c->dtype == MOE_BF16) {
    if (c->M % 64 || c->H % (swiglu ? 128 : 64)) return MOE_ERR_UNSUPPORTED;
    if (Hs % (swiglu ? 128 : 64)) return MOE_ERR_UNSUPPORTED;
  } else {
    if (c->M % 4 || c->H % 4) return MOE_ERR_UNSUPPORTED;  // 16-byte rows (copies, packing)
    if (swiglu && (c->H % 128 || Hs % 128)) return MOE_ERR_UNSUPPORTED;
    if (c->n_shared > 0 && c->H_shared % 4) return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

int capacity_of(const moe_config_t& c, int* C) {
  if (c.capacity_factor <= 0.f) {
    *C = -1;
    return MOE_OK;
  }
  const double v = ceil(double(c.capacity_factor) * c.k * (c.S / c.G) / c.E);
  if (!(v >= 1.0) || v > double(INT32_MAX)) return MOE_ERR_UNSUPPORTED;
  *C = int(v);
  return MOE_OK;
}

bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (!ws || !aligned256(ws)) return MOE_ERR_WORKSPACE;
  if (ws_bytes < need) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

int check_route_out(const moe_config_t& c, const moe_route_out_t* r) {
  if (!r || !r->expert_id || !r->gate || !r->pos || !r->drop_reason || !r->row || !r->counts ||
      !r->counts_routed || !r->expert_offsets || !r->token_of || !r->w_perm || !r->aux_loss ||
      !r->z_loss)
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

struct Prep {
  int C = -1;
  int64_t R_max = 0;
  WsLayout L;
};

int prepare(const moe_config_t* cfg, Prep* p) {
  int rc = validate(cfg);
  if (rc != MOE_OK) return rc;
  rc = capacity_of(*cfg, &p->C);
  if (rc != MOE_OK) return rc;
  p->R_max = rows_max(*cfg, p->C);
  p->L = ws_layout(*cfg, p->C);
  return MOE_OK;
}

unsigned* status_of(void* ws, const WsLayout& L) {
  return reinterpret_cast<unsigned*>(static_cast<char*>(ws) + L.status);
}

// GEMM 1 (+ activation) over `groups` row segments (offsets) or one dense segment.
int up_proj(const moe_config_t& c, const void* A, int64_t a_rows, const int32_t* offsets,
            int groups, int rows_dense, int H, const void* W_packed, void* h, unsigned* status,
            cudaStream_t st) {
  const bool swiglu = c.act == MOE_ACT_SWIGLU;
  if (c.dtype == MOE_F32)
    return launch_ffn_up_f32(c, H, static_cast<const float*>(A), offsets, groups, rows_dense,
                             a_rows, static_cast<const float*>(W_packed), static_cast<float*>(h),
                             status, st);
  GemmDesc d;
  d.epi = swiglu ? EPI_SWIGLU : EPI_RELU;
  d.A = A; d.a_rows = a_rows; d.K = c.M;
  d.N = swiglu ? 2 * H : H;
  d.B = W_packed; d.b_rows = int64_t(groups) * d.N; d.b_tiled = true;
  d.offsets = offsets; d.groups = groups; d.rows_dense = rows_dense;
  d.out = h; d.ldo = H;
  d.status = status;
  d.out_keep = true;  // GEMM 2 reads h next
  return launch_gemm_bf16(d, st);
}

// GEMM 2 (x row scale) over the same segments; W_out_packed from launch_pack_out.
int down_proj(const moe_config_t& c, const void* h, int64_t a_rows, const int32_t* offsets,
              int groups, int rows_dense, int H, const float* row_scale, const void* W_out_packed,
              void* y, unsigned* status, cudaStream_t st) {
  if (c.dtype == MOE_F32)
    return launch_ffn_down_f32(c, H, static_cast<const float*>(h), offsets, groups, rows_dense,
                               a_rows, row_scale, static_cast<const float*>(W_out_packed),
                               static_cast<float*>(y), status, st);
  GemmDesc d;
  d.epi = EPI_SCALE;
  d.A = h; d.a_rows = a_rows; d.K = H;
  d.N = c.M;
  d.B = W_out_packed; d.b_rows = int64_t(groups) * c.M; d.b_tiled = true;
  d.offsets = offsets; d.groups = groups; d.rows_dense = rows_dense;
  d.out = y; d.ldo = c.M;
  d.row_scale = row_scale;
  d.status = status;
  d.reverse = offsets != nullptr;  // h's last rows (GEMM 1's last tiles) first
  d.out_keep = true;               // the combine reads y_perm next
  return launch_gemm_bf16(d, st);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument (shape, divisibility, null pointer)";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: valid configuration not supported by this build";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace too small or not 256-byte aligned";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call or kernel launch failed";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a bounded device wait ran out";
    case MOE_ERR_NONFINITE: return "MOE_ERR_NONFINITE: non-finite router logits";
    case MOE_ERR_DEVICE_DATA: return "MOE_ERR_DEVICE_DATA: invalid index or offset on the device";
  }
  return "unknown status";
}

int moe_abi_version(void) { return 102; }

int moe_validate_config(const moe_config_t* cfg) {
  Prep p;
  return prepare(cfg, &p);
}

int moe_capacity(const moe_config_t* cfg, int32_t* C) {
  if (!C) return MOE_ERR_INVALID_ARG;
  Prep p;
  const int rc = prepare(cfg, &p);
  if (rc == MOE_OK) *C = p.C;
  return rc;
}

int moe_rows_max(const moe_config_t* cfg, int64_t* R_max) {
  if (!R_max) return MOE_ERR_INVALID_ARG;
  Prep p;
  const int rc = prepare(cfg, &p);
  if (rc == MOE_OK) *R_max = p.R_max;
  return rc;
}

int moe_workspace_bytes(const moe_config_t* cfg, int kind, size_t* bytes) {
  if (!bytes || (kind != MOE_WS_STEP && kind != MOE_WS_LAYER && kind != MOE_WS_BACKWARD))
    return MOE_ERR_INVALID_ARG;
  Prep p;
  const int rc = prepare(cfg, &p);
  if (rc == MOE_OK)
    *bytes = kind == MOE_WS_STEP ? p.L.step_bytes
             : kind == MOE_WS_LAYER ? p.L.layer_bytes
                                    : ws_layout_bwd(*cfg, p.C).bytes;
  return rc;
}

int moe_packed_sizes(const moe_config_t* cfg, int64_t* w_in_packed, int64_t* w_out_packed,
                     int64_t* ws_in_packed, int64_t* ws_out_packed) {
  Prep p;
  const int rc = prepare(cfg, &p);
  if (rc != MOE_OK) return rc;
  const int64_t f = cfg->act == MOE_ACT_SWIGLU ? 2 : 1;
  const int64_t Hs = int64_t(cfg->n_shared) * cfg->H_shared;
  if (w_in_packed) *w_in_packed = int64_t(cfg->E) * f * cfg->H * cfg->M;
  if (w_out_packed) *w_out_packed = int64_t(cfg->E) * cfg->M * cfg->H;
  if (ws_in_packed) *ws_in_packed = f * Hs * cfg->M;
  if (ws_out_packed) *ws_out_packed = Hs * cfg->M;
  return MOE_OK;
}

int moe_pack_weights(const moe_config_t* cfg, const void* W_in, const void* W_up, const void* W_out,
                     void* W_in_packed, void* W_out_packed, moe_stream_t stream) {
  Prep p;
  int rc = prepare(cfg, &p);
  if (rc != MOE_OK) return rc;
  const bool swiglu = cfg->act == MOE_ACT_SWIGLU;
  if (!W_in || !W_out || !W_in_packed || !W_out_packed || (swiglu && !W_up))
    return MOE_ERR_INVALID_ARG;
  if (W_in_packed == W_in || W_in_packed == W_up || W_out_packed == W_out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(W_in) || !aligned16(W_out) || !aligned16(W_in_packed) || !aligned16(W_out_packed) ||
      (swiglu && !aligned16(W_up)))
    return MOE_ERR_INVALID_ARG;
  rc = launch_pack_in(*cfg, cfg->E, cfg->H, W_in, W_up, W_in_packed, stream);
  if (rc != MOE_OK) return rc;
  return launch_pack_out(*cfg, cfg->E, cfg->H, 1, W_out, W_out_packed, stream);
}

int moe_pack_shared_weights(const moe_config_t* cfg, const void* Ws_in, const void* Ws_up,
                            const void* Ws_out, void* Ws_in_packed, void* Ws_out_packed,
                            moe_stream_t stream) {
  Prep p;
  int rc = prepare(cfg, &p);
  if (rc != MOE_OK) return rc;
  if (cfg->n_shared < 1) return MOE_ERR_INVALID_ARG;
  const bool swiglu = cfg->act == MOE_ACT_SWIGLU;
  if (!Ws_in || !Ws_out || !Ws_in_packed || !Ws_out_packed || (swiglu && !Ws_up))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(Ws_in) || !aligned16(Ws_out) || !aligned16(Ws_in_packed) ||
      !aligned16(Ws_out_packed) || (swiglu && !aligned16(Ws_up)))
    return MOE_ERR_INVALID_ARG;
  rc = launch_pack_in(*cfg, 1, cfg->n_shared * cfg->H_shared, Ws_in, Ws_up, Ws_in_packed, stream);
  if (rc != MOE_OK) return rc;
  return launch_pack_out(*cfg, 1, cfg->H_shared, cfg->n_shared, Ws_out, Ws_out_packed, stream);
}

int moe_router(const moe_config_t* cfg, const void* x, const void* W_g, const float* bias,
               float* logits, void* ws, size_t ws_bytes, moe_stream_t stream) {
  Prep p;
  int rc = prepare(cfg, &p);
  if (rc != MOE_OK) return rc;
  if (!x || !W_g || !logits) return MOE_ERR_INVALID_ARG;
  if ((rc = check_ws(ws, ws_bytes, p.L.step_bytes)) != MOE_OK) return rc;
  if (cfg->dtype == MOE_F32)
    return launch_router_f32(*cfg, static_cast<const float*>(x), static_cast<const float*>(W_g),
                             bias, logits, stream);
  GemmDesc d;
  d.epi = EPI_F32_BIAS;
  d.A = x; d.a_rows = cfg->S; d.K = cfg->M;
  d.B = W_g; d.b_rows = cfg->E; d.N = cfg->E;
  d.offsets = nullptr; d.groups = 1; d.rows_dense = cfg->S;
  d.out = logits; d.ldo = cfg->E;
  d.bias = bias; d.n_valid = cfg->E;
  d.status = status_of(ws, p.L);
  return launch_gemm_bf16(d, stream);
}

int moe_route(const moe_config_t* cfg, const float* logits, const float* u,
              const moe_route_out_t* out, void* ws, size_t ws_bytes, moe_stream_t stream) {
  Prep p;
  int rc = prepare(cfg, &p);
  if (rc != MOE_OK) return rc;
  if (!logits || (cfg->random_routing && !u)) return MOE_ERR_INVALID_ARG;
  if ((rc = check_route_out(*cfg, out)) != MOE_OK) return rc;
  if ((rc = check_ws(ws, ws_bytes, p.L.step_bytes)) != MOE_OK) return rc;
  return launch_route(*cfg, p.C, logits, cfg->random_routing ? u : nullptr, *out,
                      static_cast<char*>(ws), p.L, stream);
}

namespace {
// moe_router_route, optionally with the dispatch gather fused into its last kernel
int router_route(const moe_config_t* cfg, const void* x, const void* W_g, const float* bias,
                 const float* u, float* logits_out, const moe_route_out_t* out, void* ws,
                 size_t ws_bytes, const DispatchFuse* d, moe_stream_t stream) {
  Prep p;
  int rc = prepare(cfg, &p);
  if (rc != MOE_OK) return rc;
  if (!x || !W_g || (cfg->random_routing && !u)) return MOE_ERR_INVALID_ARG;
  if (cfg->dtype == MOE_F32 && !logits_out) return MOE_ERR_INVALID_ARG;
  if ((rc = check_route_out(*cfg, out)) != MOE_OK) return rc;
  if ((rc = check_ws(ws, ws_bytes, p.L.step_bytes)) != MOE_OK) return rc;
  if (d && (!d->x_perm || !aligned16(d->x) || !aligned16(d->x_perm))) return MOE_ERR_INVALID_ARG;
  char* w = static_cast<char*>(ws);
  if (cfg->dtype == MOE_F32) {
    if ((rc = moe_router(cfg, x, W_g, bias, logits_out, ws, ws_bytes, stream)) != MOE_OK) return rc;
    return launch_route(*cfg, p.C, logits_out, cfg->random_routing ? u : nullptr, *out, w, p.L,
                        stream, d);
  }
  if (logits_out && !aligned16(logits_out)) return MOE_ERR_INVALID_ARG;
  return launch_router_route(*cfg, p.C, x, W_g, bias, cfg->random_routing ? u : nullptr,
                             logits_out, *out, w, p.L, stream, d);
}
}  // namespace

int moe_router_route(const moe_config_t* cfg, const void* x, const void* W_g, const float* bias,
                     const float* u, float* logits_out, const moe_route_out_t* out, void* ws,
                     size_t ws_bytes, moe_stream_t stream) {
  return router_route(cfg, x, W_g, bias, u, logits_out, out, ws, ws_bytes, nullptr, stream);
}

int moe_dispatch(const moe_config_t* cfg, const void* x, const moe_route_out_t* r, void* x_perm,
                 moe_stream_t stream) {
  Prep p;
  int rc = prepare(cfg, &p);
  if (rc != MOE_OK) return rc;
  if (!x || !x_perm || !r || !r->token_of || !r->expert_offsets) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_INVALID_ARG;
  return launch_dispatch(*cfg, p.R_max, x, r->token_of, r->expert_offsets, x_perm, stream);
}

int moe_expert_up(const moe_config_t* cfg, const void* x_perm, const int32_t* expert_offsets,
                  const void* W_in_packed, void* h_perm, void* ws, size_t ws_bytes,
                  moe_stream_t stream) {
  Prep p;
  int rc = prepare(cfg, &p);
  if (rc != MOE_OK) return rc;
  if (!x_perm || !expert_offsets || !W_in_packed || !h_perm) return MOE_ERR_INVALID_ARG;
  if ((rc = check_ws(ws, ws_bytes, p.L.step_bytes)) != MOE_OK) return rc;
  return up_proj(*cfg, x_perm, p.R_max, expert_offsets, cfg->E, 0, cfg->H, W_in_packed, h_perm,
                 status_of(ws, p.L), stream);
}

int moe_expert_down(const moe_config_t* cfg, const void* h_perm, const int32_t* expert_offsets,
                    const float* w_perm, const void* W_out_packed, void* y_perm, void* ws,
                    size_t ws_bytes, moe_stream_t stream) {
  Prep p;
  int rc = prepare(cfg, &p);
  if (rc != MOE_OK) return rc;
  if (!h_perm || !expert_offsets || !w_perm || !W_out_packed || !y_perm) return MOE_ERR_INVALID_ARG;
  if ((rc = check_ws(ws, ws_bytes, p.L.step_bytes)) != MOE_OK) return rc;
  return down_proj(*cfg, h_perm, p.R_max, expert_offsets, cfg->E, 0, cfg->H, w_perm, W_out_packed,
                   y_perm, status_of(ws, p.L), stream);
}

int moe_expert_ffn(const moe_config_t* cfg, const void* x_perm, const int32_t* expert_offsets,
                   const float* w_perm, const void* W_in_packed, const void* W_out_packed,
                   void* h_perm, void* y_perm, void* ws, size_t ws_bytes, moe_stream_t stream) {
  int rc = moe_expert_up(cfg, x_perm, expert_offsets, W_in_packed, h_perm, ws, ws_bytes, stream);
  if (rc != MOE_OK) return rc;
  return moe_expert_down(cfg, h_perm, expert_offsets, w_perm, W_out_packed, y_perm, ws, ws_bytes,
                         stream);
}

int moe_shared_ffn(const moe_config_t* cfg, const void* x, const void* Ws_in_packed,
                   const void* Ws_out_packed, void* h_shared, void* shared_out, void* ws,
                   size_t ws_bytes, moe_stream_t stream) {
  Prep p;
  int rc = prepare(cfg, &p);
  if (rc != MOE_OK) return rc;
  if (cfg->n_shared < 1) return MOE_ERR_INVALID_ARG;
  if (!x || !Ws_in_packed || !Ws_out_packed || !h_shared || !shared_out) return MOE_ERR_INVALID_ARG;
  if ((rc = check_ws(ws, ws_bytes, p.L.step_bytes)) != MOE_OK) return rc;
  const int Hc = cfg->n_shared * cfg->H_shared;
  unsigned* st = status_of(ws, p.L);
  rc = up_proj(*cfg, x, cfg->S, nullptr, 1, cfg->S, Hc, Ws_in_packed, h_shared, st, stream);
  if (rc != MOE_OK) return rc;
  return down_proj(*cfg, h_shared, cfg->S, nullptr, 1, cfg->S, Hc, nullptr, Ws_out_packed,
                   shared_out, st, stream);
}

int moe_combine(const moe_config_t* cfg, const void* y_perm, const moe_route_out_t* r,
                const void* shared_out, const void* residual, void* y, moe_stream_t stream) {
  Prep p;
  int rc = prepare(cfg, &p);
  if (rc != MOE_OK) return rc;
  if (!y_perm || !r || !r->row || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(y) || (shared_out && !aligned16(shared_out)) ||
      (residual && !aligned16(residual)))
    return MOE_ERR_INVALID_ARG;
  return launch_combine(*cfg, y_perm, r->row, shared_out, residual, y, p.R_max, stream);
}

int moe_layer_forward(const moe_config_t* cfg, const void* x, const void* W_g, const float* bias,
                      const void* W_in_packed, const void* W_out_packed, const void* Ws_in_packed,
                      const void* Ws_out_packed, const float* u, const void* residual, void* y,
                      float* logits_out, const moe_route_out_t* r, void* ws, size_t ws_bytes,
                      moe_stream_t stream) {
  Prep p;
  int rc = prepare(cfg, &p);
  if (rc != MOE_OK) return rc;
  if (!x || !W_g || !W_in_packed || !W_out_packed || !y) return MOE_ERR_INVALID_ARG;
  if (cfg->n_shared > 0 && (!Ws_in_packed || !Ws_out_packed)) return MOE_ERR_INVALID_ARG;
  if ((rc = check_route_out(*cfg, r)) != MOE_OK) return rc;
  if ((rc = check_ws(ws, ws_bytes, p.L.layer_bytes)) != MOE_OK) return rc;
  char* w = static_cast<char*>(ws);
  float* logits = logits_out;
  void* x_perm = w + p.L.x_perm;
  void* h_perm = w + p.L.h_perm;
  void* y_perm = w + p.L.y_perm;
  void* shared_out = cfg->n_shared > 0 ? static_cast<void*>(w + p.L.s_out) : nullptr;
  if (cfg->dtype == MOE_F32 && !logits) logits = reinterpret_cast<float*>(w + p.L.logits);
  // routing's last kernel also writes x_perm, and brings GEMM 1's first wave of weight
  // tiles (one BN x M tile per CTA pair, at most 40 MB) into L2 while the routing finishes
  DispatchFuse fuse{x, x_perm, nullptr, 0, nullptr, 0};
  if (cfg->dtype == MOE_BF16) {
    fuse.h_tail = h_perm;  // zero rows past the kept ones, read by the backward
    fuse.h_cols = cfg->H;
    const bool sw = cfg->act == MOE_ACT_SWIGLU;
    const int64_t n1 = sw ? 2 * int64_t(cfg->H) : cfg->H;
    const int64_t bn = gemm_bn(int(n1), sw ? EPI_SWIGLU : EPI_RELU);
    int64_t pf = int64_t(num_sms() / 2) * bn * cfg->M * 2;
    pf = std::min<int64_t>({pf, int64_t(cfg->E) * n1 * cfg->M * 2, int64_t(40) << 20});
    fuse.prefetch = W_in_packed;
    fuse.prefetch_bytes = pf;
  }
  if ((rc = router_route(cfg, x, W_g, bias, u, logits, r, ws, ws_bytes, &fuse, stream)) != MOE_OK)
    return rc;
  if ((rc = moe_expert_ffn(cfg, x_perm, r->expert_offsets, r->w_perm, W_in_packed, W_out_packed,
                           h_perm, y_perm, ws, ws_bytes, stream)) != MOE_OK)
    return rc;
  if (cfg->n_shared > 0 &&
      (rc = moe_shared_ffn(cfg, x, Ws_in_packed, Ws_out_packed, w + p.L.h_shared, shared_out, ws,
                           ws_bytes, stream)) != MOE_OK)
    return rc;
  return moe_combine(cfg, y_perm, r, shared_out, residual, y, stream);
}

int moe_pack_weights_backward(const moe_config_t* cfg, const void* W_in, const void* W_up,
                              const void* W_out, void* Wt_in_packed, void* Wt_out_packed,
                              moe_stream_t stream) {
  Prep p;
  int rc = prepare(cfg, &p);
  if (rc != MOE_OK) return rc;
  const bool sw = cfg->act == MOE_ACT_SWIGLU;
  if (!W_in || !W_out || !Wt_in_packed || !Wt_out_packed || (sw && !W_up)) return MOE_ERR_INVALID_ARG;
  // fp32: the same transposes, row-major (the plain-FMA kernels read them a row a thread)
  auto pack = cfg->dtype == MOE_BF16 ? launch_pack_transposed : launch_pack_transposed_f32;
  rc = pack(0, 0, cfg->E, cfg->H, cfg->M, cfg->M, cfg->H, 1, W_out, nullptr, Wt_out_packed, stream);
  if (rc != MOE_OK) return rc;
  return pack(1, sw, cfg->E, cfg->M, sw ? 2 * cfg->H : cfg->H, cfg->M, cfg->H, 1, W_in, W_up,
              Wt_in_packed, stream);
}

int moe_pack_shared_weights_backward(const moe_config_t* cfg, const void* Ws_in, const void* Ws_up,
                                     const void* Ws_out, void* Wst_in_packed, void* Wst_out_packed,
                                     moe_stream_t stream) {
  Prep p;
  int rc = prepare(cfg, &p);
  if (rc != MOE_OK) return rc;
  if (cfg->n_shared < 1) return MOE_ERR_INVALID_ARG;
  const bool sw = cfg->act == MOE_ACT_SWIGLU;
  if (!Ws_in || !Ws_out || !Wst_in_packed || !Wst_out_packed || (sw && !Ws_up))
    return MOE_ERR_INVALID_ARG;
  const int Hc = cfg->n_shared * cfg->H_shared;
  auto pack = cfg->dtype == MOE_BF16 ? launch_pack_transposed : launch_pack_transposed_f32;
  rc = pack(0, 0, 1, Hc, cfg->M, cfg->M, cfg->H_shared, cfg->n_shared, Ws_out, nullptr,
            Wst_out_packed, stream);
  if (rc != MOE_OK) return rc;
  return pack(1, sw, 1, cfg->M, sw ? 2 * Hc : Hc, cfg->M, Hc, 1, Ws_in, Ws_up, Wst_in_packed,
              stream);
}

// One expert FFN's backward on (ragged or dense) row segments, the steps moe_layer_backward
// runs for the routed experts and again for the shared ones.
struct FfnBwd {
  const void* x_rows;   // forward A rows (x_perm, or x for the dense shared segment)
  int64_t rows_cap;     // rows of x_rows / the segment buffers
  const int32_t* offsets;  // ragged segments (null: one dense segment of dense_rows)
  int groups, dense_rows;
  int Hn;               // hidden units of one group
  const void* W_in_packed;  // forward pack (SwiGLU recompute)
  const void* Wt_in_packed;
  const void* Wt_out_packed;
  const void* dy_rows;  // [rows_cap, M] upstream gradient rows
  const float* w;       // per-row gate (null: 1)
  const void* h;        // forward hidden [rows_cap, Hn]
  void* dh;             // SwiGLU scratch [rows_cap, Hn]
  void* dab;            // [rows_cap, F]
  float* gpart;         // nullable
  void* dx_rows;        // [rows_cap, M]
};

int ffn_backward_data(const moe_config_t& c, const FfnBwd& f, unsigned* status, cudaStream_t st) {
  const bool sw = c.act == MOE_ACT_SWIGLU;
  const int64_t F = sw ? 2 * int64_t(f.Hn) : f.Hn;
  GemmDesc d;  // gradient through GEMM 2 (and the ReLU mask, the gate's gradient)
  d.epi = EPI_DGRAD2;
  d.A = f.dy_rows; d.a_rows = f.rows_cap; d.K = c.M;
  d.B = f.Wt_out_packed; d.N = f.Hn; d.b_rows = int64_t(f.groups) * f.Hn; d.b_tiled = true;
  d.offsets = f.offsets; d.groups = f.groups; d.rows_dense = f.dense_rows;
  d.out = sw ? f.dh : f.dab; d.ldo = f.Hn;
  d.row_scale = f.w; d.aux = f.h; d.ld_aux = f.Hn; d.gpart = f.gpart; d.relu = sw ? 0 : 1;
  d.out_keep = !sw;  // ReLU: GEMM 1's data gradient reads da next
  d.status = status;
  int rc = launch_gemm_bf16(d, st);
  if (rc != MOE_OK) return rc;
  if (sw) {  // recompute the pre-activations, apply the SwiGLU derivative
    GemmDesc e;
    e.epi = EPI_SWIGLU_BWD;
    e.A = f.x_rows; e.a_rows = f.rows_cap; e.K = c.M;
    e.B = f.W_in_packed; e.N = 2 * f.Hn; e.b_rows = int64_t(f.groups) * 2 * f.Hn; e.b_tiled = true;
    e.offsets = f.offsets; e.groups = f.groups; e.rows_dense = f.dense_rows;
    e.out = f.dab; e.ldo = F; e.aux = f.dh; e.ld_aux = f.Hn;
    e.status = status;
    if ((rc = launch_gemm_bf16(e, st)) != MOE_OK) return rc;
  }
  GemmDesc g;  // gradient through GEMM 1
  g.epi = EPI_SCALE;
  g.A = f.dab; g.a_rows = f.rows_cap; g.K = int(F);
  g.B = f.Wt_in_packed; g.N = c.M; g.b_rows = int64_t(f.groups) * c.M; g.b_tiled = true;
  g.offsets = f.offsets; g.groups = f.groups; g.rows_dense = f.dense_rows;
  g.out = f.dx_rows; g.ldo = c.M;
  g.status = status;
  return launch_gemm_bf16(g, st);
}

// dW[g] (fp32 [c1][N]) = A_g . B_g^T over group g's padded K segment (A [c1][Kp], B [N][Kp]).
// dW[g] = A_g^T . B_g over K-row ranges, both operands row-major and read in place (MN-major
// tcgen05 operands): A [a_krows, c1], B [b_krows, N]; group g takes koffs[g+1] - koffs[g]
// rows (a multiple of 64) from row aoffs[g] of A and boffs[g] of B (null: koffs[g]). k_max:
// a bound on every group's range known to the caller (0: none).
int weight_grad_mn(const void* A, int64_t a_krows, const int32_t* aoffs, int c1, const void* B,
                   int64_t b_krows, const int32_t* boffs, int N, int64_t Kp, const int32_t* koffs,
                   int groups, float* out, float* out2, unsigned* status, cudaStream_t st,
                   int k_max = 0) {
  GemmDesc d;
  d.epi = EPI_F32_BIAS;
  d.mn = true;
  d.A = A; d.a_krows = a_krows; d.a_rows = c1; d.aoffs = aoffs; d.K = int(Kp);
  d.B = B; d.b_krows = b_krows; d.boffs = boffs; d.N = N; d.b_rows = N; d.b_tiled = false;
  d.koffs = koffs; d.c1 = c1; d.groups = groups;
  d.out = out; d.ldo = N; d.n_valid = N; d.out2 = out2;
  d.status = status;
  d.k_max = k_max;
  return launch_gemm_bf16(d, st);
}

// moe_layer_backward for fp32 layers: the bf16 path's steps on plain-FMA kernels
// (backward_f32.cu), with the transposed weights row-major and every sum in a fixed order.
int layer_backward_f32(const moe_config_t& c, const Prep& p, const void* x, const void* dy,
                       const void* W_g, const void* W_in_packed, const void* Wt_in_packed,
                       const void* Wt_out_packed, const void* Ws_in_packed,
                       const void* Wst_in_packed, const void* Wst_out_packed, const float* logits,
                       const moe_route_out_t& r, const char* fw, char* w, const WsLayoutBwd& B,
                       const RouterBwdBufs& rb, int residual, float aux_coef, float z_coef,
                       const moe_grads_t& grads, unsigned* status, cudaStream_t stream) {
  const bool sw = c.act == MOE_ACT_SWIGLU;
  const int64_t R = p.R_max;
  const int F = sw ? 2 * c.H : c.H;
  int rc;
  // routed experts: data gradients over the expert segments
  if ((rc = launch_dispatch(c, R, dy, r.token_of, r.expert_offsets, w + B.dy_perm, stream)) != MOE_OK)
    return rc;
  FfnBwdF32 f;
  f.x_rows = fw + p.L.x_perm; f.rows_cap = R; f.offsets = r.expert_offsets; f.groups = c.E;
  f.dense_rows = 0; f.M = c.M; f.Hn = c.H; f.swiglu = sw ? 1 : 0;
  f.W_in_packed = W_in_packed; f.Wt_in = Wt_in_packed; f.Wt_out = Wt_out_packed;
  f.dy_rows = w + B.dy_perm; f.w = r.w_perm; f.h = fw + p.L.h_perm; f.dh = w + B.dh;
  f.dab = w + B.dab; f.gpart = reinterpret_cast<float*>(w + B.gpart); f.n_tiles = B.n_tiles2;
  f.dx_rows = w + B.dx_perm;
  if ((rc = ffn_backward_data_f32(f, stream)) != MOE_OK) return rc;
  // routed experts: dW_out = (w dy)^T h, dW_in = da^T x (dW_up = db^T x), each expert's rows
  if ((rc = weight_grad_f32(w + B.dy_perm, c.M, r.w_perm, 0, fw + p.L.h_perm, c.H,
                            r.expert_offsets, c.E, 0, c.M, c.H, grads.dW_out, stream)) != MOE_OK)
    return rc;
  if ((rc = weight_grad_f32(w + B.dab, F, nullptr, sw ? 1 : 0, fw + p.L.x_perm, c.M,
                            r.expert_offsets, c.E, 0, c.H, c.M, grads.dW_in, stream)) != MOE_OK)
    return rc;
  if (sw && (rc = weight_grad_f32(w + B.dab, F, nullptr, 2, fw + p.L.x_perm, c.M, r.expert_offsets,
                                  c.E, 0, c.H, c.M, grads.dW_up, stream)) != MOE_OK)
    return rc;
  // the router: dlogits from the gates' gradients, aux and z; then dx, dW_g, dbias
  if ((rc = launch_router_backward(c, logits, r, reinterpret_cast<const float*>(w + B.gpart),
                                   B.n_tiles2, aux_coef, z_coef, rb, x, W_g, grads.dW_g,
                                   grads.dbias, status, stream)) != MOE_OK)
    return rc;
  // shared experts: one dense segment of all S tokens, weight 1
  void* dxs = nullptr;
  if (c.n_shared > 0) {
    const int Hc = c.n_shared * c.H_shared, Fs = sw ? 2 * Hc : Hc;
    FfnBwdF32 s;
    s.x_rows = x; s.rows_cap = c.S; s.offsets = nullptr; s.groups = 1; s.dense_rows = c.S;
    s.M = c.M; s.Hn = Hc; s.swiglu = sw ? 1 : 0;
    s.W_in_packed = Ws_in_packed; s.Wt_in = Wst_in_packed; s.Wt_out = Wst_out_packed;
    s.dy_rows = dy; s.w = nullptr; s.h = fw + p.L.h_shared; s.dh = w + B.dhs; s.dab = w + B.dabs;
    s.gpart = nullptr; s.n_tiles = 1; s.dx_rows = w + B.dxs;
    if ((rc = ffn_backward_data_f32(s, stream)) != MOE_OK) return rc;
    if ((rc = weight_grad_f32(dy, c.M, nullptr, 0, fw + p.L.h_shared, Hc, nullptr, 1, c.S, c.M,
                              Hc, grads.dWs_out, stream)) != MOE_OK)
      return rc;
    if ((rc = weight_grad_f32(w + B.dabs, Fs, nullptr, sw ? 1 : 0, x, c.M, nullptr, 1, c.S, Hc,
                              c.M, grads.dWs_in, stream)) != MOE_OK)
      return rc;
    if (sw && (rc = weight_grad_f32(w + B.dabs, Fs, nullptr, 2, x, c.M, nullptr, 1, c.S, Hc, c.M,
                                    grads.dWs_up, stream)) != MOE_OK)
      return rc;
    dxs = w + B.dxs;
  }
  // dx = sum over kept choices of the rows' gradients (+ shared) (+ dy) + the router's
  return launch_combine(c, w + B.dx_perm, r.row, dxs, residual ? dy : nullptr, grads.dx, R, stream,
                        rb.dx_r);
}

int moe_layer_backward(const moe_config_t* cfg, const void* x, const void* dy, const void* W_g,
                       const void* W_in_packed, const void* Wt_in_packed, const void* Wt_out_packed,
                       const void* Ws_in_packed, const void* Wst_in_packed,
                       const void* Wst_out_packed, const float* logits, const moe_route_out_t* r,
                       const void* fwd_ws, size_t fwd_ws_bytes, int residual, float aux_coef,
                       float z_coef, const moe_grads_t* grads, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
  Prep p;
  int rc = prepare(cfg, &p);
  if (rc != MOE_OK) return rc;
  const moe_config_t& c = *cfg;
  if (c.uniform_assignment) return MOE_ERR_UNSUPPORTED;
  if (c.E > 256) return MOE_ERR_UNSUPPORTED;
  const bool sw = c.act == MOE_ACT_SWIGLU;
  const bool shared = c.n_shared > 0;
  if (!x || !dy || !W_g || !Wt_in_packed || !Wt_out_packed || !logits || !grads || !fwd_ws)
    return MOE_ERR_INVALID_ARG;
  if (sw && !W_in_packed) return MOE_ERR_INVALID_ARG;
  if (!grads->dx || !grads->dW_g || !grads->dW_in || !grads->dW_out || (sw && !grads->dW_up))
    return MOE_ERR_INVALID_ARG;
  if (shared && (!Wst_in_packed || !Wst_out_packed || (sw && !Ws_in_packed) || !grads->dWs_in ||
                 !grads->dWs_out || (sw && !grads->dWs_up)))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(dy) || !aligned16(grads->dx)) return MOE_ERR_INVALID_ARG;
  if ((rc = check_route_out(c, r)) != MOE_OK) return rc;
  if ((rc = check_ws(const_cast<void*>(fwd_ws), fwd_ws_bytes, p.L.layer_bytes)) != MOE_OK) return rc;
  const WsLayoutBwd B = ws_layout_bwd(c, p.C);
  if ((rc = check_ws(ws, ws_bytes, B.bytes)) != MOE_OK) return rc;
  char* w = static_cast<char*>(ws);
  const char* fw = static_cast<const char*>(fwd_ws);
  unsigned* status = reinterpret_cast<unsigned*>(w + B.status);
  const int64_t R = p.R_max;
  const int F = sw ? 2 * c.H : c.H;
  // the router's buffers (its GEMMs' operands on the bf16 path)
  int32_t* poff_s = reinterpret_cast<int32_t*>(w + B.poff_s);
  RouterBwdBufs rb;
  rb.dlogits = reinterpret_cast<float*>(w + B.dlogits);
  rb.dlb = w + B.dlb; rb.wgT = w + B.wgT;
  rb.dx_r = reinterpret_cast<float*>(w + B.dx_r);
  rb.koff_e = reinterpret_cast<int32_t*>(w + B.koff_e); rb.koff_s = poff_s; rb.Sp = B.Sp;
  rb.koff_split = reinterpret_cast<int32_t*>(w + B.koff_split);
  rb.dwg_part = reinterpret_cast<float*>(w + B.dwg_part);
  rb.max_split = WsLayoutBwd::kMaxSplit;
  if (c.dtype == MOE_F32)
    return layer_backward_f32(c, p, x, dy, W_g, W_in_packed, Wt_in_packed, Wt_out_packed,
                              Ws_in_packed, Wst_in_packed, Wst_out_packed, logits, *r, fw, w, B,
                              rb, residual, aux_coef, z_coef, *grads, status, stream);

  // routed experts: data gradients (tcgen05 GEMMs over the expert segments)
  if ((rc = launch_dispatch(c, R, dy, r->token_of, r->expert_offsets, w + B.dy_perm, stream)) != MOE_OK)
    return rc;
  FfnBwd f;
  f.x_rows = fw + p.L.x_perm; f.rows_cap = R; f.offsets = r->expert_offsets; f.groups = c.E;
  f.dense_rows = 0; f.Hn = c.H; f.W_in_packed = W_in_packed; f.Wt_in_packed = Wt_in_packed;
  f.Wt_out_packed = Wt_out_packed; f.dy_rows = w + B.dy_perm; f.w = r->w_perm;
  f.h = fw + p.L.h_perm; f.dh = w + B.dh; f.dab = w + B.dab;
  f.gpart = reinterpret_cast<float*>(w + B.gpart); f.dx_rows = w + B.dx_perm;
  if ((rc = ffn_backward_data(c, f, status, stream)) != MOE_OK) return rc;
  // routed experts: weight gradients, K = the expert's rows padded to 64. dW_out = (w dy)^T h:
  // A = gate-scaled dy gathered into 64-padded segments (zero rows in the padding), B = h
  // read in place from the segment's first row (its rows past the segment are the next
  // expert's, or the 64 zeroed rows after the last: A's zeros cancel them). dW_in = da^T x:
  // A = da in place (64 rows past the last zeroed here), B = x gathered padded.
  int32_t* poff = reinterpret_cast<int32_t*>(w + B.poff);
  if ((rc = launch_pad_offsets(r->expert_offsets, c.E, 0, poff, stream)) != MOE_OK) return rc;
  if ((rc = launch_pad_gather(dy, c.M, r->token_of, r->w_perm, r->expert_offsets, poff, c.E, c.S,
                              B.Rp, w + B.wdyP, nullptr, 0, status, stream)) != MOE_OK)
    return rc;
  if ((rc = launch_pad_gather(x, c.M, r->token_of, nullptr, r->expert_offsets, poff, c.E, c.S,
                              B.Rp, w + B.xP, w + B.dab, F, status, stream)) != MOE_OK)
    return rc;
  // with a capacity, an expert keeps at most C rows of each of the G groups: its padded K
  // range is at most G C rounded up to 64
  const int64_t kcap = p.C > 0 ? (int64_t(c.G) * p.C + 63) / 64 * 64 : 0;
  const int k_max = kcap <= INT32_MAX ? int(kcap) : 0;
  if ((rc = weight_grad_mn(w + B.wdyP, B.Rp, nullptr, c.M, fw + p.L.h_perm, R + 64,
                           r->expert_offsets, c.H, B.Rp, poff, c.E, grads->dW_out, nullptr, status,
                           stream, k_max)) != MOE_OK)
    return rc;
  if ((rc = weight_grad_mn(w + B.dab, R + 64, r->expert_offsets, F, w + B.xP, B.Rp, nullptr, c.M,
                           B.Rp, poff, c.E, grads->dW_in, sw ? grads->dW_up : nullptr, status,
                           stream, k_max)) != MOE_OK)
    return rc;
  // K = all S tokens (padded to 64) for the router's dW_g and the shared experts: the tensors
  // end at row S, so the padding reads as zeros
  if ((rc = launch_pad_offsets(nullptr, 1, c.S, poff_s, stream)) != MOE_OK) return rc;
  // the router: dlogits from the gates' gradients, aux and z; then dx, dW_g (tcgen05), dbias
  if ((rc = launch_router_backward(c, logits, *r, reinterpret_cast<const float*>(w + B.gpart),
                                   B.n_tiles2, aux_coef, z_coef, rb, x, W_g, grads->dW_g,
                                   grads->dbias, status, stream)) != MOE_OK)
    return rc;
  // shared experts: one dense segment of all S tokens, weight 1
  void* dxs = nullptr;
  if (shared) {
    const int Hc = c.n_shared * c.H_shared, Fs = sw ? 2 * Hc : Hc;
    FfnBwd s;
    s.x_rows = x; s.rows_cap = c.S; s.offsets = nullptr; s.groups = 1; s.dense_rows = c.S;
    s.Hn = Hc; s.W_in_packed = Ws_in_packed; s.Wt_in_packed = Wst_in_packed;
    s.Wt_out_packed = Wst_out_packed; s.dy_rows = dy; s.w = nullptr; s.h = fw + p.L.h_shared;
    s.dh = w + B.dhs; s.dab = w + B.dabs; s.gpart = nullptr; s.dx_rows = w + B.dxs;
    if ((rc = ffn_backward_data(c, s, status, stream)) != MOE_OK) return rc;
    if ((rc = weight_grad_mn(dy, c.S, nullptr, c.M, fw + p.L.h_shared, c.S, nullptr, Hc, B.Sp,
                             poff_s, 1, grads->dWs_out, nullptr, status, stream)) != MOE_OK)
      return rc;
    if ((rc = weight_grad_mn(w + B.dabs, c.S, nullptr, Fs, x, c.S, nullptr, c.M, B.Sp, poff_s, 1,
                             grads->dWs_in, sw ? grads->dWs_up : nullptr, status, stream)) != MOE_OK)
      return rc;
    dxs = w + B.dxs;
  }
  // dx = sum over kept choices of the rows' gradients (+ shared) (+ dy) + the router's
  return launch_combine(c, w + B.dx_perm, r->row, dxs, residual ? dy : nullptr, grads->dx, R,
                        stream, reinterpret_cast<const float*>(w + B.dx_r));
}

int moe_set_wait_limit(void* ws, uint64_t limit_ns, moe_stream_t stream) {
  if (!ws || reinterpret_cast<uintptr_t>(ws) % 256 != 0) return MOE_ERR_INVALID_ARG;
  // bytes 8..15 of the header (the bounded waits read them where they would give up);
  // pageable source: the copy has taken the value by the time the call returns
  const uint64_t v = limit_ns;
  if (cudaMemcpyAsync(static_cast<char*>(ws) + kWaitLimitOffset, &v, sizeof(v),
                      cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

int moe_get_device_status(void* ws, moe_stream_t stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (word != 0 && cudaMemset(ws, 0, sizeof(word)) != cudaSuccess) return MOE_ERR_CUDA;
  if (word & kStatusTimeout) return MOE_ERR_TIMEOUT;
  if (word & kStatusNonfinite) return MOE_ERR_NONFINITE;
  if (word & kStatusDeviceData) return MOE_ERR_DEVICE_DATA;
  return MOE_OK;
}

}  // extern "C"
