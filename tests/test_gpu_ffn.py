"""GPU parity of dispatch, the grouped expert GEMMs, the shared experts and combine, element
by element against the oracle at sizes that span many tiles, every N-tile width the GEMM
instantiates, ragged expert segments and ragged M tails."""

import zlib

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from gpu_util import (LOSS_RTOL, RTOL, LOGIT_RTOL, assert_close, compare_route, oracle_cfg, route_np,
                      to_np)
from top_gating_expert_gb300 import _native as N
from top_gating_expert_gb300 import moe
from top_gating_expert_gb300.inputs import make_inputs, preset

pytestmark = pytest.mark.gpu


def _cfg(**kw):
    base = dict(S=4096, G=1, E=8, M=512, H=2048, k=2, capacity_factor=0.0, random_routing=0,
                n_shared=0, H_shared=0, act="relu", dtype="bf16", bias=False)
    base.update(kw)
    return base


CASES = {
    # BN 256 (GEMM1 and GEMM2), dropless, K = 512 -> 8 k-blocks (ring wraps twice)
    "relu_E8_dropless": _cfg(),
    # SwiGLU (BN 256 packed), GEMM2 N = 384 -> BN 128; capacity + random routing; 2 groups
    "swiglu_E6_capacity_rr": _cfg(S=3000, G=2, E=6, M=384, H=640, capacity_factor=1.0,
                                  random_routing=1, act="swiglu"),
    # BN 64 on both GEMMs, k = 4, skewed bias so some experts are nearly empty
    "relu_E16_k4_bn64": _cfg(S=2500, E=16, M=192, H=320, k=4, capacity_factor=1.25, bias=True),
    # shared experts (dense segment) + routed SwiGLU, k = 6
    "shared_swiglu_k6": _cfg(S=2048, E=16, M=256, H=256, k=6, act="swiglu", n_shared=2,
                             H_shared=192),
    # the fused router with E = 64, k = 2 over 24 chunks (2 groups of 1500 tokens, the last
    # chunk of each group ragged), random routing and capacity
    "relu_E64_router_pairs": _cfg(S=3000, G=2, E=64, M=512, H=512, capacity_factor=1.0,
                                  random_routing=1),
    # the fp32 path (plain FMA), tiny GShard top-2 with random routing
    "f32_tiny": preset(1),
    "f32_swiglu_shared": _cfg(S=200, G=2, E=4, M=32, H=128, k=2, capacity_factor=1.0,
                              act="swiglu", dtype="f32", n_shared=1, H_shared=128),
}


@pytest.fixture(scope="module", params=sorted(CASES))
def run(request, native_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    name = request.param
    cfg = CASES[name]
    inp = make_inputs(cfg, seed=zlib.crc32(name.encode()) % 10000)
    dev = "cuda"
    d = {k: v.to(dev) for k, v in inp.host.items()}
    R_max = moe.rows_max(cfg)
    dt = moe.torch_dtype(cfg)
    ws = moe.workspace(cfg, N.MOE_WS_STEP, dev)
    out = moe.RouteOutputs.allocate(cfg, dev)
    logits = torch.empty((cfg["S"], cfg["E"]), dtype=torch.float32, device=dev)
    # the router and routing as the layer runs them (bf16: one fused kernel + scan + finalize)
    moe.router_route(cfg, d["x"], d["W_g"], d.get("bias"), d["u"] if cfg["random_routing"] else None,
                     logits, out, ws)
    x_perm = torch.full((R_max, cfg["M"]), float("nan"), dtype=dt, device=dev)
    moe.dispatch(cfg, d["x"], out, x_perm)
    W_in_p, W_out_p = moe.pack_weights(cfg, d["W_in"], d.get("W_up"), d["W_out"])
    h_perm = torch.full((R_max, cfg["H"]), float("nan"), dtype=dt, device=dev)
    y_perm = torch.full((R_max, cfg["M"]), float("nan"), dtype=dt, device=dev)
    moe.expert_up(cfg, x_perm, out.expert_offsets, W_in_p, h_perm, ws)
    moe.expert_down(cfg, h_perm, out.expert_offsets, out.w_perm, W_out_p, y_perm, ws)
    shared_out = None
    if cfg["n_shared"]:
        ps_in, ps_out = moe.pack_shared_weights(cfg, d["Ws_in"], d.get("Ws_up"), d["Ws_out"])
        h_sh = torch.empty((cfg["S"], cfg["n_shared"] * cfg["H_shared"]), dtype=dt, device=dev)
        shared_out = torch.empty((cfg["S"], cfg["M"]), dtype=dt, device=dev)
        moe.shared_ffn(cfg, d["x"], ps_in, ps_out, h_sh, shared_out, ws)
    y = torch.empty((cfg["S"], cfg["M"]), dtype=dt, device=dev)
    moe.combine(cfg, y_perm, out, shared_out, None, y)
    y_res = torch.empty_like(y)
    moe.combine(cfg, y_perm, out, shared_out, d["x"], y_res)
    status = moe.device_status(ws)
    return dict(name=name, cfg=cfg, inp=inp, logits=to_np(logits), route=route_np(out),
                x_perm=to_np(x_perm), h_perm=to_np(h_perm), y_perm=to_np(y_perm),
                shared_out=None if shared_out is None else to_np(shared_out), y=to_np(y),
                y_res=to_np(y_res), status=status, dev=d, W_in_p=W_in_p, out=out, ws=ws)


def test_status_ok(run):
    assert run["status"] == 0


def test_router_logits(run):
    cfg, a = run["cfg"], run["inp"].np
    ref = O.router_logits(a["x"], a["W_g"], a.get("bias"))
    assert_close(run["logits"], ref, LOGIT_RTOL[cfg["dtype"]], "logits")


def test_route_bit_exact(run):
    cfg = run["cfg"]
    o = O.route(run["logits"], oracle_cfg(cfg), run["inp"].np["u"])
    compare_route(run["route"], o, run["name"])


def _same_route(g, want, what):
    R = int(want["expert_offsets"][-1])
    for key in ("expert_id", "gate", "pos", "drop_reason", "row", "counts", "counts_routed",
                "expert_offsets"):
        assert np.array_equal(g[key], want[key]), f"{what}: {key}"
    assert np.array_equal(g["token_of"][:R], want["token_of"][:R]), f"{what}: token_of"
    assert np.array_equal(g["w_perm"][:R], want["w_perm"][:R]), f"{what}: w_perm"
    for key in ("aux_loss", "z_loss"):
        a, b = float(g[key][0]), float(want[key][0])
        assert abs(a - b) <= LOSS_RTOL * abs(b) + 1e-7, (what, key, a, b)


def test_router_route_without_logits_out(run):
    """moe_router_route that keeps its logits on chip gives the same bits as the run that
    also stored them (the fixture's)."""
    cfg, d = run["cfg"], run["dev"]
    if cfg["dtype"] != "bf16":
        pytest.skip("the fp32 path needs logits_out")
    ws = moe.workspace(cfg, N.MOE_WS_STEP, "cuda")
    out = moe.RouteOutputs.allocate(cfg, "cuda")
    moe.router_route(cfg, d["x"], d["W_g"], d.get("bias"), d["u"] if cfg["random_routing"] else None,
                     None, out, ws)
    assert moe.device_status(ws) == 0
    _same_route(route_np(out), run["route"], run["name"])


def test_unfused_router_then_route(run):
    """The two separate steps (moe_router, then moe_route from the stored logits): logits
    within tolerance of the oracle's and bit-identical to the fused kernel's, routing
    bit-exact against the oracle routed from them and equal to the fused call's."""
    cfg, d, a = run["cfg"], run["dev"], run["inp"].np
    ws = moe.workspace(cfg, N.MOE_WS_STEP, "cuda")
    out = moe.RouteOutputs.allocate(cfg, "cuda")
    logits = torch.empty((cfg["S"], cfg["E"]), dtype=torch.float32, device="cuda")
    moe.router(cfg, d["x"], d["W_g"], d.get("bias"), logits, ws)
    moe.route(cfg, logits, d["u"] if cfg["random_routing"] else None, out, ws)
    assert moe.device_status(ws) == 0
    lg = to_np(logits)
    assert_close(lg, O.router_logits(a["x"], a["W_g"], a.get("bias")), LOGIT_RTOL[cfg["dtype"]],
                 "logits")
    assert np.array_equal(lg, run["logits"]), "logits differ from the fused kernel's"
    compare_route(route_np(out), O.route(lg, oracle_cfg(cfg), a["u"]), run["name"])
    _same_route(route_np(out), run["route"], run["name"])


def test_layer_without_logits_equals_with(run):
    """A layer that does not keep its logits (the benchmark's) computes the same step."""
    cfg, d = run["cfg"], run["dev"]
    if cfg["dtype"] != "bf16":
        pytest.skip("the fp32 path always materialises logits")
    layer = moe.MoeLayer(cfg, {k: run["inp"].host[k] for k in run["inp"].host}, keep_logits=False)
    y = layer.forward(d["x"], d["u"] if cfg["random_routing"] else None)
    assert moe.device_status(layer.ws) == 0
    assert layer.logits is None
    assert np.array_equal(to_np(y), run["y"])
    _same_route(route_np(layer.route_out), run["route"], run["name"])


def test_dispatch_exact(run):
    r = run["route"]
    R = int(r["expert_offsets"][-1])
    want = O.dispatch(run["inp"].np["x"], r["token_of"][:R])
    assert np.array_equal(run["x_perm"][:R], want)


def _expert_rows(run):
    cfg, a, r = run["cfg"], run["inp"].np, run["route"]
    off = r["expert_offsets"]
    for e in range(cfg["E"]):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi > lo:
            yield e, lo, hi, a["x"][r["token_of"][lo:hi]]


def test_expert_up_gemm(run):
    cfg, a = run["cfg"], run["inp"].np
    for e, lo, hi, xr in _expert_rows(run):
        A = O._f64(xr) @ O._f64(a["W_in"][e]).T
        if cfg["act"] == "relu":
            ref = np.maximum(A, 0)
        else:
            ref = A / (1 + np.exp(-A)) * (O._f64(xr) @ O._f64(a["W_up"][e]).T)
        assert_close(run["h_perm"][lo:hi], ref, RTOL[cfg["dtype"]], f"h expert {e}")


def test_expert_down_gemm(run):
    cfg, a, r = run["cfg"], run["inp"].np, run["route"]
    for e, lo, hi, xr in _expert_rows(run):
        W_up = a["W_up"][e] if cfg["act"] == "swiglu" else None
        ref = O.expert_ffn(xr, a["W_in"][e], a["W_out"][e], cfg["act"], W_up)
        ref = ref * r["w_perm"][lo:hi, None].astype(np.float64)
        assert_close(run["y_perm"][lo:hi], ref, RTOL[cfg["dtype"]], f"y_perm expert {e}")


def test_shared_experts(run):
    cfg, a = run["cfg"], run["inp"].np
    if not cfg["n_shared"]:
        pytest.skip("no shared experts")
    ref = O.shared_ffn(O._f64(a["x"]), a, cfg)
    assert_close(run["shared_out"], ref, RTOL[cfg["dtype"]], "shared_out")


def test_combine_is_exact_sum_of_gpu_rows(run):
    """combine alone: the fp32 sum of the GPU's own y_perm rows (+ shared, + residual),
    rounded once, equals the fp64 sum to within one rounding of the output type."""
    cfg, r = run["cfg"], run["route"]
    S = cfg["S"]
    ref = np.zeros((S, cfg["M"]))
    for j in range(cfg["k"]):
        rows = r["row"][:, j]
        keep = rows >= 0
        ref[keep] += run["y_perm"][rows[keep]]
    if run["shared_out"] is not None:
        ref += run["shared_out"]
    mag = np.zeros_like(ref)  # sum of |terms|: bounds the fp32 summation error
    for j in range(cfg["k"]):
        rows = r["row"][:, j]
        keep = rows >= 0
        mag[keep] += np.abs(run["y_perm"][rows[keep]])
    if run["shared_out"] is not None:
        mag += np.abs(run["shared_out"])
    ulp = 2.0 ** -8 if cfg["dtype"] == "bf16" else 2.0 ** -23  # output rounding, relative
    sum_err = (cfg["k"] + 3) * 2.0 ** -24
    err = np.abs(run["y"] - ref)
    assert np.all(err <= ulp * np.abs(ref) + sum_err * mag), err.max()
    dropped = np.all(r["row"] < 0, axis=1)
    if run["shared_out"] is None:
        assert np.all(run["y"][dropped] == 0)
    x = run["inp"].np["x"]
    ref_res = ref + x
    mag_res = mag + np.abs(x)
    assert np.all(np.abs(run["y_res"] - ref_res) <= ulp * np.abs(ref_res) + sum_err * mag_res)


def test_layer_output_vs_oracle(run):
    cfg = run["cfg"]
    y_ref, o, _ = O.layer_forward(run["inp"].np, oracle_cfg(cfg), logits=run["logits"])
    assert_close(run["y"], y_ref, RTOL[cfg["dtype"]], "y")
    y_ref_res = y_ref + O._f64(run["inp"].np["x"])
    assert_close(run["y_res"], y_ref_res, RTOL[cfg["dtype"]], "y + residual")


def test_layer_forward_equals_step_calls(run):
    """moe_layer_forward computes the step calls' results bit for bit (its last routing
    kernel also does the dispatch gather: same routing outputs, same x_perm rows, so the
    same y)."""
    cfg, d = run["cfg"], run["dev"]
    layer = moe.MoeLayer(cfg, {k: run["inp"].host[k] for k in run["inp"].host})
    y = layer.forward(d["x"], d["u"] if cfg["random_routing"] else None)
    assert moe.device_status(layer.ws) == 0
    _same_route(route_np(layer.route_out), run["route"], run["name"])
    assert np.array_equal(to_np(y), run["y"])
    assert np.array_equal(to_np(layer.logits), run["logits"])
    y2 = layer.forward(d["x"], d["u"] if cfg["random_routing"] else None, residual=d["x"])
    assert np.array_equal(to_np(y2), run["y_res"])


def test_graph_replay_equals_eager(run):
    """The whole forward captured as a CUDA graph gives the eager call's bits."""
    cfg, d = run["cfg"], run["dev"]
    layer = moe.MoeLayer(cfg, {k: run["inp"].host[k] for k in run["inp"].host})
    u = d["u"] if cfg["random_routing"] else None
    layer.capture(d["x"], u)
    layer.y.zero_()
    y = layer.replay()
    torch.cuda.synchronize()
    assert moe.device_status(layer.ws) == 0
    assert np.array_equal(to_np(y), run["y"])


@pytest.mark.parametrize("depth", [2, 3])
def test_host_pipeline_matches_eager(run, depth):
    """HostPipeline (pinned host in/out, two or three steps in flight) returns, step by step,
    the bits of the eager forward on the same inputs; five steps, so that every buffer set
    is reused."""
    cfg = run["cfg"]
    layer = moe.MoeLayer(cfg, {k: run["inp"].host[k] for k in run["inp"].host})
    rr = bool(cfg["random_routing"])
    pipe = moe.HostPipeline(layer, has_u=rr, depth=depth)
    x0 = run["inp"].host["x"]
    n = 5
    xs = [(x0 * (1.0 + 0.25 * i)).to(x0.dtype).pin_memory() for i in range(n)]
    u_host = run["inp"].host["u"].pin_memory() if rr else None
    ys = [torch.empty_like(x0).pin_memory() for _ in range(n)]
    losses = [torch.empty(2, dtype=torch.float32).pin_memory() for _ in range(n)]
    for i in range(n):
        pipe.submit(i, xs[i], u_host, ys[i], losses[i])
    torch.cuda.synchronize()
    assert moe.device_status(layer.ws) == 0
    for i in range(n):
        y = layer.forward(xs[i].cuda(), u_host.cuda() if rr else None)
        torch.cuda.synchronize()
        assert torch.equal(ys[i], y.cpu()), i
        assert losses[i][0].item() == layer.route_out.aux_loss.item()
        assert losses[i][1].item() == layer.route_out.z_loss.item()
