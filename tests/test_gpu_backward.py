"""GPU parity of moe_layer_backward against the backward oracle (itself pinned by finite
differences): every gradient — dx, dW_g, dbias, the routed experts' and the shared experts'
weights — element by element, on layers that span several GEMM tiles, with capacity drops,
random routing, dropless top-3, shared SwiGLU experts, TopK(Softmax) and p-norm gates,
group-limited top-k and a ragged token count. The oracle starts from the GPU's own logits, so both sides hold the same
routing decisions.

Tolerance: R14's bf16 form |g - r| <= 2e-2 (|r| + rms(row)): the GPU backward's operands are
bf16 (dy, h, the activation gradients, x) with fp32 accumulation."""

import zlib

import numpy as np
import pytest
import torch

from oracle import moe_backward as B
from gpu_util import RTOL, assert_close, oracle_cfg, to_np
from top_gating_expert_gb300 import moe
from top_gating_expert_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


def _cfg(**kw):
    base = dict(S=2048, G=1, E=8, M=256, H=512, k=2, capacity_factor=0.0, random_routing=0,
                n_shared=0, H_shared=0, act="relu", dtype="bf16", bias=False)
    base.update(kw)
    return base


CASES = {
    "relu_capacity_rr_bias": (_cfg(G=2, capacity_factor=1.0, random_routing=1, bias=True), True),
    "swiglu_dropless_k3": (_cfg(S=1536, E=6, H=256, k=3, act="swiglu"), False),
    "shared_swiglu_capacity": (_cfg(S=1024, E=16, M=192, H=256, act="swiglu", capacity_factor=1.25,
                                    n_shared=2, H_shared=128), True),
    "gates_none_k4": (_cfg(S=1024, E=32, M=128, H=128, k=4, gate_norm="none"), False),
    "ragged_tokens_k1": (_cfg(S=777, E=4, M=64, H=64, k=1, capacity_factor=1.5), True),
    "pnorm2_capacity_k3": (_cfg(S=1536, E=16, M=128, H=256, k=3, capacity_factor=1.0,
                                gate_norm="pnorm", gate_p=2.0), False),
    "pnorm_half_swiglu": (_cfg(S=1024, E=8, M=128, H=128, act="swiglu", gate_norm="pnorm",
                               gate_p=0.5), True),
    "group_limited_k3": (_cfg(S=1024, E=32, M=128, H=256, k=3, capacity_factor=1.25, act="swiglu",
                              n_expert_groups=8, topk_groups=3), False),
    # weight-gradient outputs whose last 256-wide N tile ends part-way (448 = 256 + 192,
    # 320 = 256 + 64): the epilogue's chunks past N store nothing
    "ragged_n_tiles": (_cfg(S=2048, E=8, M=320, H=448, k=2), False),
    # grouped routing with a capacity bounding every expert's rows by groups x capacity
    # <= 256: both routed weight gradients run the resident-B kernel. 8 x 32 = 256 rows (four
    # 64-row k-blocks) at most, ragged per expert, with random routing
    "grouped_short_k_rr": (_cfg(S=2048, G=8, E=16, capacity_factor=1.0, random_routing=1), False),
    # 4 x 48 = 192 (three k-blocks); SwiGLU (dW_in's rows split between dW_in and dW_up),
    # dW_out's last N tile ending part-way (384 = 256 + 128)
    "grouped_short_k_swiglu": (_cfg(S=1024, G=4, E=8, H=384, capacity_factor=0.75,
                                    act="swiglu"), True),
}
AUX, Z = 0.7, 0.3


@pytest.fixture(scope="module", params=sorted(CASES))
def run(request, native_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    name = request.param
    cfg, residual = CASES[name]
    seed = zlib.crc32(name.encode()) % 10000
    inp = make_inputs(cfg, seed=seed)
    layer = moe.MoeLayer(cfg, inp.host)
    layer.enable_backward(inp.host)
    x = inp.host["x"].cuda()
    u = inp.host["u"].cuda() if cfg["random_routing"] else None
    layer.forward(x, u, residual=x if residual else None)
    g = torch.Generator().manual_seed(seed)
    dy = torch.randn((cfg["S"], cfg["M"]), generator=g).to(torch.bfloat16)
    grads = layer.backward(x, dy.cuda(), residual=residual, aux_coef=AUX, z_coef=Z)
    status = moe.device_status(layer.ws_bwd)
    logits = to_np(layer.logits)
    ref = B.layer_backward(inp.np, oracle_cfg(cfg), dy.float().numpy(), AUX, Z, logits=logits,
                           residual=residual)
    got = {f: (None if getattr(grads, f) is None else to_np(getattr(grads, f)))
           for f in ("dx", "dW_g", "dbias", "dW_in", "dW_up", "dW_out", "dWs_in", "dWs_up", "dWs_out")}
    return dict(name=name, cfg=cfg, got=got, ref=ref, status=status)


def test_status_ok(run):
    assert run["status"] == 0


def test_dx(run):
    assert_close(run["got"]["dx"], run["ref"]["dx"], RTOL["bf16"], f"{run['name']} dx")


def test_router_grads(run):
    assert_close(run["got"]["dW_g"], run["ref"]["dW_g"], RTOL["bf16"], f"{run['name']} dW_g")
    if run["got"]["dbias"] is not None:
        r = run["ref"]["dbias"]
        assert_close(run["got"]["dbias"][None], r[None], RTOL["bf16"], f"{run['name']} dbias")


def test_expert_weight_grads(run):
    cfg, got, ref = run["cfg"], run["got"], run["ref"]
    E = cfg["E"]
    for key in ("dW_in", "dW_out") + (("dW_up",) if cfg["act"] == "swiglu" else ()):
        g, r = got[key], ref[key]
        assert g.shape == r.shape, key
        for e in range(E):  # per expert, so that a row's scale is that expert's
            assert_close(g[e], r[e], RTOL["bf16"], f"{run['name']} {key}[{e}]")


def test_shared_weight_grads(run):
    cfg, got, ref = run["cfg"], run["got"], run["ref"]
    if not cfg["n_shared"]:
        pytest.skip("no shared experts")
    ns, Hs, M = cfg["n_shared"], cfg["H_shared"], cfg["M"]
    # the ABI's shared layout: hidden units side by side
    assert_close(got["dWs_in"], ref["dWs_in"].reshape(ns * Hs, M), RTOL["bf16"], "dWs_in")
    if cfg["act"] == "swiglu":
        assert_close(got["dWs_up"], ref["dWs_up"].reshape(ns * Hs, M), RTOL["bf16"], "dWs_up")
    ref_out = np.concatenate([ref["dWs_out"][s] for s in range(ns)], axis=1)  # [M, ns*Hs]
    assert_close(got["dWs_out"], ref_out, RTOL["bf16"], "dWs_out")


def test_unused_experts_get_zero_weight_grads(run):
    """An expert with no kept rows has an empty K segment: its weight gradients are 0."""
    ref = run["ref"]
    counts = ref["route"]["counts"].sum(axis=0)
    for e in np.nonzero(counts == 0)[0]:
        assert not run["got"]["dW_in"][e].any() and not run["got"]["dW_out"][e].any()


@pytest.mark.parametrize("name", ["relu_capacity_rr_bias", "shared_swiglu_capacity", "gates_none_k4"])
def test_stale_workspace_bytes_are_never_read(name, native_lib):
    """The weight-gradient GEMMs read 64-row blocks that run past each expert's rows (into
    the next expert's, or into 64 rows after the last that the forward and the backward
    zero). With every workspace byte past the status header set to 0xFF (NaN in bf16 and
    fp32) and the unwritten rows of token_of / w_perm poisoned too, every gradient must come
    out bit for bit as from zero-filled workspaces, and so must the forward's y."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cfg, residual = CASES[name]
    seed = zlib.crc32(name.encode()) % 10000
    inp = make_inputs(cfg, seed=seed)
    g = torch.Generator().manual_seed(seed)
    dy = torch.randn((cfg["S"], cfg["M"]), generator=g).to(torch.bfloat16).cuda()
    x = inp.host["x"].cuda()
    u = inp.host["u"].cuda() if cfg["random_routing"] else None

    def grads(poison):
        layer = moe.MoeLayer(cfg, inp.host)
        layer.enable_backward(inp.host)
        if poison:
            for ws in (layer.ws, layer.ws_bwd):
                ws[256:].fill_(0xFF)  # past the status word and the scan's ticket
            layer.route_out.token_of.fill_(-1)
            layer.route_out.w_perm.fill_(float("nan"))
        y = to_np(layer.forward(x, u, residual=x if residual else None))
        out = layer.backward(x, dy, residual=residual, aux_coef=AUX, z_coef=Z)
        assert moe.device_status(layer.ws) == 0 and moe.device_status(layer.ws_bwd) == 0
        res = {f: to_np(getattr(out, f)) for f in ("dx", "dW_g", "dbias", "dW_in", "dW_up",
                                                    "dW_out", "dWs_in", "dWs_up", "dWs_out")
               if getattr(out, f) is not None}
        res["y"] = y
        return res

    clean, dirty = grads(False), grads(True)
    for f in clean:
        assert np.isfinite(dirty[f]).all(), f"{name}: {f} not finite"
        assert np.array_equal(clean[f], dirty[f]), f"{name}: {f} differs with a stale workspace"
