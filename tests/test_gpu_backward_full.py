"""The backward pass at full preset size (the training step the benchmark times), checked on
outputs the oracle can form one by one: the weight gradients of sampled experts (from those
experts' rows alone) and dx of sampled tokens (their kept choices, the shared experts, the
residual and the router's term through the token's own logits row). The oracle routes from
the GPU's logits, so both sides hold the same routing decisions; dW_g and dbias need every
token's gate gradient and are checked by the small layers of test_gpu_backward.

Tolerance: R14's bf16 form, as in test_gpu_backward. The ReLU's mask is a decision that
floating point takes: where a pre-activation lies within rounding of zero the GPU (fp32
accumulation, the sign of its stored h) and an fp64 recomputation can disagree, and with
millions of (row, hidden unit) pairs an expert at full size has a few such flips, each
moving one of its K terms. So for ReLU the reference takes the mask from the GPU's own h
(GEMM 1 of the step-wise calls, the layer's h bit for bit) and everything else in fp64."""

import numpy as np
import pytest
import torch

from oracle import moe_backward as B
from oracle import moe_oracle as O
from gpu_util import RTOL, assert_close, oracle_cfg, to_np
from top_gating_expert_gb300 import moe
from top_gating_expert_gb300.inputs import PRESETS, make_inputs

pytestmark = pytest.mark.gpu
AUX, Z = 0.7, 0.3


def _expert_backward(x_rows, a, e, act, do, mask):
    """The oracle's expert backward with the ReLU mask given (None: its own, for SwiGLU)."""
    if mask is None:
        return B._ffn_backward(x_rows, a["W_in"][e], a["W_out"][e], act,
                               a["W_up"][e] if act == "swiglu" else None, do)
    xr = np.asarray(x_rows, np.float64)
    W_in, W_out = np.asarray(a["W_in"][e], np.float64), np.asarray(a["W_out"][e], np.float64)
    h = np.maximum(xr @ W_in.T, 0.0) * mask
    da = (do @ W_out) * mask
    return da @ W_in, da.T @ xr, None, do.T @ h, h @ W_out.T


@pytest.mark.parametrize("n", [2, 4, 5])
def test_backward_full_size_sampled(n, native_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cfg = PRESETS[n]
    inp = make_inputs(cfg, preset_number=n)
    layer = moe.MoeLayer(cfg, inp.host)
    layer.enable_backward(inp.host)
    dev = layer.device
    x = inp.host["x"].to(dev)
    u = inp.host["u"].to(dev) if cfg["random_routing"] else None
    residual = n == 5
    layer.forward(x, u, residual=x if residual else None)
    g = torch.Generator().manual_seed(1000 + n)
    dy_h = torch.randn((cfg["S"], cfg["M"]), generator=g).to(torch.bfloat16)
    grads = layer.backward(x, dy_h.to(dev), residual=residual, aux_coef=AUX, z_coef=Z)
    assert moe.device_status(layer.ws_bwd) == 0

    h_gpu = None
    if cfg["act"] == "relu":  # GEMM 1's h through the step-wise calls: the mask's decisions
        out = layer.route_out
        R = moe.rows_max(cfg)
        x_perm = torch.empty((R, cfg["M"]), dtype=torch.bfloat16, device=dev)
        h_perm = torch.empty((R, cfg["H"]), dtype=torch.bfloat16, device=dev)
        moe.dispatch(cfg, x, out, x_perm)
        moe.expert_up(cfg, x_perm, out.expert_offsets, layer.W_in_packed, h_perm, layer.ws)
        assert moe.device_status(layer.ws) == 0
        h_gpu = to_np(h_perm) > 0
        del x_perm, h_perm
    rows_gpu = to_np(layer.route_out.row)

    a = inp.np
    ocfg = oracle_cfg(cfg)
    logits = to_np(layer.logits)
    r = O.route(logits, ocfg, a.get("u"))
    dy = dy_h.float().numpy().astype(np.float64)
    act, k = cfg["act"], cfg["k"]
    ids, gate, pos = r["expert_id"], r["gate"], r["pos"]
    swiglu = act == "swiglu"

    # (i) weight gradients of two experts: the busiest and one near the median
    counts = np.bincount(ids[pos >= 0].ravel(), minlength=cfg["E"])
    order = np.argsort(counts)
    for e in (int(order[-1]), int(order[len(order) // 2])):
        ti, tj = np.nonzero((ids == e) & (pos >= 0))
        mask = None if h_gpu is None else h_gpu[rows_gpu[ti, tj]]
        _, dWi, dWu, dWo, _ = _expert_backward(a["x"][ti], a, e, act,
                                               gate[ti, tj][:, None] * dy[ti], mask)
        assert_close(to_np(grads.dW_out[e]), dWo, RTOL["bf16"], f"preset {n} dW_out[{e}]")
        assert_close(to_np(grads.dW_in[e]), dWi, RTOL["bf16"], f"preset {n} dW_in[{e}]")
        if swiglu:
            assert_close(to_np(grads.dW_up[e]), dWu, RTOL["bf16"], f"preset {n} dW_up[{e}]")

    # (ii) dx of sampled tokens: kept choices, shared experts, residual, router term
    rng = np.random.default_rng(n)
    tokens = rng.choice(cfg["S"], size=6, replace=False)
    dropped = np.nonzero((pos < 0).all(axis=1))[0]
    if len(dropped):
        tokens = np.append(tokens, dropped[0])
    dgate = np.zeros((cfg["S"], k))
    ref = np.zeros((len(tokens), cfg["M"]))
    for q, t in enumerate(tokens):
        for j in range(k):
            if pos[t, j] < 0:
                continue
            e = ids[t, j]
            mask = None if h_gpu is None else h_gpu[rows_gpu[t, j]][None]
            dxe, _, _, _, o = _expert_backward(a["x"][t:t + 1], a, e, act,
                                               gate[t, j] * dy[t:t + 1], mask)
            ref[q] += dxe[0]
            dgate[t, j] = float(np.dot(dy[t], o[0]))
        for s in range(cfg.get("n_shared", 0)):
            dxs, _, _, _, _ = B._ffn_backward(a["x"][t:t + 1], a["Ws_in"][s], a["Ws_out"][s], act,
                                              a["Ws_up"][s] if swiglu else None, dy[t:t + 1])
            ref[q] += dxs[0]
        if residual:
            ref[q] += dy[t]
    dl = B.router_logit_grad(np.asarray(logits, np.float64), r, dgate, ocfg, AUX, Z)
    ref += dl[tokens] @ np.asarray(a["W_g"], np.float64)
    assert_close(to_np(grads.dx)[tokens], ref, RTOL["bf16"], f"preset {n} dx (sampled tokens)")
