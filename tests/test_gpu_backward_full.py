"""The backward pass at full preset size (the training step the benchmark times), checked on
outputs the oracle can form one by one: the weight gradients of sampled experts (from those
experts' rows alone) and dx of sampled tokens (their kept choices, the shared experts, the
residual and the router's term through the token's own logits row). The oracle routes from
the GPU's logits, so both sides hold the same routing decisions; dW_g and dbias need every
token's gate gradient and are checked by the small layers of test_gpu_backward. Every
expected value comes from the oracle (oracle/moe_backward.py's expert backward, its own
fp64 ReLU mask); nothing the GPU computed enters the reference.

Tolerance: R14's bf16 form, as in test_gpu_backward, widened only where the ReLU's mask is
ambiguous. The mask is a decision that floating point takes: the GPU masks by the sign of
its stored h, whose pre-activation it accumulated in fp32 over K = M products of exact bf16
values, and the oracle by the sign of the fp64 pre-activation a. Recursive fp32 summation of
K terms is off by at most (K - 1) u sum|terms| with u = 2^-24 (round to nearest), 2^-23 if
the accumulator truncates; the bound used is

    |a32 - a| <= 2 K 2^-24 sum_m |x_m| |w_m|,

so the two masks can differ only at (row, unit) pairs whose |a| lies within it. Those pairs
are counted and printed. Each one may move, by the size of its own term, the elements that
it feeds: dW_in[j, :] by |dh[r, j]| |x[r, :]|, dx of its token by |dh[r, j]| |W_in[j, :]|,
dW_out[:, j] by |do[r, :]| times its h (at most twice the bound), and dx's router term
through the gate gradient, which takes h once more. The tolerance of exactly those elements
is widened by the sum of those terms; every other element is compared at R14's tolerance."""

import numpy as np
import pytest
import torch

from oracle import moe_backward as B
from oracle import moe_oracle as O
from gpu_util import RTOL, check_close, oracle_cfg, relu_band, to_np
from top_gating_expert_gb300 import moe
from top_gating_expert_gb300.inputs import PRESETS, make_inputs

pytestmark = pytest.mark.gpu
AUX, Z = 0.7, 0.3


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

    a = inp.np
    ocfg = oracle_cfg(cfg)
    logits = to_np(layer.logits)
    r = O.route(logits, ocfg, a.get("u"))
    dy = dy_h.float().numpy().astype(np.float64)
    act, k = cfg["act"], cfg["k"]
    ids, gate, pos = r["expert_id"], r["gate"], r["pos"]
    relu = act == "relu"
    rt = RTOL["bf16"]

    def expert(e, t_idx, do):
        W_up = a["W_up"][e] if not relu else None
        return B._ffn_backward(a["x"][t_idx], a["W_in"][e], a["W_out"][e], act, W_up, do)

    # (i) weight gradients of two experts: the busiest and one near the median
    counts = np.bincount(ids[pos >= 0].ravel(), minlength=cfg["E"])
    order = np.argsort(counts)
    n_band = n_pairs = 0
    for e in (int(order[-1]), int(order[len(order) // 2])):
        ti, tj = np.nonzero((ids == e) & (pos >= 0))
        do = gate[ti, tj][:, None] * dy[ti]
        _, dWi, dWu, dWo, _ = expert(e, ti, do)
        dev_in = dev_out = 0.0
        if relu:
            band, bound = relu_band(a["x"][ti], a["W_in"][e])
            n_band += int(band.sum())
            n_pairs += band.size
            dh = np.abs(do @ np.asarray(a["W_out"][e], np.float64))
            dev_in = (band * dh).T @ np.abs(np.asarray(a["x"][ti], np.float64))
            dev_out = np.abs(do).T @ (band * 2.0 * bound)
        check_close(to_np(grads.dW_out[e]), dWo, rt, dev_out, f"preset {n} dW_out[{e}]")
        check_close(to_np(grads.dW_in[e]), dWi, rt, dev_in, f"preset {n} dW_in[{e}]")
        if not relu:
            check_close(to_np(grads.dW_up[e]), dWu, rt, 0.0, f"preset {n} dW_up[{e}]")

    # (ii) dx of sampled tokens: kept choices, shared experts, residual, router term
    rng = np.random.default_rng(n)
    tokens = rng.choice(cfg["S"], size=6, replace=False)
    dropped = np.nonzero((pos < 0).all(axis=1))[0]
    if len(dropped):
        tokens = np.append(tokens, dropped[0])
    dgate = np.zeros((cfg["S"], k))
    ref = np.zeros((len(tokens), cfg["M"]))
    dev_dx = np.zeros((len(tokens), cfg["M"]))
    dev_dgate = np.zeros((len(tokens), k))
    for q, t in enumerate(tokens):
        for j in range(k):
            if pos[t, j] < 0:
                continue
            e = ids[t, j]
            do = gate[t, j] * dy[t:t + 1]
            dxe, _, _, _, o = expert(e, [t], do)
            ref[q] += dxe[0]
            dgate[t, j] = float(np.dot(dy[t], o[0]))
            if relu:
                band, bound = relu_band(a["x"][t:t + 1], a["W_in"][e])
                n_band += int(band.sum())
                n_pairs += band.size
                W_out = np.asarray(a["W_out"][e], np.float64)
                dh = np.abs(do @ W_out)
                dev_dx[q] += ((band * dh) @ np.abs(np.asarray(a["W_in"][e], np.float64)))[0]
                # the expert output o, hence the gate gradient dy . o, through h
                dev_dgate[q, j] = float(((band * 2.0 * bound) @ np.abs(W_out).T)[0] @ np.abs(dy[t]))
        for s in range(cfg.get("n_shared", 0)):
            dxs, _, _, _, _ = B._ffn_backward(a["x"][t:t + 1], a["Ws_in"][s], a["Ws_out"][s], act,
                                              a["Ws_up"][s] if not relu else None, dy[t:t + 1])
            ref[q] += dxs[0]
        if residual:
            ref[q] += dy[t]
    dl = B.router_logit_grad(np.asarray(logits, np.float64), r, dgate, ocfg, AUX, Z)
    W_g = np.asarray(a["W_g"], np.float64)
    ref += dl[tokens] @ W_g
    # a gate gradient off by d moves the token's logit gradients by at most 2 d in all
    # (gates <= 1), hence dx by 2 d max_e |W_g[e, m]|
    dev_dx += 2.0 * dev_dgate.sum(axis=1, keepdims=True) * np.abs(W_g).max(axis=0)[None, :]
    check_close(to_np(grads.dx)[tokens], ref, rt, dev_dx, f"preset {n} dx (sampled tokens)")
    if relu:
        print(f"preset {n}: {n_band} of {n_pairs} (row, unit) pairs of the checked rows lie "
              f"within the fp32-accumulation bound of zero (their ReLU mask may differ)")
