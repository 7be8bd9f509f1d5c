"""CPU oracle for the backward pass of one GPU's Mixture-of-Experts layer.

TEST INFRASTRUCTURE ONLY, like moe_oracle (which it imports, and nothing else of this
repository): only the test-suite, the smoke check and the benchmark's CPU legs may use it.

The loss whose gradients are returned is

    L = sum(dy * y) + aux_coef * aux + z_coef * z

with y the layer output of moe_oracle.layer_forward and aux, z its two losses, i.e. dy is
the upstream gradient of the layer output and the two coefficients weight the losses
(MegaBlocks router chapter §3: the load-balancing loss is a differentiable proxy whose
gradient reaches the router only through the expert scores; §2: z-loss). Everything is
fp64 numpy, the chain rule written out step by step.

Readings (repeated in the design notes):
  R19 routing decisions (which experts, which assignments are kept) are piecewise
      constant in the logits and are held fixed: gradients flow through the gate values,
      the softmax probabilities of the aux loss and the logsumexp of the z-loss, as the
      pages' loss description says ("the gradient reaches the router only through
      expert_scores"). A dropped assignment contributes nothing to y, so its gate gets no
      gradient. The counts f_e of the aux loss are constants.
  R20 the backward covers the default gates (softmax over the k selected logits), the
      un-normalised full-softmax gates ("none") and the p-norm gates; uniform assignment
      (a benchmark switch whose ids do not come from the logits) is forward-only.

Pins: tests/test_oracle_backward.py checks every gradient against central finite
differences of the (separately pinned) forward on tiny layers, away from routing ties.
"""

from __future__ import annotations

import numpy as np

from oracle import moe_oracle as O

_f64 = O._f64


def _ffn_backward(x_rows, W_in, W_out, act, W_up, do):
    """One expert on rows x [n, M] with output gradient do [n, M] (already gate-scaled).
    Returns (dx [n, M], dW_in [H, M], dW_up [H, M] or None, dW_out [M, H], o [n, M] the
    unscaled expert output)."""
    xr, W_in, W_out = _f64(x_rows), _f64(W_in), _f64(W_out)
    a = xr @ W_in.T
    if act == "relu":
        h = np.maximum(a, 0.0)
    else:
        b = xr @ _f64(W_up).T
        s = 1.0 / (1.0 + np.exp(-a))
        h = a * s * b
    o = h @ W_out.T
    dW_out = do.T @ h
    dh = do @ W_out
    if act == "relu":
        da = dh * (a > 0.0)
        return da @ W_in, da.T @ xr, None, dW_out, o
    # d silu(a) / da = s * (1 + a * (1 - s))
    da = dh * b * s * (1.0 + a * (1.0 - s))
    db = dh * a * s
    return da @ W_in + db @ _f64(W_up), da.T @ xr, db.T @ xr, dW_out, o


def router_logit_grad(logits, r: dict, dgate, cfg: dict, aux_coef: float, z_coef: float):
    """dL/dlogits [S, E]: the gate term (through the k gates), then the aux term (through
    the full-softmax probabilities P_e, counts fixed) and the z term (through logsumexp)."""
    S, E, k, G = cfg["S"], cfg["E"], cfg["k"], cfg["G"]
    Sg = S // G
    ids = r["expert_id"]
    p, lse = O.log_softmax_parts(logits)
    dl = np.zeros((S, E))
    rows = np.repeat(np.arange(S), k)
    if cfg.get("gate_norm", "softmax_topk") == "softmax_topk":
        # g_i = softmax over the k selected logits: dl_{id_i} = g_i (dg_i - sum_j g_j dg_j)
        sel = r["gate_raw"]
        inner = np.sum(sel * dgate, axis=1, keepdims=True)
        np.add.at(dl, (rows, ids.ravel()), (sel * (dgate - inner)).ravel())
    elif cfg.get("gate_norm") == "pnorm":
        # g_i = w_i / ||w||_p with w_i = exp(l_i): dg_i/dl_j = g_i (delta_ij - g_j^p), so
        # dl_{id_j} = g_j dg_j - g_j^p sum_i g_i dg_i (p = 1: the softmax case above)
        pw = float(cfg["gate_p"])
        sel = O.normalised_gates(logits, ids, "pnorm", pw)
        inner = np.sum(sel * dgate, axis=1, keepdims=True)
        np.add.at(dl, (rows, ids.ravel()), (sel * dgate - sel ** pw * inner).ravel())
    else:
        # g_j = p_{id_j}: dl_i = sum_j dg_j p_{id_j} (delta(i, id_j) - p_i)
        sel = np.take_along_axis(p, ids, axis=1)
        np.add.at(dl, (rows, ids.ravel()), (sel * dgate).ravel())
        dl -= p * np.sum(sel * dgate, axis=1, keepdims=True)
    if aux_coef:
        f = r["counts_routed"] / float(Sg * k)                    # [G, E], constant
        fg = np.repeat(f, Sg, axis=0)                              # per token
        dl += aux_coef * (E / (G * Sg)) * p * (fg - np.sum(fg * p, axis=1, keepdims=True))
    if z_coef:
        dl += z_coef * (2.0 / S) * lse[:, None] * p
    return dl


def layer_backward(arrays: dict, cfg: dict, dy, aux_coef: float = 0.0, z_coef: float = 0.0,
                   logits=None, residual: bool = False) -> dict:
    """Gradients of L (module docstring) w.r.t. x, W_g, bias, W_in, W_up, W_out and the
    shared experts' weights, plus dlogits [S, E] and dgate [S, k] (0 where not kept)."""
    x = _f64(arrays["x"])
    S, E, k = cfg["S"], cfg["E"], cfg["k"]
    norm = cfg.get("gate_norm", "softmax_topk")
    if norm not in ("softmax_topk", "none", "pnorm") or cfg.get("uniform_assignment", 0):
        raise ValueError("the backward covers the softmax_topk, none and pnorm gates, no uniform "
                         "assignment (reading R20)")
    if logits is None:
        logits = O.router_logits(x, arrays["W_g"], arrays.get("bias"))
    logits = _f64(logits)
    r = O.route(logits, cfg, arrays.get("u"))
    dy = _f64(dy)
    swiglu = cfg["act"] == "swiglu"

    dx = np.zeros_like(x)
    dW_in = np.zeros((E,) + np.shape(arrays["W_in"])[1:])
    dW_up = np.zeros_like(dW_in) if swiglu else None
    dW_out = np.zeros((E,) + np.shape(arrays["W_out"])[1:])
    dgate = np.zeros((S, k))
    ids, gate, pos = r["expert_id"], r["gate"], r["pos"]
    for e in range(E):
        ti, tj = np.nonzero((ids == e) & (pos >= 0))
        if len(ti) == 0:
            continue
        g = gate[ti, tj][:, None]
        W_up = arrays["W_up"][e] if swiglu else None
        dxe, dWi, dWu, dWo, o = _ffn_backward(x[ti], arrays["W_in"][e], arrays["W_out"][e],
                                              cfg["act"], W_up, g * dy[ti])
        np.add.at(dx, ti, dxe)
        dW_in[e] += dWi
        if swiglu:
            dW_up[e] += dWu
        dW_out[e] += dWo
        dgate[ti, tj] = np.sum(dy[ti] * o, axis=1)

    out = dict(dgate=dgate)
    if cfg.get("n_shared", 0) > 0:
        ns = cfg["n_shared"]
        dWs_in = np.zeros(np.shape(arrays["Ws_in"]))
        dWs_up = np.zeros_like(dWs_in) if swiglu else None
        dWs_out = np.zeros(np.shape(arrays["Ws_out"]))
        for s in range(ns):
            W_up = arrays["Ws_up"][s] if swiglu else None
            dxs, dWi, dWu, dWo, _ = _ffn_backward(x, arrays["Ws_in"][s], arrays["Ws_out"][s],
                                                  cfg["act"], W_up, dy)
            dx += dxs
            dWs_in[s] = dWi
            if swiglu:
                dWs_up[s] = dWu
            dWs_out[s] = dWo
        out.update(dWs_in=dWs_in, dWs_up=dWs_up, dWs_out=dWs_out)
    if residual:
        dx += dy

    dl = router_logit_grad(logits, r, dgate, cfg, aux_coef, z_coef)
    W_g = _f64(arrays["W_g"])
    dx += dl @ W_g
    out.update(dx=dx, dW_g=dl.T @ x, dbias=dl.sum(axis=0), dW_in=dW_in, dW_up=dW_up,
               dW_out=dW_out, dlogits=dl, route=r)
    return out


def layer_loss(arrays: dict, cfg: dict, dy, aux_coef: float = 0.0, z_coef: float = 0.0,
               residual: bool = False):
    """L of the module docstring through the forward oracle (for finite differences);
    also returns the routing so that a caller can check no decision changed."""
    x = arrays["x"]
    y, r, _ = O.layer_forward(arrays, cfg, residual=x if residual else None)
    return float(np.sum(_f64(dy) * y) + aux_coef * r["aux_loss"] + z_coef * r["z_loss"]), r
