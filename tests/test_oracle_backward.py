"""Pins of the backward oracle: every gradient against central finite differences of the
forward oracle (itself pinned by brute force, closed forms and worked examples), on tiny
layers whose routing does not change within the step; and planted mistakes that the
finite differences must catch."""

import numpy as np
import pytest

from oracle import moe_backward as B
from oracle import moe_oracle as O

EPS = 1e-6


def _layer(seed, act, S=12, G=2, E=4, M=6, H=4, k=2, cf=1.0, rr=0, n_shared=0, bias=True,
           norm="softmax_topk", p=1.0, ng=0, tg=0):
    rng = np.random.default_rng(seed)
    cfg = dict(S=S, G=G, E=E, M=M, H=H, k=k, capacity_factor=cf, random_routing=rr,
               n_shared=n_shared, H_shared=3 if n_shared else 0, act=act, gate_norm=norm,
               gate_p=p)
    if ng:
        cfg.update(n_expert_groups=ng, topk_groups=tg)
    a = dict(x=rng.standard_normal((S, M)), W_g=rng.standard_normal((E, M)),
             W_in=rng.standard_normal((E, H, M)) * 0.5, W_up=rng.standard_normal((E, H, M)) * 0.5,
             W_out=rng.standard_normal((E, M, H)) * 0.5, u=rng.random(S, dtype=np.float32))
    if bias:
        a["bias"] = rng.standard_normal(E) * 0.3
    if n_shared:
        a.update(Ws_in=rng.standard_normal((n_shared, 3, M)) * 0.5,
                 Ws_up=rng.standard_normal((n_shared, 3, M)) * 0.5,
                 Ws_out=rng.standard_normal((n_shared, M, 3)) * 0.5)
    dy = rng.standard_normal((S, M))
    return cfg, a, dy


def _fd(cfg, a, dy, name, direction, aux, z, residual):
    """Central difference of L along `direction` on parameter `name`; None if the routing
    differs between the two points (the derivative is then not the gradient's)."""
    lo, hi = dict(a), dict(a)
    lo[name] = a[name] - EPS * direction
    hi[name] = a[name] + EPS * direction
    Llo, rlo = B.layer_loss(lo, cfg, dy, aux, z, residual)
    Lhi, rhi = B.layer_loss(hi, cfg, dy, aux, z, residual)
    if not (np.array_equal(rlo["expert_id"], rhi["expert_id"]) and np.array_equal(rlo["pos"], rhi["pos"])):
        return None
    return (Lhi - Llo) / (2 * EPS)


GRAD_OF = {"x": "dx", "W_g": "dW_g", "bias": "dbias", "W_in": "dW_in", "W_up": "dW_up",
           "W_out": "dW_out", "Ws_in": "dWs_in", "Ws_up": "dWs_up", "Ws_out": "dWs_out"}

CASES = [
    dict(seed=1, act="relu"),
    dict(seed=2, act="swiglu"),
    dict(seed=3, act="relu", G=1, cf=0.0, k=3, E=5),                    # dropless, k = 3
    dict(seed=4, act="swiglu", n_shared=2, cf=0.5),                     # drops + shared
    dict(seed=5, act="relu", rr=1, cf=1.0),                             # random routing
    dict(seed=6, act="swiglu", norm="none", G=3, S=15, E=6),            # TopK(Softmax) gates
    dict(seed=7, act="relu", norm="pnorm", p=2.0, k=3, E=6),            # p-norm gates
    dict(seed=8, act="swiglu", norm="pnorm", p=0.5, cf=0.75),           # p < 1, drops
    dict(seed=9, act="relu", E=8, k=3, ng=4, tg=2),                     # group-limited top-k
    dict(seed=10, act="swiglu", E=8, ng=4, tg=1, norm="none", cf=0.0),  # one group, dropless
]


def check_all(case, aux=0.7, z=0.3, residual=True, tol=2e-6):
    cfg, a, dy = _layer(**case)
    g = B.layer_backward(a, cfg, dy, aux, z, residual=residual)
    rng = np.random.default_rng(case["seed"] + 100)
    names = [n for n in GRAD_OF if n in a and not (n == "W_up" and cfg["act"] != "swiglu")
             and not (n == "Ws_up" and cfg["act"] != "swiglu")]
    checked = 0
    for name in names:
        for _ in range(3):
            v = rng.standard_normal(np.shape(a[name]))
            fd = _fd(cfg, a, dy, name, v, aux, z, residual)
            if fd is None:
                continue
            an = float(np.sum(g[GRAD_OF[name]] * v))
            assert abs(fd - an) <= tol * (1 + abs(fd)), (name, fd, an)
            checked += 1
    assert checked >= 2 * len(names)
    return g


@pytest.mark.parametrize("i", range(len(CASES)))
def test_gradients_match_finite_differences(i):
    check_all(CASES[i])


def test_loss_terms_separately():
    # only the aux term; only the z term; only the output term
    for aux, z, dyscale in ((1.0, 0.0, 0.0), (0.0, 1.0, 0.0), (0.0, 0.0, 1.0)):
        cfg, a, dy = _layer(seed=11, act="relu")
        dy = dy * dyscale
        g = B.layer_backward(a, cfg, dy, aux, z)
        v = np.random.default_rng(3).standard_normal(a["W_g"].shape)
        fd = _fd(cfg, a, dy, "W_g", v, aux, z, False)
        assert fd is not None
        assert abs(fd - float(np.sum(g["dW_g"] * v))) <= 2e-6 * (1 + abs(fd))


def test_dgate_is_output_derivative_and_zero_when_dropped():
    cfg, a, dy = _layer(seed=4, act="swiglu", n_shared=0, cf=0.5)
    g = B.layer_backward(a, cfg, dy)
    r = g["route"]
    assert np.all(g["dgate"][r["pos"] < 0] == 0.0)
    assert np.any(r["pos"] < 0)  # the case does drop assignments


def test_rejects_forward_only_variants():
    cfg, a, dy = _layer(seed=1, act="relu", norm="softmax_topk")
    with pytest.raises(ValueError):
        B.layer_backward(a, dict(cfg, uniform_assignment=1), dy)


# ------------------------------------------------------------------ planted mistakes
def _pins_ok():
    try:
        for c in CASES[:2] + CASES[3:5]:
            check_all(c)
    except AssertionError:
        return False
    return True


_orig_ffn_bwd = B._ffn_backward


def _silu_derivative_wrong(x_rows, W_in, W_out, act, W_up, do):
    if act != "swiglu":
        return _orig_ffn_bwd(x_rows, W_in, W_out, act, W_up, do)
    xr = np.asarray(x_rows, float)
    a, b = xr @ np.asarray(W_in).T, xr @ np.asarray(W_up).T
    s = 1.0 / (1.0 + np.exp(-a))
    h = a * s * b
    dh = do @ np.asarray(W_out)
    da = dh * b * s            # missing the (1 + a (1 - s)) factor
    db = dh * a * s
    return (da @ W_in + db @ W_up, da.T @ xr, db.T @ xr, do.T @ h, h @ np.asarray(W_out).T)


def _wout_grad_transposed(x_rows, W_in, W_out, act, W_up, do):
    dx, dWi, dWu, dWo, o = _orig_ffn_bwd(x_rows, W_in, W_out, act, W_up, do)
    return dx, dWi, dWu, dWo[::-1].copy(), o


@pytest.mark.parametrize("name,fn", [("silu derivative missing a factor", _silu_derivative_wrong),
                                     ("dW_out rows reversed", _wout_grad_transposed)])
def test_planted_mistake_is_caught(name, fn, monkeypatch):
    monkeypatch.setattr(B, "_ffn_backward", fn)
    assert not _pins_ok(), name


_orig_router = B.router_logit_grad


def _gate_term_without_inner(logits, r, dgate, cfg, aux_coef, z_coef):
    dl = _orig_router(logits, r, dgate, cfg, aux_coef, z_coef)
    sel = r["gate_raw"]
    inner = np.sum(sel * dgate, axis=1, keepdims=True)
    np.add.at(dl, (np.repeat(np.arange(cfg["S"]), cfg["k"]), r["expert_id"].ravel()),
              (sel * inner).ravel())  # undoes the -g_i sum_j g_j dg_j part
    return dl


def _aux_without_E(logits, r, dgate, cfg, aux_coef, z_coef):
    return _orig_router(logits, r, dgate, cfg, aux_coef / cfg["E"], z_coef)


def _z_sign_flipped(logits, r, dgate, cfg, aux_coef, z_coef):
    return _orig_router(logits, r, dgate, cfg, aux_coef, -z_coef)


@pytest.mark.parametrize("name,fn", [("gate softmax Jacobian missing its second term", _gate_term_without_inner),
                                     ("aux gradient missing the factor E", _aux_without_E),
                                     ("z gradient sign flipped", _z_sign_flipped)])
def test_planted_router_mistake_is_caught(name, fn, monkeypatch):
    monkeypatch.setattr(B, "router_logit_grad", fn)
    assert not _pins_ok(), name


def _pnorm_power_dropped(logits, r, dgate, cfg, aux_coef, z_coef):
    """p-norm gates with g_j in place of g_j^p in the Jacobian's second term."""
    if cfg.get("gate_norm") != "pnorm":
        return _orig_router(logits, r, dgate, cfg, aux_coef, z_coef)
    dl = _orig_router(logits, r, np.zeros_like(dgate), cfg, aux_coef, z_coef)  # aux and z only
    ids = r["expert_id"]
    g = O.normalised_gates(logits, ids, "pnorm", float(cfg["gate_p"]))
    inner = np.sum(g * dgate, axis=1, keepdims=True)
    np.add.at(dl, (np.repeat(np.arange(cfg["S"]), cfg["k"]), ids.ravel()),
              (g * dgate - g * inner).ravel())
    return dl


def test_planted_pnorm_mistake_is_caught(monkeypatch):
    case = next(c for c in CASES if c.get("norm") == "pnorm" and c.get("p") == 2.0)
    check_all(case)  # the pin holds for the oracle as written
    monkeypatch.setattr(B, "router_logit_grad", _pnorm_power_dropped)
    with pytest.raises(AssertionError):
        check_all(case)
