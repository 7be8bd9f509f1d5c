"""The fp32 path's backward (plain-FMA kernels) against the oracle's fp64 backward
(oracle/moe_backward.py): every gradient at R14's fp32 tolerance (rtol 1e-5), on small
layers of each kind the fp32 path runs. The kinds are the tiny GShard preset itself; ReLU
with groups, capacity, random routing and a router bias; SwiGLU dropless top-3 with a
residual; SwiGLU with p-norm gates; shared experts (SwiGLU, and ReLU at ragged sizes,
d_model 68 and d_ff 132). The oracle routes from the GPU's logits, so both sides hold the
same routing decisions.

The ReLU mask is a decision that floating point takes. The GPU masks by the sign of its
fp32 h; the oracle by the sign of the fp64 pre-activation a. The two can differ only at
(row, unit) pairs whose |a| lies within the fp32-accumulation bound of zero
(gpu_util.relu_band). Such pairs are counted. Each may move the elements it feeds by the
size of its own term, and the tolerance of exactly those elements is widened by those
terms:
- dW_in's row of the unit, by |dh| |x|;
- dW_out's column, by |do| times its h (at most twice the bound);
- the token's dx, by |dh| |W_in|;
- through the gate gradient (the expert output takes h once more), the token's router
  logits, and so dx's router term, dW_g and dbias. A token's gate gradients off by d in
  all move its logit gradients by at most 2 d in all (gates <= 1).
Every other element is compared at the plain tolerance."""

import zlib

import numpy as np
import pytest
import torch

from oracle import moe_backward as B
from gpu_util import RTOL, check_close, oracle_cfg, relu_band, to_np
from top_gating_expert_gb300 import moe
from top_gating_expert_gb300.inputs import PRESETS, make_inputs

pytestmark = pytest.mark.gpu
AUX, Z = 0.7, 0.3
RT = RTOL["f32"]
FIELDS = ("dx", "dW_g", "dbias", "dW_in", "dW_up", "dW_out", "dWs_in", "dWs_up", "dWs_out")


def _cfg(**kw):
    base = dict(S=512, G=1, E=8, M=64, H=128, k=2, capacity_factor=0.0, random_routing=0,
                n_shared=0, H_shared=0, act="relu", dtype="f32", bias=False)
    base.update(kw)
    return base


CASES = {
    "preset1_gshard_rr": (dict(PRESETS[1]), False),
    "relu_groups_capacity_rr_bias": (_cfg(G=2, capacity_factor=1.0, random_routing=1, bias=True),
                                     False),
    "swiglu_dropless_k3_residual": (_cfg(S=384, E=6, k=3, act="swiglu"), True),
    "shared_swiglu_capacity": (_cfg(S=256, M=96, act="swiglu", capacity_factor=1.25, n_shared=2,
                                    H_shared=128), True),
    "relu_shared_ragged_k1": (_cfg(S=300, E=4, M=68, H=132, k=1, capacity_factor=1.5, n_shared=1,
                                   H_shared=68), False),
    # p-norm gates (the router's backward through gate_norm), top-3 with a capacity
    "swiglu_pnorm2_capacity_k3": (_cfg(S=256, k=3, act="swiglu", capacity_factor=1.0,
                                       gate_norm="pnorm", gate_p=2.0), False),
}


def _f64(a):
    return np.asarray(a, np.float64)


def _widening(a, cfg, ref, dy):
    """The per-element widening of every gradient (module docstring) and the number of
    (row, unit) pairs in the band."""
    S, E, M, H = cfg["S"], cfg["E"], cfg["M"], cfg["H"]
    ns, Hs = cfg.get("n_shared", 0), cfg.get("H_shared", 0)
    dev = dict(dx=np.zeros((S, M)), dW_in=np.zeros((E, H, M)), dW_out=np.zeros((E, M, H)),
               dW_g=np.zeros((E, M)), dbias=np.zeros(E), dWs_in=np.zeros((ns, Hs, M)),
               dWs_out=np.zeros((ns, M, Hs)))
    if cfg["act"] != "relu":
        return dev, 0
    r = ref["route"]
    ids, gate, pos = r["expert_id"], r["gate"], r["pos"]
    x = _f64(a["x"])
    n_band = 0
    d_gate = np.zeros(S)  # per token: how far its gate gradients may be off, in all
    for e in range(E):
        ti, tj = np.nonzero((ids == e) & (pos >= 0))
        if len(ti) == 0:
            continue
        band, bound = relu_band(x[ti], a["W_in"][e])
        if not band.any():
            continue
        n_band += int(band.sum())
        Wi, Wo = _f64(a["W_in"][e]), _f64(a["W_out"][e])
        do = gate[ti, tj][:, None] * dy[ti]
        dh = np.abs(do @ Wo)
        dev["dW_in"][e] += (band * dh).T @ np.abs(x[ti])
        dev["dW_out"][e] += np.abs(do).T @ (band * 2.0 * bound)
        np.add.at(dev["dx"], ti, (band * dh) @ np.abs(Wi))
        np.add.at(d_gate, ti, (((band * 2.0 * bound) @ np.abs(Wo).T) * np.abs(dy[ti])).sum(axis=1))
    for s in range(ns):
        band, bound = relu_band(x, a["Ws_in"][s])
        if not band.any():
            continue
        n_band += int(band.sum())
        dh = np.abs(dy @ _f64(a["Ws_out"][s]))
        dev["dWs_in"][s] += (band * dh).T @ np.abs(x)
        dev["dWs_out"][s] += np.abs(dy).T @ (band * 2.0 * bound)
        dev["dx"] += (band * dh) @ np.abs(_f64(a["Ws_in"][s]))
    dl = 2.0 * d_gate  # bound on each token's logit-gradient change, in all
    dev["dx"] += dl[:, None] * np.abs(_f64(a["W_g"])).max(axis=0)[None, :]
    dev["dW_g"] += (dl[:, None] * np.abs(x)).sum(axis=0)[None, :]
    dev["dbias"] += dl.sum()
    return dev, n_band


def _backward(cfg, residual, seed):
    inp = make_inputs(cfg, seed=seed)
    layer = moe.MoeLayer(cfg, inp.host)
    layer.enable_backward(inp.host)
    x = inp.host["x"].cuda()
    u = inp.host["u"].cuda() if cfg["random_routing"] else None
    layer.forward(x, u, residual=x if residual else None)
    dy = torch.randn((cfg["S"], cfg["M"]), generator=torch.Generator().manual_seed(seed))
    grads = layer.backward(x, dy.cuda(), residual=residual, aux_coef=AUX, z_coef=Z)
    status = moe.device_status(layer.ws_bwd)
    got = {f: (None if getattr(grads, f) is None else to_np(getattr(grads, f))) for f in FIELDS}
    return inp, layer, dy, got, status


@pytest.fixture(scope="module", params=sorted(CASES))
def run(request, native_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    name = request.param
    cfg, residual = CASES[name]
    seed = zlib.crc32(name.encode()) % 10000
    inp, layer, dy, got, status = _backward(cfg, residual, seed)
    dy64 = dy.numpy().astype(np.float64)
    ref = B.layer_backward(inp.np, oracle_cfg(cfg), dy64, AUX, Z, logits=to_np(layer.logits),
                           residual=residual)
    dev, n_band = _widening(inp.np, cfg, ref, dy64)
    print(f"{name}: {n_band} (row, unit) pairs within the fp32-accumulation bound of zero")
    return dict(name=name, cfg=cfg, residual=residual, seed=seed, got=got, ref=ref, dev=dev,
                status=status)


def test_status_ok(run):
    assert run["status"] == 0


def test_dx(run):
    check_close(run["got"]["dx"], run["ref"]["dx"], RT, run["dev"]["dx"], f"{run['name']} dx")


def test_router_grads(run):
    got, ref, dev = run["got"], run["ref"], run["dev"]
    check_close(got["dW_g"], ref["dW_g"], RT, dev["dW_g"], f"{run['name']} dW_g")
    if got["dbias"] is not None:
        check_close(got["dbias"][None], ref["dbias"][None], RT, dev["dbias"][None],
                    f"{run['name']} dbias")


def test_expert_weight_grads(run):
    cfg, got, ref, dev = run["cfg"], run["got"], run["ref"], run["dev"]
    for e in range(cfg["E"]):  # per expert, so that a row's scale is that expert's
        check_close(got["dW_in"][e], ref["dW_in"][e], RT, dev["dW_in"][e], f"{run['name']} dW_in[{e}]")
        check_close(got["dW_out"][e], ref["dW_out"][e], RT, dev["dW_out"][e],
                    f"{run['name']} dW_out[{e}]")
        if cfg["act"] == "swiglu":
            check_close(got["dW_up"][e], ref["dW_up"][e], RT, 0.0, f"{run['name']} dW_up[{e}]")


def test_shared_weight_grads(run):
    cfg, got, ref, dev = run["cfg"], run["got"], run["ref"], run["dev"]
    if not cfg["n_shared"]:
        pytest.skip("no shared experts")
    ns, Hs, M = cfg["n_shared"], cfg["H_shared"], cfg["M"]
    # the ABI's shared layout: hidden units side by side
    check_close(got["dWs_in"], ref["dWs_in"].reshape(ns * Hs, M), RT,
                dev["dWs_in"].reshape(ns * Hs, M), f"{run['name']} dWs_in")
    if cfg["act"] == "swiglu":
        check_close(got["dWs_up"], ref["dWs_up"].reshape(ns * Hs, M), RT, 0.0,
                    f"{run['name']} dWs_up")
    cat = lambda t: np.concatenate([t[s] for s in range(ns)], axis=1)  # [M, ns * Hs]
    check_close(got["dWs_out"], cat(ref["dWs_out"]), RT, cat(dev["dWs_out"]),
                f"{run['name']} dWs_out")


def test_unused_experts_get_zero_weight_grads(run):
    """An expert with no kept rows sums over no rows: its weight gradients are exactly 0."""
    counts = run["ref"]["route"]["counts"].sum(axis=0)
    for e in np.nonzero(counts == 0)[0]:
        assert not run["got"]["dW_in"][e].any() and not run["got"]["dW_out"][e].any()


def test_repeatable(run):
    """Every sum has a fixed order: a second backward on the same inputs gives the same bits."""
    _, _, _, got2, status = _backward(run["cfg"], run["residual"], run["seed"])
    assert status == 0
    for f in FIELDS:
        if run["got"][f] is not None:
            assert np.array_equal(run["got"][f], got2[f]), f"{run['name']}: {f}"
