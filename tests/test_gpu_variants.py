"""GPU parity of the routing variants (group-limited top-k, gate normalisations, uniform
assignment) against the oracle: routing bit-exact from the GPU's own logits through both
entry points (moe_router + moe_route, and the fused moe_router_route), the whole layer
within tolerance, and tie-heavy logits through moe_route directly.

Lec16 Systems for MoE Models, "DeepSeek V3 MoE": 256 routed experts in 8 groups, 4 kept,
top-8, TopK(Softmax) gates, one shared SwiGLU expert. MegaBlocks router chapter §2: p-norm
normalisation of the top-k weights; a benchmark switch forcing uniform assignment."""

import zlib

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from gpu_util import (LOGIT_RTOL, RTOL, assert_close, compare_route, gate_rtol, gpu_route,
                      oracle_cfg, route_np, to_np)
from top_gating_expert_gb300 import _native as N
from top_gating_expert_gb300 import moe
from top_gating_expert_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


def _cfg(**kw):
    base = dict(S=1000, G=1, E=16, M=256, H=256, k=2, capacity_factor=0.0, random_routing=0,
                n_shared=0, H_shared=0, act="relu", dtype="bf16", bias=False)
    base.update(kw)
    return base


CASES = {
    # DeepSeek-V3-like routing at a small width: 256 experts in 8 groups, 4 kept, top-8,
    # un-normalised gates, one shared SwiGLU expert; ragged token count
    "deepseek_groups_none": _cfg(S=700, E=256, k=8, M=256, H=128, act="swiglu", n_shared=1,
                                 H_shared=128, n_expert_groups=8, topk_groups=4,
                                 gate_norm="none"),
    # p = 2 normalisation with capacity, 2 groups of tokens, k = 3
    "pnorm2_capacity_k3": _cfg(S=1536, G=2, E=16, k=3, capacity_factor=1.0, gate_norm="pnorm",
                               gate_p=2.0),
    # group limit + random routing + p = 0.5
    "groups_rr_pnorm05": _cfg(S=1024, G=4, E=32, k=2, capacity_factor=1.25, random_routing=1,
                              n_expert_groups=4, topk_groups=1, gate_norm="pnorm", gate_p=0.5),
    # benchmark uniform assignment with capacity
    "uniform_capacity": _cfg(S=2048, E=8, k=2, capacity_factor=1.0, uniform_assignment=1),
    # the fp32 path with groups and TopK(Softmax) gates
    "f32_groups_none": _cfg(S=300, E=12, k=3, M=32, H=64, dtype="f32", n_expert_groups=3,
                            topk_groups=2, gate_norm="none", capacity_factor=1.0),
    # no variant, top-6 of 128 (the selection's threshold pass) through both entry points
    "plain_top6_E128": _cfg(S=900, G=3, E=128, k=6, capacity_factor=1.0),
    # 16 single-expert groups (E = 16): group-limited = plain top-k over the kept groups
    "sixteen_groups": _cfg(S=640, E=16, k=4, n_expert_groups=16, topk_groups=5, bias=True),
}


@pytest.fixture(scope="module", params=sorted(CASES))
def run(request, native_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    name = request.param
    cfg = CASES[name]
    assert moe.validate(cfg) == 0
    inp = make_inputs(cfg, seed=zlib.crc32(name.encode()) % 10000)
    layer = moe.MoeLayer(cfg, inp.host)
    x = inp.host["x"].cuda()
    u = inp.host["u"].cuda() if cfg["random_routing"] else None
    y = layer.forward(x, u)
    status = moe.device_status(layer.ws)
    return dict(name=name, cfg=cfg, inp=inp, layer=layer, x=x, u=u, y=to_np(y),
                logits=to_np(layer.logits), route=route_np(layer.route_out), status=status)


def test_status_ok(run):
    assert run["status"] == 0


def test_route_bit_exact_from_gpu_logits(run):
    cfg = run["cfg"]
    o = O.route(run["logits"], oracle_cfg(cfg), run["inp"].np["u"])
    compare_route(run["route"], o, run["name"], gate_rtol(cfg, run["logits"]))


def test_logits_vs_oracle(run):
    a = run["inp"].np
    ref = O.router_logits(a["x"], a["W_g"], a.get("bias"))
    assert_close(run["logits"], ref, LOGIT_RTOL[run["cfg"]["dtype"]], "logits")


def test_unfused_entry_points_agree(run):
    """moe_router + moe_route give the same logits and routing as the layer's call."""
    cfg, layer = run["cfg"], run["layer"]
    ws = moe.workspace(cfg, N.MOE_WS_STEP, "cuda")
    out = moe.RouteOutputs.allocate(cfg, "cuda")
    lg = torch.empty((cfg["S"], cfg["E"]), dtype=torch.float32, device="cuda")
    moe.router(cfg, run["x"], layer.W_g, layer.bias, lg, ws)
    moe.route(cfg, lg, run["u"], out, ws)
    assert moe.device_status(ws) == 0
    assert np.array_equal(to_np(lg), run["logits"])
    g = route_np(out)
    for key in ("expert_id", "gate", "pos", "drop_reason", "row", "counts", "counts_routed",
                "expert_offsets"):
        assert np.array_equal(g[key], run["route"][key]), key


def test_layer_output_vs_oracle(run):
    cfg, a = run["cfg"], run["inp"].np
    y_ref, _, _ = O.layer_forward(a, oracle_cfg(cfg), logits=run["logits"])
    assert_close(run["y"], y_ref, RTOL[cfg["dtype"]], run["name"])


def test_variant_structure(run):
    """What each variant guarantees whatever the logits."""
    cfg, r = run["cfg"], run["route"]
    ids = r["expert_id"].astype(np.int64)
    S, E, k = cfg["S"], cfg["E"], cfg["k"]
    if cfg.get("uniform_assignment"):
        assert np.array_equal(ids, (np.arange(S)[:, None] * k + np.arange(k)) % E)
    ng = cfg.get("n_expert_groups", 0)
    if ng and ng > 1:
        groups = ids // (E // ng)
        assert all(len(set(row)) <= cfg["topk_groups"] for row in groups.tolist())
    if cfg.get("gate_norm") == "pnorm":
        kept_all = np.all(r["pos"] >= 0, axis=1)
        p = cfg["gate_p"]
        norms = np.sum(r["gate"][kept_all].astype(np.float64) ** p, axis=1)
        assert np.allclose(norms, 1.0, rtol=1e-5)
    if cfg.get("gate_norm") == "none":
        assert np.all(r["gate"].sum(axis=1) <= 1.0 + 1e-6)


# tie-heavy logits straight into moe_route: group maxima tie, expert logits tie
TIE_CASES = {
    "group_ties_top1": dict(S=512, G=1, E=32, k=2, capacity_factor=0.0, n_expert_groups=8,
                            topk_groups=3),
    "group_ties_none_capacity": dict(S=777, G=3, E=64, k=6, capacity_factor=0.8,
                                     n_expert_groups=16, topk_groups=4, gate_norm="none"),
    "uniform_ties": dict(S=300, G=1, E=24, k=5, capacity_factor=0.5, uniform_assignment=1),
}


@pytest.mark.parametrize("name", sorted(TIE_CASES))
def test_tie_heavy_routing(name, native_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cfg = dict(M=64, H=64, act="relu", dtype="bf16", random_routing=0, n_shared=0, H_shared=0,
               **TIE_CASES[name])
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    logits = (rng.integers(-2, 3, size=(cfg["S"], cfg["E"])) * 0.5).astype(np.float32)
    out, status = gpu_route(cfg, logits, None)
    assert status == 0
    o = O.route(logits, oracle_cfg(cfg), None)
    compare_route(route_np(out), o, name, gate_rtol(cfg, logits))
