"""Degenerate and edge cases of the whole layer (moe_layer_forward) against the oracle routed
from the GPU's logits: experts with no rows, a single expert, every token to every expert,
near-total overflow, a single token, ragged token counts with groups."""

import zlib

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from gpu_util import RTOL, assert_close, compare_route, oracle_cfg, route_np, to_np
from top_gating_expert_gb300 import moe
from top_gating_expert_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


def _cfg(**kw):
    base = dict(S=512, G=1, E=8, M=128, H=256, k=2, capacity_factor=0.0, random_routing=0,
                n_shared=0, H_shared=0, act="relu", dtype="bf16", bias=False)
    base.update(kw)
    return base


CASES = {
    "one_expert_takes_all": (_cfg(S=700, E=16, k=1), "bias0"),
    "single_expert": (_cfg(S=300, E=1, k=1), None),
    "every_token_every_expert": (_cfg(S=256, E=4, k=4, act="swiglu"), None),
    "near_total_overflow": (_cfg(S=1024, G=4, E=8, capacity_factor=0.02), None),
    "single_token": (_cfg(S=1, E=8, k=2, capacity_factor=1.0, random_routing=1), None),
    "ragged_groups_shared": (_cfg(S=387, G=3, E=6, k=3, capacity_factor=1.5, act="swiglu",
                                  n_shared=1, H_shared=128), None),
    "fp32_all_to_one": (_cfg(S=200, E=4, k=2, M=32, H=64, dtype="f32", capacity_factor=1.0), "bias0"),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_layer_edge_case(name, native_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cfg, twist = CASES[name]
    inp = make_inputs(cfg, seed=zlib.crc32(name.encode()) % 10000)
    weights = dict(inp.host)
    if twist == "bias0":  # a router bias that sends (almost) every token to expert 0 first
        b = np.zeros(cfg["E"], np.float32)
        b[0] = 50.0
        weights["bias"] = torch.from_numpy(b)
        inp.np["bias"] = b
    layer = moe.MoeLayer(cfg, weights)
    x = inp.host["x"].cuda()
    u = inp.host["u"].cuda() if cfg["random_routing"] else None
    y = layer.forward(x, u, residual=x)
    assert moe.device_status(layer.ws) == 0
    logits = to_np(layer.logits)
    ocfg = oracle_cfg(cfg)
    o = O.route(logits, ocfg, inp.np["u"])
    compare_route(route_np(layer.route_out), o, name)
    y_ref, _, _ = O.layer_forward(inp.np, ocfg, logits=logits, residual=inp.np["x"])
    assert_close(to_np(y), y_ref, RTOL[cfg["dtype"]], name)
    dropped = np.all(o["pos"] < 0, axis=1)
    if dropped.any() and not cfg["n_shared"]:
        assert np.array_equal(to_np(y)[dropped], inp.np["x"][dropped])
    if name == "one_expert_takes_all":
        assert (o["counts"].sum(0) > 0).sum() == 1  # every other expert has no rows
