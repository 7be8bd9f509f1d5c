"""The routing variants the benchmark times, at its full size: preset 2's 16384 tokens in 16
groups (x, W_g and u of that preset; a seeded 256-row router for DeepSeek-V3's routing),
through the fused moe_router_route as the benchmark calls it, with the logits kept. The
oracle routes from those logits; routing must be bit-exact (ids, slots, drops, rows,
counts, offsets) and the gates within their fp32 bound."""

import os
import sys

import pytest
import torch

from gpu_util import compare_route, gate_rtol, oracle_cfg, route_np, to_np
from oracle import moe_oracle as O
from top_gating_expert_gb300 import _native as N
from top_gating_expert_gb300 import moe
from top_gating_expert_gb300.inputs import PRESETS, make_inputs

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def preset2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return make_inputs(PRESETS[2], preset_number=2, names=("x", "W_g"))


@pytest.mark.parametrize("name", sorted(bench.VARIANTS))
def test_bench_variant_routing_full_size(name, preset2, native_lib):
    cfg = dict(PRESETS[2], **bench.VARIANTS[name])
    assert moe.validate(cfg) == 0
    x = preset2.host["x"].cuda()
    if cfg["E"] != PRESETS[2]["E"]:
        W_g = bench.variant_router_weights(cfg["E"], cfg["M"]).to(torch.bfloat16).cuda()
    else:
        W_g = preset2.host["W_g"].cuda()
    u = preset2.host["u"].cuda() if cfg["random_routing"] else None
    out = moe.RouteOutputs.allocate(cfg, "cuda")
    ws = moe.workspace(cfg, N.MOE_WS_STEP, "cuda")
    logits = torch.empty((cfg["S"], cfg["E"]), dtype=torch.float32, device="cuda")
    moe.router_route(cfg, x, W_g, None, u, logits, out, ws)
    assert moe.device_status(ws) == 0
    lg = to_np(logits)
    o = O.route(lg, oracle_cfg(cfg), preset2.np["u"])
    compare_route(route_np(out), o, name, gate_rtol(cfg, lg))
