"""The fused router + routing on layers with more 128-token chunks than the GPU has SMs,
where moe_router_route runs its persistent form (one CTA per SM walking the chunks, the
next chunk's loads and MMAs overlapping the current chunk's routing): logits bit-identical
to the separate router GEMM's (moe_router) and within tolerance of the oracle's fp64
projection; routing bit-exact against the oracle routed from those logits and equal to
moe_route's from them. The cases cover every lane count a token gets (2 and 4), tile
widths 16, 32 and 64 with E below the tile, k from 1 to 8, groups whose last chunk is
ragged, random routing, a router bias, and chunk counts that do not divide evenly over the
SMs."""

import zlib

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from gpu_util import LOGIT_RTOL, LOSS_RTOL, assert_close, compare_route, oracle_cfg, route_np, to_np
from top_gating_expert_gb300 import _native as N
from top_gating_expert_gb300 import moe
from top_gating_expert_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


def _cfg(S, G, E, k, M, cf=1.0, rr=0, bias=False):
    return dict(S=S, G=G, E=E, k=k, M=M, H=128, capacity_factor=cf, random_routing=rr,
                n_shared=0, H_shared=0, act="relu", dtype="bf16", bias=bias)


CASES = {
    # 157 chunks: five SMs take two
    "E64_k2_rr_bias": _cfg(20000, 1, 64, 2, 128, rr=1, bias=True),
    # three groups of 7717 tokens: each group's last chunk holds 37
    "E48_k3_groups_ragged": _cfg(3 * 7717, 3, 48, 3, 192, cf=1.25, bias=True),
    # 512 chunks in 4 groups, two lanes a token, a 16-wide tile, top-1
    "E16_k1_groups": _cfg(65536, 4, 16, 1, 64, cf=1.0),
    # two lanes a token, a 32-wide tile, top-8, dropless
    "E32_k8_dropless": _cfg(40000, 1, 32, 8, 256, cf=0.0),
    # four lanes, top-6 (the threshold selection), dropless, a longer K loop
    "E64_k6_dropless_M1024": _cfg(24576, 1, 64, 6, 1024, cf=0.0),
    # E below the 64-wide tile, capacity with overflow
    "E40_k2_cap": _cfg(19968 + 128 * 10, 2, 40, 2, 128, cf=0.75),
}


@pytest.fixture(scope="module", autouse=True)
def _lib(native_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("name", sorted(CASES))
def test_persistent_router_route(name):
    cfg = CASES[name]
    n_chunks = cfg["G"] * -(-(cfg["S"] // cfg["G"]) // 128)
    assert n_chunks > torch.cuda.get_device_properties(0).multi_processor_count
    inp = make_inputs(cfg, seed=zlib.crc32(name.encode()) % 9973)
    d = {k: v.cuda() for k, v in inp.host.items()}
    a = inp.np
    u = d["u"] if cfg["random_routing"] else None
    ws = moe.workspace(cfg, N.MOE_WS_STEP)
    out = moe.RouteOutputs.allocate(cfg)
    logits = torch.full((cfg["S"], cfg["E"]), float("nan"), dtype=torch.float32, device="cuda")
    moe.router_route(cfg, d["x"], d["W_g"], d.get("bias"), u, logits, out, ws)
    assert moe.device_status(ws) == 0
    lg = to_np(logits)

    # the separate router GEMM: the same logits bit for bit
    ref_logits = torch.empty_like(logits)
    moe.router(cfg, d["x"], d["W_g"], d.get("bias"), ref_logits, ws)
    assert moe.device_status(ws) == 0
    assert np.array_equal(lg, to_np(ref_logits)), "logits differ from moe_router's"
    rows = np.random.default_rng(3).choice(cfg["S"], 256, replace=False)
    assert_close(lg[rows], O.router_logits(a["x"][rows], a["W_g"], a.get("bias")),
                 LOGIT_RTOL["bf16"], "logits vs the oracle")

    # routing: bit-exact against the oracle from those logits, equal to moe_route's
    got = route_np(out)
    compare_route(got, O.route(lg, oracle_cfg(cfg), a["u"]), name)
    out2 = moe.RouteOutputs.allocate(cfg)
    moe.route(cfg, logits, u, out2, ws)
    assert moe.device_status(ws) == 0
    ref = route_np(out2)
    R = int(ref["expert_offsets"][-1])
    for key in ("expert_id", "pos", "drop_reason", "row", "counts", "counts_routed",
                "expert_offsets", "gate"):
        assert np.array_equal(got[key], ref[key]), key
    # the losses' per-chunk probability sums are added in an order that depends on the lanes
    # a token gets, which differ between the two kernels when E <= 16: within their tolerance
    for key in ("aux_loss", "z_loss"):
        x, y = float(got[key][0]), float(ref[key][0])
        assert abs(x - y) <= LOSS_RTOL * abs(y) + 1e-7, (key, x, y)
    for key in ("token_of", "w_perm"):
        assert np.array_equal(got[key][:R], ref[key][:R]), key

    # without logits_out: the same routing
    out3 = moe.RouteOutputs.allocate(cfg)
    moe.router_route(cfg, d["x"], d["W_g"], d.get("bias"), u, None, out3, ws)
    assert moe.device_status(ws) == 0
    g3 = route_np(out3)
    for key in ("expert_id", "pos", "row", "gate", "aux_loss", "z_loss"):
        assert np.array_equal(g3[key], got[key]), key
    for key in ("token_of", "w_perm"):
        assert np.array_equal(g3[key][:R], got[key][:R]), key
