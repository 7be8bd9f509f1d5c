"""GPU routing parity: given identical fp32 logits and u, expert ids, slots, drop masks,
rows, counts and offsets are bit-exact with the oracle; gates and losses within tolerance."""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from gpu_util import compare_route, gpu_route, oracle_cfg, route_np
from top_gating_expert_gb300 import moe
from top_gating_expert_gb300.inputs import PRESETS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(native_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _case(S, G, E, k, cf, rr, seed=0, kind="normal", M=64, H=128):
    return dict(S=S, G=G, E=E, k=k, capacity_factor=cf, random_routing=rr, M=M, H=H,
                n_shared=0, H_shared=0, act="relu", dtype="bf16"), seed, kind


CASES = {
    # several chunks, ragged last chunk inside each group, non-power-of-two E
    "ragged_groups_E5_k3": _case(1000, 4, 5, 3, 0.5, 0),
    "E256_k8_dropless": _case(777, 1, 256, 8, 0.0, 0),
    "E1_k1": _case(300, 1, 1, 1, 1.0, 0),
    "one_token_per_group": _case(64, 64, 8, 2, 1.0, 1),
    "coarse_ties_rr": _case(2048, 2, 16, 2, 1.0, 1, kind="coarse"),
    "all_equal_logits": _case(1536, 3, 32, 2, 1.0, 0, kind="equal"),
    "skewed_to_expert0": _case(4096, 1, 64, 2, 1.25, 0, kind="skew"),
    "E128_k2_groups_rr": _case(8192, 8, 128, 2, 1.0, 1),
    "E64_k6_dropless": _case(5000, 1, 64, 6, 0.0, 0),
    "E48_k4_cap": _case(3000, 2, 48, 4, 2.0, 0),
    # 4 <= k <= lanes a token: the selection keeps only logits at or above the smallest lane
    # maximum; with ties at that bound, all-equal rows and a dominant expert
    "coarse_ties_E128_k6": _case(1500, 3, 128, 6, 1.0, 0, kind="coarse"),
    "all_equal_E200_k8": _case(640, 1, 200, 8, 0.0, 0, kind="equal"),
    "skew_E96_k5": _case(1200, 1, 96, 5, 1.5, 0, kind="skew"),
}


def _logits(S, E, seed, kind):
    rng = np.random.default_rng(seed + 17)
    if kind == "coarse":
        l = rng.integers(-4, 5, size=(S, E)).astype(np.float32) * 0.25
    elif kind == "equal":
        l = np.zeros((S, E), np.float32)
    elif kind == "skew":
        l = rng.standard_normal((S, E)).astype(np.float32)
        l[:, 0] += 4.0
    else:
        l = (rng.standard_normal((S, E)) * 2).astype(np.float32)
    return l, rng.random(S, dtype=np.float32)


@pytest.mark.parametrize("name", sorted(CASES))
def test_route_parity_cases(name):
    cfg, seed, kind = CASES[name]
    logits, u = _logits(cfg["S"], cfg["E"], seed, kind)
    out, status = gpu_route(cfg, logits, u if cfg["random_routing"] else None)
    assert status == 0
    o = O.route(logits, oracle_cfg(cfg), u)
    compare_route(route_np(out), o, name)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_route_parity_presets_full_size(n):
    """Full-size routing on the preset's own logits (oracle router, rounded to fp32)."""
    cfg = PRESETS[n]
    inp = make_inputs(cfg, preset_number=n, names=("x", "W_g", "u", "bias"))
    logits = O.router_logits(inp.np["x"], inp.np["W_g"], inp.np.get("bias")).astype(np.float32)
    out, status = gpu_route(cfg, logits, inp.np["u"] if cfg["random_routing"] else None)
    assert status == 0
    compare_route(route_np(out), O.route(logits, oracle_cfg(cfg), inp.np["u"]), f"preset {n}")


def test_route_is_deterministic():
    cfg, seed, kind = CASES["E128_k2_groups_rr"]
    logits, u = _logits(cfg["S"], cfg["E"], 5, kind)
    a, _ = gpu_route(cfg, logits, u)
    b, _ = gpu_route(cfg, logits, u)
    for f in ("expert_id", "pos", "row", "token_of", "gate", "w_perm", "aux_loss", "z_loss"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f


def test_nonfinite_logits_reported_on_host():
    cfg, _, _ = CASES["E48_k4_cap"]
    logits, u = _logits(cfg["S"], cfg["E"], 1, "normal")
    logits[17, 3] = np.nan
    logits[400, 0] = np.inf
    _, status = gpu_route(cfg, logits, None)
    assert status == -6  # MOE_ERR_NONFINITE, context still usable
    logits2, _ = _logits(cfg["S"], cfg["E"], 2, "normal")
    _, status2 = gpu_route(cfg, logits2, None)
    assert status2 == 0
