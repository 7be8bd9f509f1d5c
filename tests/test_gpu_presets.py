"""The five workload presets at full size, through moe_layer_forward (the call the
benchmark times): routing bit-exact over all tokens against the oracle routed from the
GPU's own logits; the layer output against the oracle, element by element, on every token
of presets 1, 2, 4 and 5 and, for preset 3 (whose oracle is the slowest), on every token
that owns a row of each expert's first and last 256-row m-tile (the GEMMs' CTA-pair tile),
plus a random sample; logits against the oracle's own fp64 logits on a sample; and the
tokens whose routing a near-tie changes counted apart."""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from gpu_util import (LOGIT_RTOL, RTOL, assert_close, compare_route, near_tie_tokens, oracle_cfg,
                      route_np, to_np)
from top_gating_expert_gb300 import moe
from top_gating_expert_gb300.inputs import PRESETS, make_inputs

pytestmark = pytest.mark.gpu

TILE_ROWS = 256  # rows of one output tile of the expert GEMMs (a CTA pair)


def tile_tokens(route: dict, tile_rows: int = TILE_ROWS) -> np.ndarray:
    """Tokens owning a row of each expert's first and last m-tile (all rows of both tiles,
    the ragged last one included)."""
    offs = np.asarray(route["expert_offsets"], np.int64)
    token_of = np.asarray(route["token_of"], np.int64)
    rows = []
    for e in range(len(offs) - 1):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi == lo:
            continue
        rows.append(np.arange(lo, min(hi, lo + tile_rows)))
        last = lo + (hi - lo - 1) // tile_rows * tile_rows
        rows.append(np.arange(last, hi))
    return np.unique(token_of[np.concatenate(rows)]) if rows else np.zeros(0, np.int64)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_preset_full_size(n, native_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cfg = PRESETS[n]
    inp = make_inputs(cfg, preset_number=n)
    layer = moe.MoeLayer(cfg, inp.host)
    dev = layer.device
    x = inp.host["x"].to(dev)
    u = inp.host["u"].to(dev) if cfg["random_routing"] else None
    residual = x if n == 5 else None  # the overflow workload: dropped tokens pass through
    y = layer.forward(x, u, residual)
    assert moe.device_status(layer.ws) == 0
    y = to_np(y)
    logits = to_np(layer.logits)
    g = route_np(layer.route_out)
    ocfg = oracle_cfg(cfg)
    a = inp.np
    S = cfg["S"]

    # (i) routing from the GPU's logits: bit-exact for every token
    o = O.route(logits, ocfg, a["u"])
    compare_route(g, o, f"preset {n}")
    dropped = np.nonzero(np.all(o["pos"] < 0, axis=1))[0]

    # router logits against the oracle's own fp64 projection on a sample
    rng = np.random.default_rng(n)
    sample = np.array(sorted(set(rng.choice(S, size=min(S, 64), replace=False).tolist())
                             | {0, S - 1} | set(dropped[:8].tolist())))
    ref_logits = O.router_logits(a["x"][sample], a["W_g"], a.get("bias"))
    assert_close(logits[sample], ref_logits, LOGIT_RTOL[cfg["dtype"]], "logits")

    # the layer output (oracle routed from the GPU logits): every token, or for preset 3
    # the tokens of each expert's first and last m-tile and the sample
    if n == 3:
        tokens = np.union1d(tile_tokens(o), sample)
    else:
        tokens = np.arange(S)
    y_ref, _, _ = O.layer_forward(a, ocfg, logits=logits, tokens=tokens,
                                  residual=None if residual is None else a["x"])
    maxrel = assert_close(y[tokens], y_ref, RTOL[cfg["dtype"]], f"y preset {n}")
    if len(dropped) and residual is not None:
        assert np.array_equal(y[dropped], a["x"][dropped])  # pure pass-through

    # (ii) the oracle's own routing: tokens that differ must sit on a near-tie
    own = O.route(O.router_logits(a["x"], a["W_g"], a.get("bias")), ocfg, a["u"])
    differ = np.nonzero(np.any(own["expert_id"] != o["expert_id"], axis=1))[0]
    loose = set(near_tie_tokens(logits, cfg["k"], gap=1e-4).tolist())
    assert set(differ.tolist()) <= loose, sorted(set(differ.tolist()) - loose)[:10]
    cascade = np.nonzero(np.any((own["pos"] >= 0) != (o["pos"] >= 0), axis=1))[0]
    print(f"preset {n}: y compared on {len(tokens)} of {S} tokens (max rel err {maxrel:.3e}), "
          f"kept {float((o['pos'] >= 0).mean()):.4f}, near-tie tokens (gap<1e-6) "
          f"{len(near_tie_tokens(logits, cfg['k']))}, ids changed by near-ties {len(differ)}, "
          f"drop status changed (incl. cascades) {len(cascade)}")
