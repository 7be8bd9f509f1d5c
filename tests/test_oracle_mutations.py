"""Plant plausible mistakes in the oracle (on the CPU, by monkeypatching) and check that
its pins catch each one: the pins are only worth something if a wrong oracle fails them."""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from bruteforce import bf_route, bf_layer

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_ok():
    with open(os.path.join(GOLDEN, "route_worked_example.json")) as f:
        g = json.load(f)
    cfg = dict(g["config"], M=4, H=4, act="relu")
    r = O.route(np.array(g["logits"], float), cfg, np.array(g["u"], np.float32))
    return all(np.array_equal(np.asarray(r[k]), np.asarray(v)) for k, v in g["expected"].items()
               if k in r)


def _bruteforce_ok():
    rng = np.random.default_rng(11)
    for S, G, E, k, cf, rr in ((16, 2, 4, 2, 0.75, 1), (24, 1, 5, 3, 0.5, 0), (16, 4, 3, 2, 0.0, 0)):
        logits = rng.integers(-3, 4, size=(S, E)).astype(float) * 0.5
        u = rng.random(S, dtype=np.float32)
        cfg = dict(S=S, G=G, E=E, k=k, capacity_factor=cf, random_routing=rr)
        r, b = O.route(logits, cfg, u), bf_route(logits.tolist(), cfg, u)
        for key in ("expert_id", "pos", "drop_reason", "counts", "row", "token_of"):
            if not np.array_equal(np.asarray(r[key]), np.asarray(b[key])):
                return False
        if abs(r["aux_loss"] - b["aux_loss"]) > 1e-9 or abs(r["z_loss"] - b["z_loss"]) > 1e-9:
            return False
        if not np.allclose(r["gate"], np.asarray(b["gate"]), rtol=1e-12):
            return False
    return True


def _closed_forms_ok():
    E = 7
    if abs(O.z_loss(np.zeros((5, E))) - math.log(E) ** 2) > 1e-12:
        return False
    l = np.zeros((64, 8)); l[:, 0] = 60.0
    c = np.zeros((1, 8), int); c[0, 0] = 64
    return abs(O.aux_loss(l, c, 1, 1) - 8) < 1e-9


def _layer_ok():
    rng = np.random.default_rng(12)
    S, E, M, H, k = 12, 3, 5, 4, 2
    for act in ("relu", "swiglu"):
        cfg = dict(S=S, G=1, E=E, M=M, H=H, k=k, capacity_factor=0.0, random_routing=0,
                   n_shared=1, H_shared=3, act=act)
        arr = dict(x=rng.standard_normal((S, M)), W_g=rng.standard_normal((E, M)),
                   W_in=rng.standard_normal((E, H, M)), W_up=rng.standard_normal((E, H, M)),
                   W_out=rng.standard_normal((E, M, H)), Ws_in=rng.standard_normal((1, 3, M)),
                   Ws_up=rng.standard_normal((1, 3, M)), Ws_out=rng.standard_normal((1, M, 3)))
        logits = arr["x"] @ arr["W_g"].T
        try:
            y, _, _ = O.layer_forward(arr, cfg, logits=logits)
        except Exception:
            return False
        yb, _ = bf_layer(arr, cfg, logits.tolist())
        if not np.allclose(y, np.asarray(yb), rtol=1e-10, atol=1e-10):
            return False
    return True


def _rr_rate_ok():
    rng = np.random.default_rng(13)
    S = 50000
    l = rng.standard_normal((S, 4))
    r = O.route(l, dict(S=S, G=1, E=4, k=2, capacity_factor=0.0, random_routing=1),
                rng.random(S, dtype=np.float32))
    g2 = torch.softmax(torch.from_numpy(np.take_along_axis(l, r["expert_id"], 1)), 1)[:, 1].numpy()
    p = np.minimum(1, 2 * g2)
    return abs((r["pos"][:, 1] >= 0).mean() - p.mean()) < 4 * math.sqrt(np.sum(p * (1 - p))) / S


def all_pins_ok():
    return _golden_ok() and _bruteforce_ok() and _closed_forms_ok() and _layer_ok() and _rr_rate_ok()


def test_unmutated_oracle_passes_every_pin():
    assert all_pins_ok()


# --- the mutations -------------------------------------------------------------------
def _token_major_slots(ids, candidate, G, E, C):
    S, k = ids.shape
    Sg = S // G
    pos = np.full((S, k), -1, np.int64)
    reason = np.where(candidate, 0, 2).astype(np.uint8)
    counts = np.zeros((G, E), np.int64)
    for g in range(G):
        q = np.zeros(E, np.int64)
        for t in range(g * Sg, (g + 1) * Sg):
            for j in range(k):
                if candidate[t, j]:
                    s = q[ids[t, j]]; q[ids[t, j]] += 1
                    if C is None or s < C:
                        pos[t, j] = s
                    else:
                        reason[t, j] = 1
        counts[g] = q if C is None else np.minimum(q, C)
    return pos, reason, counts


def _unstable_topk(logits, k):
    return np.argsort(-np.asarray(logits, float)[:, ::-1], axis=1, kind="stable")[:, :k] * -1 + (np.asarray(logits).shape[1] - 1)


def _rr_flipped(logits, ids, u):
    l = np.asarray(logits, float)
    l1 = np.take_along_axis(l, ids[:, :1], 1)[:, 0]
    l2 = np.take_along_axis(l, ids[:, 1:2], 1)[:, 0]
    return np.asarray(u, float) < 2.0 / (1.0 + np.exp(l2 - l1))


def _aux_without_E(logits, counts_routed, G, k):
    p, _ = O.log_softmax_parts(logits)
    Sg = p.shape[0] // G
    return sum(float(np.dot(np.asarray(counts_routed[g], float) / (Sg * k),
                            p[g * Sg:(g + 1) * Sg].mean(0))) for g in range(G)) / G


def _z_unsquared(logits):
    return float(np.mean(O.log_softmax_parts(logits)[1]))


def _capacity_floor(S, G, E, k, cf):
    return None if cf <= 0 else int(math.floor(cf * k * (S // G) / E - 1e-9))


def _ffn_swapped(x_rows, W_in, W_out, act, W_up=None):
    return _orig["expert_ffn"](x_rows, W_up if act == "swiglu" else W_in, W_out, act,
                               W_in if act == "swiglu" else None)


def _gates_full_softmax(logits, ids):
    p, _ = O.log_softmax_parts(logits)
    return np.take_along_axis(p, ids, 1)


def _rows_group_major(ids, pos, G, E, counts):
    S, k = ids.shape
    Sg = S // G
    base = np.cumsum(counts.ravel()) - counts.ravel()
    row = np.full((S, k), -1, np.int64)
    for t in range(S):
        for j in range(k):
            if pos[t, j] >= 0:
                row[t, j] = base[(t // Sg) * E + ids[t, j]] + pos[t, j]
    R = int(counts.sum())
    tok, ch = np.full(R, -1), np.full(R, -1)
    tt, jj = np.nonzero(pos >= 0)
    tok[row[tt, jj]] = tt; ch[row[tt, jj]] = jj
    offs = np.concatenate([[0], np.cumsum(counts.sum(0))])
    return row, offs, tok, ch


_orig = {name: getattr(O, name) for name in ("expert_ffn",)}

MUTATIONS = {
    "token-major slot order": ("assign_slots", _token_major_slots),
    "ties to the higher index": ("top_k", _unstable_topk),
    "random-routing sign flipped": ("random_routing_keep", _rr_flipped),
    "aux loss missing the factor E": ("aux_loss", _aux_without_E),
    "z-loss not squared": ("z_loss", _z_unsquared),
    "capacity rounded down": ("capacity", _capacity_floor),
    "gate and up projections swapped": ("expert_ffn", _ffn_swapped),
    "gates not renormalised over the top-k": ("top_k_gates", _gates_full_softmax),
    "rows ordered group-major": ("compact_rows", _rows_group_major),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(O, attr, fn)
    assert not all_pins_ok(), f"no pin caught: {name}"
