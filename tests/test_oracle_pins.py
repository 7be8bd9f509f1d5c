"""Pins for the CPU oracle: brute force, hand-worked examples, closed forms, invariants and
library routines. None of these re-types the oracle's own formulas."""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from bruteforce import bf_route, bf_layer, bf_capacity
from top_gating_expert_gb300.inputs import PRESETS, make_inputs, preset

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _tiny_logits(rng, S, E, coarse):
    if coarse:  # values on a coarse grid, so many exact ties occur
        return rng.integers(-3, 4, size=(S, E)).astype(np.float64) * 0.5
    return rng.standard_normal((S, E))


def _cfg(S, G, E, k, cf, rr):
    return dict(S=S, G=G, E=E, k=k, capacity_factor=cf, random_routing=rr, M=4, H=4,
                act="relu", n_shared=0)


# ---------------------------------------------------------------- hand-worked example
def test_worked_example_matches_hand_derivation():
    with open(os.path.join(GOLDEN, "route_worked_example.json")) as f:
        g = json.load(f)
    cfg = dict(g["config"], M=4, H=4, act="relu")
    r = O.route(np.array(g["logits"], float), cfg, np.array(g["u"], np.float32))
    exp = g["expected"]
    assert r["capacity"] == exp["capacity"]
    for key in ("expert_id", "pos", "drop_reason", "counts", "counts_routed",
                "expert_offsets", "row", "token_of"):
        np.testing.assert_array_equal(np.asarray(r[key]), np.asarray(exp[key]), err_msg=key)
    fully = [t for t in range(cfg["S"]) if np.all(r["pos"][t] < 0)]
    assert fully == exp["fully_dropped_tokens"]
    # gates: softmax over the two selected logits, zero where dropped (closed form)
    L = g["logits"]
    for t, (e1, e2) in enumerate(exp["expert_id"]):
        d = L[t][e1] - L[t][e2]
        g1, g2 = 1.0 / (1.0 + math.exp(-d)), 1.0 / (1.0 + math.exp(d))
        want = [g1 if exp["pos"][t][0] >= 0 else 0.0, g2 if exp["pos"][t][1] >= 0 else 0.0]
        np.testing.assert_allclose(r["gate"][t], want, rtol=1e-15, atol=0)


# ---------------------------------------------------------------- brute force
CASES = [(S, G, E, k, cf, rr, coarse)
         for (S, G) in ((8, 1), (16, 2), (64, 4), (48, 3))
         for E in (2, 5, 8)
         for k in (1, 2, 3)
         for cf in (0.0, 0.5, 1.0, 1.25)
         for rr in (0, 1)
         for coarse in (False, True)
         if k <= E and not (rr and k != 2)]


@pytest.mark.parametrize("S,G,E,k,cf,rr,coarse", CASES)
def test_route_matches_brute_force(S, G, E, k, cf, rr, coarse):
    rng = np.random.default_rng(hash((S, G, E, k, cf, rr, coarse)) % (2 ** 32))
    logits = _tiny_logits(rng, S, E, coarse)
    u = rng.random(S, dtype=np.float32)
    cfg = _cfg(S, G, E, k, cf, rr)
    r = O.route(logits, cfg, u)
    b = bf_route(logits.tolist(), cfg, u)
    assert r["capacity"] == b["capacity"]
    for key in ("expert_id", "pos", "drop_reason", "counts", "counts_routed", "row",
                "token_of", "expert_offsets"):
        np.testing.assert_array_equal(np.asarray(r[key]), np.asarray(b[key]), err_msg=key)
    np.testing.assert_allclose(r["gate"], np.asarray(b["gate"]), rtol=1e-13, atol=1e-15)
    assert r["aux_loss"] == pytest.approx(b["aux_loss"], rel=1e-12)
    assert r["z_loss"] == pytest.approx(b["z_loss"], rel=1e-12)


@pytest.mark.parametrize("act", ["relu", "swiglu"])
@pytest.mark.parametrize("cf,rr,n_shared", [(1.0, 1, 0), (0.0, 0, 0), (0.5, 0, 2)])
def test_layer_matches_brute_force(act, cf, rr, n_shared):
    rng = np.random.default_rng(7)
    S, G, E, M, H, k = 16, 2, 4, 6, 5, 2
    cfg = dict(S=S, G=G, E=E, M=M, H=H, k=k, capacity_factor=cf, random_routing=rr,
               n_shared=n_shared, H_shared=3, act=act)
    arr = dict(x=rng.standard_normal((S, M)), W_g=rng.standard_normal((E, M)),
               W_in=rng.standard_normal((E, H, M)), W_up=rng.standard_normal((E, H, M)),
               W_out=rng.standard_normal((E, M, H)), u=rng.random(S),
               Ws_in=rng.standard_normal((n_shared, 3, M)),
               Ws_up=rng.standard_normal((n_shared, 3, M)),
               Ws_out=rng.standard_normal((n_shared, M, 3)))
    logits = arr["x"] @ arr["W_g"].T
    y, r, _ = O.layer_forward(arr, cfg, logits=logits)
    yb, rb = bf_layer(arr, cfg, logits.tolist())
    np.testing.assert_allclose(y, np.asarray(yb), rtol=1e-12, atol=1e-12)
    residual = rng.standard_normal((S, M))
    y2, _, _ = O.layer_forward(arr, cfg, logits=logits, residual=residual)
    np.testing.assert_allclose(y2, np.asarray(yb) + residual, rtol=1e-12, atol=1e-12)
    # a token subset gives the same rows
    sub = np.array([3, 0, 9])
    y3, _, _ = O.layer_forward(arr, cfg, logits=logits, tokens=sub)
    np.testing.assert_allclose(y3, y[sub], rtol=1e-14, atol=1e-14)


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("n", [1, 2, 5])
def test_capacity_is_2N_over_GE(n):
    """cf = 1, k = 2 reproduces GShard's 2N/(G*E); cf = 1.25 scales it."""
    c = PRESETS[n]
    C = O.capacity(c["S"], c["G"], c["E"], c["k"], c["capacity_factor"])
    want = {1: 2 * 256 // (1 * 8), 2: 2 * 16384 // (16 * 128), 5: int(1.25 * 2 * 65536 // 64)}[n]
    assert C == want == bf_capacity(c["S"], c["G"], c["E"], c["k"], c["capacity_factor"])
    assert O.capacity(8, 2, 3, 2, 0.0) is None


def test_k1_is_switch_argmax():
    rng = np.random.default_rng(3)
    l = rng.integers(-2, 3, size=(500, 7)).astype(float)  # many ties
    ids = O.top_k(l, 1)[:, 0]
    np.testing.assert_array_equal(ids, np.argmax(l, axis=1))  # first occurrence on ties
    g = O.top_k_gates(l, O.top_k(l, 1))
    assert np.all(g == 1.0)


def test_topk_gates_equal_renormalised_softmax():
    """Softmax(KeepTopK(l)) equals the full softmax's top-k probabilities renormalised."""
    rng = np.random.default_rng(4)
    l = rng.standard_normal((300, 16)) * 3
    ids = O.top_k(l, 4)
    g = O.top_k_gates(l, ids)
    p = torch.softmax(torch.from_numpy(l), dim=1).numpy()
    pk = np.take_along_axis(p, ids, axis=1)
    np.testing.assert_allclose(g, pk / pk.sum(1, keepdims=True), rtol=1e-13)
    np.testing.assert_allclose(g.sum(1), 1.0, rtol=1e-14)
    # ids agree with torch.topk on tie-free values (descending order)
    np.testing.assert_array_equal(ids, torch.topk(torch.from_numpy(l), 4, dim=1).indices.numpy())


def test_z_loss_closed_forms():
    E = 7
    assert O.z_loss(np.zeros((5, E))) == pytest.approx(math.log(E) ** 2, rel=1e-15)
    assert O.z_loss(np.full((3, E), 2.5)) == pytest.approx((2.5 + math.log(E)) ** 2, rel=1e-15)
    l = np.array([[0.0, math.log(3.0)]])  # lse = ln 4
    assert O.z_loss(l) == pytest.approx(math.log(4.0) ** 2, rel=1e-15)


def test_aux_loss_closed_forms():
    E, S, k = 8, 64, 2
    # uniform router probabilities: aux = 1 whatever the counts
    counts = np.zeros((1, E), int); counts[0, :k] = S
    assert O.aux_loss(np.zeros((S, E)), counts, 1, k) == pytest.approx(1.0, rel=1e-14)
    # everything to expert 0 with probability ~1 at k = 1: aux = E
    l = np.zeros((S, E)); l[:, 0] = 60.0
    c1 = np.zeros((1, E), int); c1[0, 0] = S
    assert O.aux_loss(l, c1, 1, 1) == pytest.approx(E, rel=1e-12)
    # perfectly balanced counts with uniform P: 1
    cb = np.full((1, E), S * k // E)
    assert O.aux_loss(np.zeros((S, E)), cb, 1, k) == pytest.approx(1.0, rel=1e-14)


def test_aux_loss_equals_other_pages_forms():
    """Equal to MegaBlocks' E/(tokens*top_k) * dot(tokens_per_expert, mean scores) and to
    the DeepSeek form sum_i f_i P_i with f_i = (E/K) * count_i / S, written here with torch."""
    rng = np.random.default_rng(5)
    S, E, k = 200, 10, 3
    l = rng.standard_normal((S, E)) * 2
    r = O.route(l, dict(S=S, G=1, E=E, k=k, capacity_factor=0.0, random_routing=0))
    lt = torch.from_numpy(l)
    scores = torch.softmax(lt, dim=1)
    tpe = torch.bincount(torch.topk(lt, k, dim=1).indices.reshape(-1), minlength=E).double()
    megablocks = E / (S * k) * torch.dot(tpe, scores.mean(0)).item()
    deepseek = torch.sum((E / k) * tpe / S * scores.mean(0)).item()
    assert r["aux_loss"] == pytest.approx(megablocks, rel=1e-13)
    assert r["aux_loss"] == pytest.approx(deepseek, rel=1e-13)


def test_random_routing_special_cases_and_rate():
    rng = np.random.default_rng(6)
    S = 200000
    l = rng.standard_normal((S, 6))
    cfg = dict(S=S, G=1, E=6, k=2, capacity_factor=0.0, random_routing=1)
    zero = O.route(l, cfg, np.zeros(S, np.float32))
    assert np.all(zero["pos"][:, 1] >= 0)            # u = 0: every 2nd choice kept
    one = O.route(l, cfg, np.ones(S, np.float32))
    assert np.all(one["drop_reason"][:, 1] == 2)       # u = 1: none kept
    tie = np.zeros((4, 6))                              # exact ties: threshold 1, always kept
    rt = O.route(tie, dict(cfg, S=4), np.full(4, 0.999999, np.float32))
    assert np.all(rt["pos"][:, 1] >= 0)
    u = rng.random(S, dtype=np.float32)
    r = O.route(l, cfg, u)
    ids = r["expert_id"]
    g2 = torch.softmax(torch.from_numpy(np.take_along_axis(l, ids, 1)), 1)[:, 1].numpy()
    p = np.minimum(1.0, 2.0 * g2)
    kept = (r["pos"][:, 1] >= 0).mean()
    sigma = math.sqrt(np.sum(p * (1 - p))) / S
    assert abs(kept - p.mean()) < 4 * sigma
    # first choices are never random-dropped
    assert np.all(r["pos"][:, 0] >= 0)


def test_combine_pairs_gates_with_their_expert():
    """With expert e's FFN output set to the one-hot vector of e, y[t, e_j] = gate_j."""
    rng = np.random.default_rng(8)
    S, E, k = 40, 6, 3
    l = rng.standard_normal((S, E))
    cfg = dict(S=S, G=2, E=E, k=k, capacity_factor=0.5, random_routing=0)
    r = O.route(l, cfg)
    ffn_out = np.eye(E)[np.asarray([r["expert_id"][t, j] for t, j in
                                    zip(r["token_of"], r["choice_of"])], dtype=int)]
    y = O.combine(ffn_out, r, np.arange(S))
    for t in range(S):
        want = np.zeros(E)
        for j in range(k):
            if r["pos"][t, j] >= 0:
                want[r["expert_id"][t, j]] = r["gate_raw"][t, j]
        np.testing.assert_array_equal(y[t], want)
    # identity experts: tokens with all k kept get back x; fully dropped ones get 0
    x = rng.standard_normal((S, 5))
    ident = O.dispatch(x, r["token_of"])
    yi = O.combine(ident, r, np.arange(S))
    allk = np.all(r["pos"] >= 0, axis=1)
    none = np.all(r["pos"] < 0, axis=1)
    np.testing.assert_allclose(yi[allk], x[allk], rtol=1e-14, atol=1e-15)
    assert np.all(yi[none] == 0.0)


@pytest.mark.parametrize("act", ["relu", "swiglu"])
def test_ffn_reduces_to_dense_library_ffn(act):
    """One expert, all tokens: a dense two-layer FFN written with torch (fp64)."""
    rng = np.random.default_rng(9)
    n, M, H = 33, 24, 40  # non-square so a transposed operand cannot pass
    x, Wi, Wu, Wo = (rng.standard_normal(s) for s in ((n, M), (H, M), (H, M), (M, H)))
    y = O.expert_ffn(x, Wi, Wo, act, Wu)
    fc1 = torch.nn.functional.linear(torch.from_numpy(x), torch.from_numpy(Wi))
    if act == "relu":
        h = torch.relu(fc1)
    else:
        h = torch.nn.functional.silu(fc1) * torch.nn.functional.linear(torch.from_numpy(x), torch.from_numpy(Wu))
    want = torch.nn.functional.linear(h, torch.from_numpy(Wo)).numpy()
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)


def test_two_shared_experts_equal_one_with_concatenated_hidden():
    """Summing two experts equals one expert whose hidden units are both sets (the
    split-FFN identity the L16 notes ask the reader to check in NumPy)."""
    rng = np.random.default_rng(10)
    n, M, H = 9, 12, 7
    x = rng.standard_normal((n, M))
    Wi, Wu, Wo = rng.standard_normal((2, H, M)), rng.standard_normal((2, H, M)), rng.standard_normal((2, M, H))
    cfg = dict(n_shared=2, act="swiglu", M=M)
    s = O.shared_ffn(x, dict(Ws_in=Wi, Ws_up=Wu, Ws_out=Wo), cfg)
    cat = O.expert_ffn(x, np.concatenate(Wi), np.concatenate(Wo, axis=1), "swiglu", np.concatenate(Wu))
    np.testing.assert_allclose(s, cat, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- invariants on the presets
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_route_invariants_on_presets(n):
    cfg = PRESETS[n]
    inp = make_inputs(cfg, preset_number=n, names=("x", "W_g", "u", "bias"))
    logits = O.router_logits(inp.np["x"], inp.np["W_g"], inp.np.get("bias")).astype(np.float32)
    r = O.route(logits, cfg, inp.np["u"])
    S, G, E, k = cfg["S"], cfg["G"], cfg["E"], cfg["k"]
    ids, pos, counts = r["expert_id"], r["pos"], r["counts"]
    # at most k distinct experts per token
    assert all(len(set(row)) == k for row in ids[: min(S, 4096)])
    C = r["capacity"]
    if C is not None:
        assert counts.max() <= C
    else:
        assert np.all(pos >= 0)  # dropless keeps everything
    kept = pos >= 0
    assert counts.sum() == kept.sum() == r["expert_offsets"][-1]
    Sg = S // G
    for g in range(G):
        for e in range(E):
            sel = (ids[g * Sg:(g + 1) * Sg] == e) & kept[g * Sg:(g + 1) * Sg]
            p = np.sort(pos[g * Sg:(g + 1) * Sg][sel])
            np.testing.assert_array_equal(p, np.arange(counts[g, e]))
    assert r["counts_routed"].sum() == S * k
    np.testing.assert_allclose(np.where(kept, r["gate_raw"], 0).sum(1)[kept.all(1)], 1.0, rtol=1e-12)
    # token_of inverts row
    tt, jj = np.nonzero(kept)
    np.testing.assert_array_equal(r["token_of"][r["row"][tt, jj]], tt)
    if n == 5:
        drop = 1.0 - kept.mean()
        assert 0.2 < drop < 0.45, drop  # the skewed workload overflows substantially
