"""Pins of the oracle's routing variants (group-limited top-k, gate normalisations, uniform
assignment) against things other than the oracle's own code: hand-worked examples,
library routines for the special cases that reduce to them, invariants, and the
pure-Python brute force of tests/bruteforce.py on tiny inputs.

Sources: Lec16 Systems for MoE Models, "DeepSeek V3 MoE" (256 routed experts in 8 groups,
4 groups kept; TopK(Softmax(h W), 8)); MegaBlocks router chapter §2 (optional p-norm
normalisation of the top-k weights; a benchmark switch forcing uniform assignment)."""

import math

import numpy as np
import pytest
from scipy.special import softmax

from oracle import moe_oracle as O
from bruteforce import bf_route

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ------------------------------------------------------------------ group-limited top-k
def test_group_limited_hand_worked():
    # E = 8 in 4 groups of 2: g0 = {5, 0}, g1 = {4.9, 4.8}, g2 = {0, 0}, g3 = {4.85, 0}.
    # Group bests: 5, 4.9, 0, 4.85 -> the 2 best groups are g0, g1 (experts 0..3).
    l = np.array([[5.0, 0.0, 4.9, 4.8, 0.0, 0.0, 4.85, 0.0]])
    assert O.top_k(l, 3).tolist() == [[0, 2, 6]]                       # unrestricted
    assert O.group_limited_top_k(l, 3, 4, 2).tolist() == [[0, 2, 3]]   # 6 is in g3: out
    # one group kept: only g0's experts, so the 2nd choice is expert 1 (logit 0)
    assert O.group_limited_top_k(l, 2, 4, 1).tolist() == [[0, 1]]
    # every group kept: the plain top-k
    assert O.group_limited_top_k(l, 3, 4, 4).tolist() == [[0, 2, 6]]


def test_group_limited_ties_prefer_lower_group():
    # g0 and g1 tie on their best logit; with one group kept, g0 wins
    l = np.array([[1.0, 3.0, 3.0, 2.0]])
    assert O.group_limited_top_k(l, 2, 2, 1).tolist() == [[1, 0]]


@pytest.mark.parametrize("E,ng,tg,k", [(8, 4, 2, 2), (12, 3, 1, 3), (16, 8, 4, 4), (6, 6, 3, 2)])
def test_group_limited_reductions_and_invariants(E, ng, tg, k):
    rng = np.random.default_rng(E * 100 + ng)
    l = rng.integers(-4, 5, size=(200, E)).astype(float) * 0.25   # many ties
    ids = O.group_limited_top_k(l, k, ng, tg)
    size = E // ng
    # all groups kept: numpy's stable argsort of the negated logits
    full = O.group_limited_top_k(l, k, ng, ng)
    assert np.array_equal(full, np.argsort(-l, axis=1, kind="stable")[:, :k])
    for t in range(l.shape[0]):
        best = [l[t, g * size:(g + 1) * size].max() for g in range(ng)]
        kept = sorted(range(ng), key=lambda g: (-best[g], g))[:tg]
        chosen = ids[t].tolist()
        assert len(set(chosen)) == k
        assert all(e // size in kept for e in chosen)
        # listed by logit, ties by index
        assert chosen == sorted(chosen, key=lambda e: (-l[t, e], e))
        # nothing left out of a kept group beats the last chosen expert
        last = chosen[-1]
        for e in range(E):
            if e // size in kept and e not in chosen:
                assert (l[t, e], -e) < (l[t, last], -last)


def test_group_limited_singleton_groups_is_top_k():
    rng = np.random.default_rng(5)
    l = rng.standard_normal((50, 10))
    assert np.array_equal(O.group_limited_top_k(l, 2, 10, 3), O.top_k(l, 2))


def test_group_limited_rejects_too_few_experts():
    with pytest.raises(ValueError):
        O.group_limited_top_k(np.zeros((1, 8)), 3, 4, 1)   # one group of 2 experts, k = 3


# ------------------------------------------------------------------ gate normalisations
def test_gates_none_are_full_softmax_probabilities():
    rng = np.random.default_rng(7)
    l = rng.standard_normal((40, 6)) * 3
    ids = O.top_k(l, 6)                       # k = E: every probability, reordered
    g = O.normalised_gates(l, ids, "none")
    assert np.allclose(g, np.take_along_axis(softmax(l, axis=1), ids, axis=1), rtol=1e-13)
    assert np.allclose(g.sum(axis=1), 1.0, rtol=1e-13)
    g2 = O.normalised_gates(l, O.top_k(l, 2), "none")
    assert np.all(g2.sum(axis=1) < 1.0)       # a strict part of the distribution


def test_pnorm_special_cases():
    rng = np.random.default_rng(8)
    l = rng.standard_normal((40, 8)) * 2
    ids = O.top_k(l, 3)
    # p = 1: the renormalised top-k softmax
    assert np.allclose(O.normalised_gates(l, ids, "pnorm", 1.0), O.top_k_gates(l, ids), rtol=1e-13)
    for p in (0.5, 2.0, 3.0):
        g = O.normalised_gates(l, ids, "pnorm", p)
        assert np.allclose(np.sum(g ** p, axis=1), 1.0, rtol=1e-12)
        # invariant under a shift of a token's logits
        assert np.allclose(O.normalised_gates(l + 7.5, ids, "pnorm", p), g, rtol=1e-12)


def test_pnorm_two_hand_worked():
    # two logits 1 and 0: weights (1, e^-1) up to scale; p = 2 divides by sqrt(1 + e^-2)
    g = O.normalised_gates(np.array([[1.0, 0.0, -9.0]]), np.array([[0, 1]]), "pnorm", 2.0)
    n = math.sqrt(1.0 + math.exp(-2.0))
    assert np.allclose(g, [[1.0 / n, math.exp(-1.0) / n]], rtol=1e-14)


# ------------------------------------------------------------------ uniform assignment
def test_uniform_ids():
    ids = O.uniform_ids(12, 8, 2)
    assert ids[0].tolist() == [0, 1] and ids[4].tolist() == [0, 1] and ids[3].tolist() == [6, 7]
    assert np.array_equal(np.bincount(O.uniform_ids(64, 8, 3).ravel(), minlength=8), [24] * 8)


# ------------------------------------------------------------------ whole routing vs brute force
VARIANTS = [
    dict(S=16, G=2, E=8, k=2, capacity_factor=0.75, n_expert_groups=4, topk_groups=2),
    dict(S=24, G=1, E=6, k=3, capacity_factor=0.0, n_expert_groups=3, topk_groups=2,
         gate_norm="none"),
    dict(S=16, G=4, E=4, k=2, capacity_factor=1.0, gate_norm="pnorm", gate_p=2.0),
    dict(S=20, G=1, E=5, k=2, capacity_factor=0.5, uniform_assignment=1, gate_norm="none"),
    dict(S=16, G=2, E=8, k=2, capacity_factor=1.0, random_routing=1, n_expert_groups=2,
         topk_groups=1, gate_norm="pnorm", gate_p=0.5),
]


@pytest.mark.parametrize("i", range(len(VARIANTS)))
def test_route_variants_match_bruteforce(i):
    cfg = dict(dict(random_routing=0), **VARIANTS[i])
    rng = np.random.default_rng(40 + i)
    logits = rng.integers(-3, 4, size=(cfg["S"], cfg["E"])).astype(float) * 0.5
    u = rng.random(cfg["S"], dtype=np.float32)
    r, b = O.route(logits, cfg, u), bf_route(logits.tolist(), cfg, u)
    for key in ("expert_id", "pos", "drop_reason", "counts", "row", "token_of"):
        assert np.array_equal(np.asarray(r[key]), np.asarray(b[key])), key
    assert np.allclose(r["gate"], np.asarray(b["gate"]), rtol=1e-12)
    assert abs(r["aux_loss"] - b["aux_loss"]) < 1e-9 and abs(r["z_loss"] - b["z_loss"]) < 1e-9


def test_uniform_assignment_rejects_random_routing():
    cfg = dict(S=8, G=1, E=4, k=2, capacity_factor=0.0, random_routing=1, uniform_assignment=1)
    with pytest.raises(ValueError):
        O.route(np.zeros((8, 4)), cfg, np.zeros(8, np.float32))


def test_uniform_assignment_balances_counts_and_aux():
    # S*k a multiple of E: every expert gets S*k/E choices, so f_e = 1/E and aux = sum_e P_e = 1
    rng = np.random.default_rng(9)
    logits = rng.standard_normal((64, 8))
    r = O.route(logits, dict(S=64, G=1, E=8, k=2, capacity_factor=0.0, uniform_assignment=1))
    assert np.array_equal(r["counts_routed"][0], [16] * 8)
    assert abs(r["aux_loss"] - 1.0) < 1e-12


# ------------------------------------------------------------------ planted mistakes
def _variant_pins_ok():
    checks = [test_group_limited_hand_worked, test_group_limited_ties_prefer_lower_group,
              test_group_limited_singleton_groups_is_top_k, test_gates_none_are_full_softmax_probabilities,
              test_pnorm_special_cases, test_pnorm_two_hand_worked, test_uniform_ids,
              test_uniform_assignment_balances_counts_and_aux]
    checks += [lambda a=a: test_group_limited_reductions_and_invariants(*a)
               for a in [(8, 4, 2, 2), (12, 3, 1, 3), (16, 8, 4, 4), (6, 6, 3, 2)]]
    checks += [lambda i=i: test_route_variants_match_bruteforce(i) for i in range(len(VARIANTS))]
    try:
        for f in checks:
            f()
    except (AssertionError, ValueError):
        return False
    return True


def _groups_by_sum(logits, k, n_groups, topk_groups):
    l = np.asarray(logits, float)
    S, E = l.shape
    size = E // n_groups
    score = l.reshape(S, n_groups, size).sum(axis=2)
    kept = np.argsort(-score, axis=1, kind="stable")[:, :topk_groups]
    allowed = np.zeros((S, n_groups), bool)
    np.put_along_axis(allowed, kept, True, axis=1)
    return np.argsort(-np.where(np.repeat(allowed, size, 1), l, -np.inf), 1, kind="stable")[:, :k]


def _groups_ties_high(logits, k, n_groups, topk_groups):
    l = np.asarray(logits, float)
    S, E = l.shape
    size = E // n_groups
    best = l.reshape(S, n_groups, size).max(axis=2)[:, ::-1]
    kept = n_groups - 1 - np.argsort(-best, axis=1, kind="stable")[:, :topk_groups]
    allowed = np.zeros((S, n_groups), bool)
    np.put_along_axis(allowed, kept, True, axis=1)
    return np.argsort(-np.where(np.repeat(allowed, size, 1), l, -np.inf), 1, kind="stable")[:, :k]


_orig_gates = O.normalised_gates


def _pnorm_without_root(logits, ids, norm="softmax_topk", p=1.0):
    if norm != "pnorm":
        return _orig_gates(logits, ids, norm, p)
    probs, _ = O.log_softmax_parts(logits)
    sel = np.take_along_axis(probs, ids, axis=1)
    return sel / np.sum(np.power(sel, p), axis=1, keepdims=True)


def _none_renormalised(logits, ids, norm="softmax_topk", p=1.0):
    return _orig_gates(logits, ids, "softmax_topk" if norm == "none" else norm, p)


def _uniform_without_k(S, E, k):
    return (np.arange(S)[:, None] + np.arange(k)[None, :]) % E


VARIANT_MUTATIONS = {
    "group score = sum of its logits": ("group_limited_top_k", _groups_by_sum),
    "group ties to the higher group": ("group_limited_top_k", _groups_ties_high),
    "p-norm without the 1/p root": ("normalised_gates", _pnorm_without_root),
    "un-normalised gates renormalised": ("normalised_gates", _none_renormalised),
    "uniform ids ignore k": ("uniform_ids", _uniform_without_k),
}


def test_unmutated_variants_pass():
    assert _variant_pins_ok()


@pytest.mark.parametrize("name", sorted(VARIANT_MUTATIONS))
def test_planted_variant_mistake_is_caught(name, monkeypatch):
    attr, fn = VARIANT_MUTATIONS[name]
    monkeypatch.setattr(O, attr, fn)
    assert not _variant_pins_ok(), f"no pin caught: {name}"
