"""Brute-force restatement of the MoE routing and layer on tiny inputs, in pure Python.

Independent of the oracle's vectorised code: experts are ranked with ``sorted``, the
slot queue is walked one assignment at a time with explicit counters, losses and FFNs
are written as nested loops over Python floats. Meant for S <= 64, E <= 8.
"""

from __future__ import annotations

import math


def bf_capacity(S, G, E, k, cf):
    if cf <= 0:
        return None
    # smallest integer >= cf * k * (S/G) / E, found by counting up
    target = cf * k * (S // G) / E
    c = 0
    while c < target:
        c += 1
    return c


def bf_group_limited(row, k, n_groups, topk_groups):
    """Exhaustive search: the groups are ranked by their best logit (lower group first on
    ties) and the best topk_groups kept; among every k-subset of their experts the one
    whose members, listed by (logit desc, index asc), compare largest wins."""
    import itertools
    E = len(row)
    size = E // n_groups
    best = [max(row[g * size:(g + 1) * size]) for g in range(n_groups)]
    groups = sorted(range(n_groups), key=lambda g: (-best[g], g))[:topk_groups]
    allowed = [e for e in range(E) if e // size in groups]
    winner, win_key = None, None
    for sub in itertools.combinations(allowed, k):
        listed = sorted(sub, key=lambda e: (-row[e], e))
        key = [(-row[e], e) for e in listed]
        if win_key is None or key < win_key:
            winner, win_key = listed, key
    return winner


def bf_route(logits, cfg, u=None):
    """logits: list of S lists of E floats. Returns a dict of plain lists."""
    S, G, E, k = cfg["S"], cfg["G"], cfg["E"], cfg["k"]
    Sg = S // G
    C = bf_capacity(S, G, E, k, cfg["capacity_factor"])
    ids, gates, cand = [], [], []
    ng = int(cfg.get("n_expert_groups", 0) or 0)
    norm = cfg.get("gate_norm", "softmax_topk")
    for t in range(S):
        if ng > 1:
            order = bf_group_limited(logits[t], k, ng, int(cfg["topk_groups"]))
        else:
            order = sorted(range(E), key=lambda e: (-logits[t][e], e))[:k]
        ids.append(order)
        top = logits[t][order[0]]
        if norm == "softmax_topk":
            w = [math.exp(logits[t][e] - top) for e in order]
            tot = sum(w)
            gates.append([wi / tot for wi in w])
        else:
            mx = max(logits[t])
            den = sum(math.exp(v - mx) for v in logits[t])
            pr = [math.exp(logits[t][e] - mx) / den for e in order]
            if norm == "pnorm":
                p = float(cfg["gate_p"])
                nrm = sum(v ** p for v in pr) ** (1.0 / p)
                pr = [v / nrm for v in pr]
            gates.append(pr)
        c = [True] * k
        if cfg.get("random_routing", 0):
            l1, l2 = logits[t][order[0]], logits[t][order[1]]
            g2 = math.exp(l2) / (math.exp(l1) + math.exp(l2))
            c[1] = float(u[t]) < min(1.0, 2.0 * g2)
        cand.append(c)
    if cfg.get("uniform_assignment", 0):
        ids = [[(t * k + j) % E for j in range(k)] for t in range(S)]
    pos = [[-1] * k for _ in range(S)]
    reason = [[0] * k for _ in range(S)]
    counts = [[0] * E for _ in range(G)]
    for g in range(G):
        queue_len = [0] * E
        for j in range(k):
            for t in range(g * Sg, (g + 1) * Sg):
                e = ids[t][j]
                if not cand[t][j]:
                    reason[t][j] = 2
                    continue
                slot = queue_len[e]
                queue_len[e] += 1
                if C is not None and slot >= C:
                    reason[t][j] = 1
                    continue
                pos[t][j] = slot
                counts[g][e] += 1
    counts_routed = [[0] * E for _ in range(G)]
    for t in range(S):
        for j in range(k):
            counts_routed[t // Sg][ids[t][j]] += 1
    # rows: experts in order, inside an expert groups in order, inside a group slots
    row = [[-1] * k for _ in range(S)]
    token_of = []
    offsets = [0]
    for e in range(E):
        for g in range(G):
            for slot in range(counts[g][e]):
                for t in range(g * Sg, (g + 1) * Sg):
                    for j in range(k):
                        if ids[t][j] == e and pos[t][j] == slot:
                            row[t][j] = len(token_of)
                            token_of.append(t)
        offsets.append(len(token_of))
    # losses
    aux = 0.0
    for g in range(G):
        P = [0.0] * E
        for t in range(g * Sg, (g + 1) * Sg):
            den = sum(math.exp(v) for v in logits[t])
            for e in range(E):
                P[e] += math.exp(logits[t][e]) / den / Sg
        aux += sum(E * counts_routed[g][e] / (Sg * k) * P[e] for e in range(E))
    aux /= G
    z = sum(math.log(sum(math.exp(v) for v in logits[t])) ** 2 for t in range(S)) / S
    gate_out = [[gates[t][j] if pos[t][j] >= 0 else 0.0 for j in range(k)] for t in range(S)]
    return dict(expert_id=ids, gate=gate_out, pos=pos, drop_reason=reason, counts=counts,
                counts_routed=counts_routed, row=row, token_of=token_of,
                expert_offsets=offsets, capacity=C, aux_loss=aux, z_loss=z)


def _mat_vec(W, v):
    return [sum(W[i][m] * v[m] for m in range(len(v))) for i in range(len(W))]


def bf_ffn(xv, W_in, W_out, act, W_up=None):
    a = _mat_vec(W_in, xv)
    if act == "relu":
        h = [ai if ai > 0 else 0.0 for ai in a]
    else:
        b = _mat_vec(W_up, xv)
        h = [ai / (1.0 + math.exp(-ai)) * bi for ai, bi in zip(a, b)]
    return _mat_vec(W_out, h)


def bf_layer(arrays, cfg, logits):
    """y for every token, looping over tokens and their kept choices."""
    r = bf_route(logits, cfg, arrays.get("u"))
    S, M, k = cfg["S"], cfg["M"], cfg["k"]
    tolist = lambda a: a.tolist() if hasattr(a, "tolist") else a
    x = tolist(arrays["x"])
    y = []
    for t in range(S):
        acc = [0.0] * M
        for j in range(k):
            if r["pos"][t][j] < 0:
                continue
            e = r["expert_id"][t][j]
            W_up = tolist(arrays["W_up"][e]) if cfg["act"] == "swiglu" else None
            out = bf_ffn(x[t], tolist(arrays["W_in"][e]), tolist(arrays["W_out"][e]), cfg["act"], W_up)
            acc = [a + r["gate"][t][j] * o for a, o in zip(acc, out)]
        for s in range(cfg.get("n_shared", 0)):
            W_up = tolist(arrays["Ws_up"][s]) if cfg["act"] == "swiglu" else None
            out = bf_ffn(x[t], tolist(arrays["Ws_in"][s]), tolist(arrays["Ws_out"][s]), cfg["act"], W_up)
            acc = [a + o for a, o in zip(acc, out)]
        y.append(acc)
    return y, r
