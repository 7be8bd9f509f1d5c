"""CPU oracle for one GPU's Mixture-of-Experts layer forward.

TEST INFRASTRUCTURE ONLY. Only the test-suite, the smoke check and the benchmark's
CPU-baseline / reference leg may import this module. The product path (the CUDA
library and its Python binding) never imports, calls or links it, and this module
imports nothing from the product package.

Everything here is plain numpy in float64: inputs arrive as fp32 (or bf16 values held
exactly in fp32) and are upcast exactly; every dot product, softmax, sum and loss is
evaluated in fp64; the expert hidden activation is NOT rounded. A library primitive
(matmul, a stable sort, a cumulative sum) serves as one step where the definition
calls for it; nothing is blocked, fused or reordered beyond the definition.

Sources (titles of the pages, with the section followed):
  [GShard]     "GShard: Scaling Giant Models with Conditional Computation and Automatic
               Sharding" (summary page): "MoE Transformer"; "Top-2 gating" -- "Expert
               capacity", "Local group dispatching", "Auxiliary loss", "Random routing";
               "MoE 系统的重点是 dispatch/combine" (the dispatch path listing).
  [MegaBlocks] "04 · 路由、负载均衡与专家并行" (MegaBlocks router and parallelism):
               §2 router, §3 load-balancing loss, §6 shared experts.
  [Lec16]      "Lec16 Systems for MoE Models" (CMU 11-868): "Switch Transformer"
               (softmax gate, KeepTopK), "共享专家 vs. 路由专家", "MoE 训练中的负载均衡",
               "DeepSeek V3 MoE" (SwiGLU), "DeepSeek MoE 的负载均衡".
  [L16/L17]    CMU 11-868 L16/L17 notes (model parallel and MoE): "負載平衡".

Readings where the pages are silent or garbled (each is repeated in the design notes):
  R1 random routing keeps the 2nd choice iff u < 2*g2 with g2 the renormalised 2nd gate,
     i.e. probability min(1, 2*g2), evaluated in fp64; g2 = 1/(1+exp(l1-l2)).
  R2 a 2nd choice skipped by random routing takes no slot; the 1st gate is unchanged.
  R3 slot order per (group, expert): all 1st choices in token order, then all 2nd
     choices, and so on (choice-major). The same rule serves dropless mode.
  R4 capacity C = ceil(capacity_factor * k * S_g / E); capacity_factor <= 0: dropless.
     capacity_factor = 1, k = 2 gives the page's 2N/(G*E).
  R5 an assignment is dropped only from the expert that is full; a token whose k
     assignments are all dropped gets zero expert output (residual pass-through).
     Kept gates are not renormalised after drops.
  R6 top-k ranks logits by value, ties to the lower expert index; non-finite logits
     are an error.
  R7 aux = E * sum_e f_e * P_e with f_e = (top-k choices of e, before random routing
     and capacity) / (S_g * k) and P_e the mean full-softmax probability, per group,
     averaged over groups. It is 1 under perfect balance.
  R8 z = mean over tokens of logsumexp(logits)^2 (no coefficient).
  R9 shared experts are dense FFNs added with weight 1 each.
  R10 SwiGLU uses Swish = SiLU (beta = 1): (silu(x W_in^T) * (x W_up^T)) W_out^T.
  R11 the layer returns the expert output; with a residual given, y = residual + that.
  R12 the garbled GShard output formula is read as y = sum_i G(x)_i E_i(x) (Lec16).
  R16 group-limited top-k (Lec16 "DeepSeek V3 MoE": 256 experts in 8 groups, 4 groups
      kept): the experts form n_groups contiguous groups of E/n_groups; a group's score
      is its largest logit (the page does not say; the max is monotone in the softmax
      score); each token keeps the topk_groups best groups (ties to the lower group)
      and takes its top-k among their experts. Softmax, logsumexp and the losses still
      run over all E experts.
  R17 gate normalisation (MegaBlocks §2 "权重归一化": optional p-norm of the top-k
      weights; Lec16 "DeepSeek V3 MoE": TopK(Softmax(h W), 8)): "softmax_topk" (the
      default) renormalises the k selected probabilities to sum 1 (the p = 1 norm);
      "none" keeps the k full-softmax probabilities as they are; "pnorm" divides them
      by their p-norm.
  R18 uniform assignment (MegaBlocks §2 benchmark switch): the k expert ids of token t
      become (t*k + j) mod E; the gates stay those of the router's own top-k; random
      routing is not combined with it. Counts and the aux loss follow the new ids.

Parity status: every function below is pinned by tests that do not re-type it
(brute force on tiny inputs, closed forms, invariants, library routines, hand-worked
examples). None is "parity unpinned".
"""

from __future__ import annotations

import math

import numpy as np

KEPT, DROP_CAPACITY, DROP_RANDOM = 0, 1, 2


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------------------------------
# capacity  -- [GShard] "Expert capacity", "Local group dispatching"
# ---------------------------------------------------------------------------------------
def capacity(S: int, G: int, E: int, k: int, capacity_factor: float):
    """Per-(group, expert) capacity, or None in dropless mode (reading R4).

    GShard gives each expert a fractional capacity of 2N/(G*E) tokens in each of the G
    groups (N tokens, top-2). With a capacity factor cf and top-k this is
    ceil(cf * k * (S/G) / E).
    """
    if S % G != 0:
        raise ValueError("S must be a multiple of G")
    if capacity_factor <= 0:
        return None
    return int(math.ceil(float(capacity_factor) * k * (S // G) / E))


# ---------------------------------------------------------------------------------------
# router  -- [MegaBlocks] §2 (bias-free linear), [Lec16] "Switch Transformer"
# ---------------------------------------------------------------------------------------
def router_logits(x, W_g, bias=None) -> np.ndarray:
    """logits[t, e] = sum_m x[t, m] * W_g[e, m]  (a linear layer without bias).

    ``bias`` is an optional per-expert offset that the skewed-load workload adds to the
    logits; the pages' router itself has none.
    """
    logits = _f64(x) @ _f64(W_g).T
    if bias is not None:
        logits = logits + _f64(bias)[None, :]
    return logits


def log_softmax_parts(logits):
    """Return (softmax probabilities, logsumexp) over the expert axis, fp64."""
    l = _f64(logits)
    m = l.max(axis=1, keepdims=True)
    z = np.exp(l - m)
    s = z.sum(axis=1, keepdims=True)
    return z / s, (m + np.log(s))[:, 0]


# ---------------------------------------------------------------------------------------
# top-k and gates  -- [Lec16] "Switch Transformer": G(x) = Softmax(KeepTopK(x W_g, k))
# ---------------------------------------------------------------------------------------
def top_k(logits, k: int) -> np.ndarray:
    """Expert ids of the k largest logits per token, largest first; equal logits rank
    the lower expert index first (reading R6). A stable sort of the negated logits."""
    l = _f64(logits)
    if not np.all(np.isfinite(l)):
        raise ValueError("non-finite router logits")
    return np.argsort(-l, axis=1, kind="stable")[:, :k].astype(np.int64)


def top_k_gates(logits, ids) -> np.ndarray:
    """Softmax over the k selected logits: KeepTopK sets the others to -inf before the
    softmax, so gate_j = exp(l_j - l_1) / sum_i exp(l_i - l_1) over the selected i."""
    sel = np.take_along_axis(_f64(logits), ids, axis=1)
    z = np.exp(sel - sel[:, :1])
    return z / z.sum(axis=1, keepdims=True)


def group_limited_top_k(logits, k: int, n_groups: int, topk_groups: int) -> np.ndarray:
    """[Lec16] "DeepSeek V3 MoE" group-limited routing (reading R16): keep each token's
    topk_groups groups of largest best logit (stable: lower group first on ties), then
    the k largest logits among the experts of those groups (reading R6 order)."""
    l = _f64(logits)
    if not np.all(np.isfinite(l)):
        raise ValueError("non-finite router logits")
    S, E = l.shape
    if E % n_groups or k > topk_groups * (E // n_groups):
        raise ValueError("groups must divide E and hold at least k experts")
    size = E // n_groups
    best = l.reshape(S, n_groups, size).max(axis=2)
    kept_groups = np.argsort(-best, axis=1, kind="stable")[:, :topk_groups]
    allowed = np.zeros((S, n_groups), dtype=bool)
    np.put_along_axis(allowed, kept_groups, True, axis=1)
    masked = np.where(np.repeat(allowed, size, axis=1), l, -np.inf)
    return np.argsort(-masked, axis=1, kind="stable")[:, :k].astype(np.int64)


def normalised_gates(logits, ids, norm: str = "softmax_topk", p: float = 1.0) -> np.ndarray:
    """Gates of the selected experts under the three normalisations of reading R17."""
    if norm == "softmax_topk":
        return top_k_gates(logits, ids)
    probs, _ = log_softmax_parts(logits)
    sel = np.take_along_axis(probs, ids, axis=1)
    if norm == "none":
        return sel
    if norm == "pnorm":
        if not p > 0:
            raise ValueError("p must be positive")
        return sel / np.power(np.sum(np.power(sel, p), axis=1, keepdims=True), 1.0 / p)
    raise ValueError(f"unknown gate normalisation {norm!r}")


def uniform_ids(S: int, E: int, k: int) -> np.ndarray:
    """Reading R18: token t's j-th expert is (t*k + j) mod E."""
    return (np.arange(S, dtype=np.int64)[:, None] * k + np.arange(k, dtype=np.int64)[None, :]) % E


# ---------------------------------------------------------------------------------------
# random routing  -- [GShard] "Random routing" (reading R1)
# ---------------------------------------------------------------------------------------
def random_routing_keep(logits, ids, u) -> np.ndarray:
    """Keep the 2nd choice with probability proportional to its gate: u < 2 * g2 with
    g2 = 1 / (1 + exp(l1 - l2)) the renormalised 2nd gate of a top-2 token."""
    l = _f64(logits)
    l1 = np.take_along_axis(l, ids[:, :1], axis=1)[:, 0]
    l2 = np.take_along_axis(l, ids[:, 1:2], axis=1)[:, 0]
    threshold = 2.0 / (1.0 + np.exp(l1 - l2))
    return _f64(u) < threshold


# ---------------------------------------------------------------------------------------
# slots  -- [GShard] "Expert capacity", "Local group dispatching";
#           the dispatch path's "capacity / token position assignment" (readings R2-R5)
# ---------------------------------------------------------------------------------------
def assign_slots(ids, candidate, G: int, E: int, C):
    """Positions of each assignment in its (group, expert) queue.

    Within a group, the 1st choices of all tokens are queued first (token order), then
    the 2nd choices, and so on; a position is the count of earlier candidates for the
    same expert, computed as GShard does, by a cumulative sum of one-hot masks.
    Returns pos [S,k] (-1 when not kept), reason [S,k] (KEPT / DROP_CAPACITY /
    DROP_RANDOM) and counts [G,E] of kept assignments.
    """
    ids = np.asarray(ids, dtype=np.int64)
    candidate = np.asarray(candidate, dtype=bool)
    S, k = ids.shape
    Sg = S // G
    pos = np.full((S, k), -1, dtype=np.int64)
    reason = np.where(candidate, KEPT, DROP_RANDOM).astype(np.uint8)
    counts = np.zeros((G, E), dtype=np.int64)
    rows = np.arange(Sg)
    for g in range(G):
        t0 = g * Sg
        queued = np.zeros(E, dtype=np.int64)  # candidates already queued per expert
        for j in range(k):
            e = ids[t0:t0 + Sg, j]
            c = candidate[t0:t0 + Sg, j]
            onehot = np.zeros((Sg, E), dtype=np.int64)
            onehot[rows, e] = c
            before = np.cumsum(onehot, axis=0) - onehot + queued[None, :]
            slot = before[rows, e]
            queued += onehot.sum(axis=0)
            if C is None:
                keep = c
            else:
                keep = c & (slot < C)
                reason[t0:t0 + Sg, j][c & ~keep] = DROP_CAPACITY
            pos[t0:t0 + Sg, j][keep] = slot[keep]
        counts[g] = queued if C is None else np.minimum(queued, C)
    return pos, reason, counts


def compact_rows(ids, pos, G: int, E: int, counts):
    """Expert-contiguous row of every kept assignment.

    Rows of expert e start at expert_offsets[e] (exclusive scan of per-expert kept
    counts); inside an expert, group g's rows follow those of groups < g, in slot order.
    Returns row [S,k] (-1 when not kept), expert_offsets [E+1] and the inverse map
    token_of [R] plus choice_of [R] (which of the token's k choices the row holds).
    """
    ids = np.asarray(ids, dtype=np.int64)
    S, k = ids.shape
    Sg = S // G
    per_expert = counts.sum(axis=0)
    offsets = np.concatenate([[0], np.cumsum(per_expert)]).astype(np.int64)
    group_base = offsets[None, :E] + (np.cumsum(counts, axis=0) - counts)  # [G,E]
    g_of_t = np.arange(S) // Sg
    kept = pos >= 0
    row = np.full((S, k), -1, dtype=np.int64)
    row[kept] = group_base[np.broadcast_to(g_of_t[:, None], (S, k))[kept], ids[kept]] + pos[kept]
    R = int(offsets[-1])
    token_of = np.full(R, -1, dtype=np.int64)
    choice_of = np.full(R, -1, dtype=np.int64)
    tt, jj = np.nonzero(kept)
    token_of[row[tt, jj]] = tt
    choice_of[row[tt, jj]] = jj
    return row, offsets, token_of, choice_of


# ---------------------------------------------------------------------------------------
# losses  -- [GShard] "Auxiliary loss"; [MegaBlocks] §2 z-loss, §3 load-balancing loss;
#            [Lec16] "MoE 训练中的负载均衡"; [L16/L17] "負載平衡"  (readings R7, R8)
# ---------------------------------------------------------------------------------------
def aux_loss(logits, counts_routed, G: int, k: int) -> float:
    """E * sum_e f_e * P_e per group, averaged over groups.

    f_e = share of the group's S_g * k top-k choices that picked e (counted before
    random routing and capacity); P_e = mean over the group's tokens of the full
    softmax probability of e.
    """
    p, _ = log_softmax_parts(logits)
    S, E = p.shape
    Sg = S // G
    total = 0.0
    for g in range(G):
        P = p[g * Sg:(g + 1) * Sg].mean(axis=0)
        f = np.asarray(counts_routed[g], dtype=np.float64) / (Sg * k)
        total += E * float(np.dot(f, P))
    return total / G


def z_loss(logits) -> float:
    """Mean over tokens of logsumexp over experts, squared."""
    _, lse = log_softmax_parts(logits)
    return float(np.mean(lse * lse))


# ---------------------------------------------------------------------------------------
# routing as one step
# ---------------------------------------------------------------------------------------
def route(logits, cfg: dict, u=None) -> dict:
    """Every routing output of the layer from router logits [S, E].

    The returned dict holds: expert_id, gate (0 where not kept), pos, drop_reason,
    counts [G,E], counts_routed [G,E], row, expert_offsets, token_of, choice_of,
    w_perm (gate of each row), capacity, aux_loss, z_loss.
    """
    S, G, E, k = cfg["S"], cfg["G"], cfg["E"], cfg["k"]
    logits = _f64(logits)
    assert logits.shape == (S, E)
    C = capacity(S, G, E, k, cfg["capacity_factor"])
    ng = int(cfg.get("n_expert_groups", 0) or 0)
    if ng > 1:
        ids = group_limited_top_k(logits, k, ng, int(cfg["topk_groups"]))
    else:
        ids = top_k(logits, k)
    gates = normalised_gates(logits, ids, cfg.get("gate_norm", "softmax_topk"),
                             float(cfg.get("gate_p", 1.0)))
    candidate = np.ones((S, k), dtype=bool)
    if cfg.get("random_routing", 0):
        if k != 2 or u is None or cfg.get("uniform_assignment", 0):
            raise ValueError("random routing needs k == 2, a uniform draw per token and "
                             "no uniform assignment")
        candidate[:, 1] = random_routing_keep(logits, ids, u)
    if cfg.get("uniform_assignment", 0):
        ids = uniform_ids(S, E, k)
    pos, reason, counts = assign_slots(ids, candidate, G, E, C)
    Sg = S // G
    counts_routed = np.zeros((G, E), dtype=np.int64)
    for g in range(G):
        counts_routed[g] = np.bincount(ids[g * Sg:(g + 1) * Sg].ravel(), minlength=E)
    row, offsets, token_of, choice_of = compact_rows(ids, pos, G, E, counts)
    kept = pos >= 0
    gate_out = np.where(kept, gates, 0.0)
    w_perm = np.zeros(len(token_of))
    if len(token_of):
        w_perm = gates[token_of, choice_of]
    return dict(expert_id=ids, gate=gate_out, gate_raw=gates, pos=pos, drop_reason=reason,
                counts=counts, counts_routed=counts_routed, row=row,
                expert_offsets=offsets, token_of=token_of, choice_of=choice_of,
                w_perm=w_perm, capacity=C, aux_loss=aux_loss(logits, counts_routed, G, k),
                z_loss=z_loss(logits))


# ---------------------------------------------------------------------------------------
# experts  -- [GShard] "MoE Transformer" (two-layer FFN per expert);
#             [Lec16] "DeepSeek V3 MoE" (SwiGLU)  (reading R10)
# ---------------------------------------------------------------------------------------
def expert_ffn(x_rows, W_in, W_out, act: str, W_up=None) -> np.ndarray:
    """One expert's FFN on rows [n, M]: W_in, W_up [H, M]; W_out [M, H] (nn.Linear
    [out, in] layout). ReLU: relu(x W_in^T) W_out^T. SwiGLU: (silu(x W_in^T) *
    (x W_up^T)) W_out^T with silu(a) = a / (1 + exp(-a))."""
    xr = _f64(x_rows)
    a = xr @ _f64(W_in).T
    if act == "relu":
        h = np.maximum(a, 0.0)
    elif act == "swiglu":
        with np.errstate(over="ignore"):
            h = a / (1.0 + np.exp(-a)) * (xr @ _f64(W_up).T)
    else:
        raise ValueError(act)
    return h @ _f64(W_out).T


def dispatch(x, token_of) -> np.ndarray:
    """Expert-contiguous copy of the token rows: x_perm[r] = x[token_of[r]]."""
    return np.asarray(x)[np.asarray(token_of, dtype=np.int64)]


def combine(ffn_out, route_out: dict, tokens) -> np.ndarray:
    """y[t] = sum over kept choices j of gate[t, j] * ffn_out[row[t, j]] ([Lec16]
    "Switch Transformer": y = sum_i G(x)_i E_i(x)); a token with nothing kept gets 0
    ([GShard] "Expert capacity": overflow tokens get no expert computation)."""
    tokens = np.asarray(tokens, dtype=np.int64)
    M = ffn_out.shape[1] if ffn_out.ndim == 2 else 0
    y = np.zeros((len(tokens), M))
    row, gate = route_out["row"], route_out["gate"]
    for i, t in enumerate(tokens):
        for j in range(row.shape[1]):
            if row[t, j] >= 0:
                y[i] += gate[t, j] * ffn_out[row[t, j]]
    return y


# ---------------------------------------------------------------------------------------
# the layer  -- [GShard] dispatch path listing; [Lec16] "共享专家 vs. 路由专家" (R9, R11)
# ---------------------------------------------------------------------------------------
def shared_ffn(x_rows, arrays: dict, cfg: dict) -> np.ndarray:
    """Sum of the always-on shared experts' outputs (weight 1 each)."""
    out = np.zeros((len(x_rows), cfg["M"]))
    for s in range(cfg.get("n_shared", 0)):
        W_up = arrays["Ws_up"][s] if cfg["act"] == "swiglu" else None
        out += expert_ffn(x_rows, arrays["Ws_in"][s], arrays["Ws_out"][s], cfg["act"], W_up)
    return out


def layer_forward(arrays: dict, cfg: dict, logits=None, tokens=None, residual=None):
    """The MoE layer output for ``tokens`` (default: all).

    ``arrays`` holds x, W_g, W_in, (W_up), W_out, (Ws_in, Ws_up, Ws_out), u, (bias).
    With ``logits`` given, routing starts from those values instead of the oracle's own
    router projection (so both sides take identical routing decisions).
    Returns (y [len(tokens), M], route dict, logits used).
    """
    x = arrays["x"]
    S = cfg["S"]
    if logits is None:
        logits = router_logits(x, arrays["W_g"], arrays.get("bias"))
    r = route(logits, cfg, arrays.get("u"))
    tokens = np.arange(S) if tokens is None else np.asarray(tokens, dtype=np.int64)
    y = np.zeros((len(tokens), cfg["M"]))
    ids, gate, pos = r["expert_id"], r["gate"], r["pos"]
    for e in range(cfg["E"]):
        sel_i, sel_j = np.nonzero((ids[tokens] == e) & (pos[tokens] >= 0))
        if len(sel_i) == 0:
            continue
        W_up = arrays["W_up"][e] if cfg["act"] == "swiglu" else None
        out = expert_ffn(_f64(x[tokens[sel_i]]), arrays["W_in"][e], arrays["W_out"][e],
                         cfg["act"], W_up)
        np.add.at(y, sel_i, gate[tokens[sel_i], sel_j][:, None] * out)
    if cfg.get("n_shared", 0) > 0:
        y += shared_ffn(_f64(x[tokens]), arrays, cfg)
    if residual is not None:
        y += _f64(residual)[tokens]
    return y, r, logits
