"""Seeded synthetic inputs for the MoE layer forward, shared by the tests and the benchmark.

This module only *draws numbers*: it holds no part of the layer's arithmetic (no routing,
no capacity, no FFN). Both the CUDA path and the CPU oracle receive exactly the values
produced here.

Workload recipe (one preset per workload shape, numbered 1..5):

* x ~ N(0, 1); every weight ~ N(0, 1/fan_in) with fan_in = M for the router, gate and up
  projections and fan_in = H (H_shared for shared experts) for the down projection.
* Draw order is fixed: x, W_g, W_in, W_up, W_out, Ws_in, Ws_up, Ws_out, u, bias; a
  tensor the preset does not use is skipped.
* Every tensor is drawn from its own child of ``SeedSequence(seed)`` (seed defaults to
  1000 + preset number), in blocks of 2**22 elements, each block from its own grandchild
  generator (PCG64). The values therefore do not depend on the thread count.
* Values are drawn in fp32. For bf16 presets each tensor is rounded to bf16
  (round-to-nearest-even); the fp32 arrays handed to the oracle hold exactly those
  rounded values.
* u ~ U[0, 1) per token, the uniform draw for random second-expert dispatch.
* The skewed-overflow preset adds a per-expert router bias b_e = -lam * s * ln(r_e) with
  s = 1.2, lam = 0.33 and r_e in 1..E the rank of expert e under a seeded permutation.
  It stands in for a router that prefers a few experts (a Zipf-like popularity), so that
  a sizeable share of assignments overflows capacity.

The pages' own workloads (a translation corpus, trained weights) are not available; these
shapes stand in for them with random values.
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

# Workload presets. capacity_factor <= 0 means dropless.
PRESETS = {
    1: dict(name="tiny_gshard_top2_fp32", S=256, G=1, E=8, M=64, H=128, k=2,
            capacity_factor=1.0, random_routing=1, n_shared=0, H_shared=0,
            act="relu", dtype="f32", bias=False),
    2: dict(name="gshard_grouped_top2", S=16384, G=16, E=128, M=1024, H=4096, k=2,
            capacity_factor=1.0, random_routing=1, n_shared=0, H_shared=0,
            act="relu", dtype="bf16", bias=False),
    3: dict(name="megablocks_dropless_top2_swiglu", S=8192, G=1, E=8, M=4096, H=14336, k=2,
            capacity_factor=0.0, random_routing=0, n_shared=0, H_shared=0,
            act="swiglu", dtype="bf16", bias=False),
    4: dict(name="shared_plus_finegrained_top6", S=16384, G=1, E=64, M=2048, H=1408, k=6,
            capacity_factor=0.0, random_routing=0, n_shared=2, H_shared=1408,
            act="swiglu", dtype="bf16", bias=False),
    5: dict(name="skewed_overflow_top2", S=65536, G=1, E=64, M=1024, H=4096, k=2,
            capacity_factor=1.25, random_routing=0, n_shared=0, H_shared=0,
            act="relu", dtype="bf16", bias=True),
}

_BLOCK = 1 << 22
_BIAS_S = 1.2
_BIAS_LAMBDA = 0.33


def preset(n: int, **overrides) -> dict:
    """Return a copy of preset ``n`` with fields overridden (e.g. a smaller S)."""
    cfg = dict(PRESETS[n])
    cfg.update(overrides)
    return cfg


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _fill_normal(seq: np.random.SeedSequence, shape, scale: float) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    nb = (n + _BLOCK - 1) // _BLOCK
    kids = seq.spawn(nb)

    def work(i):
        g = np.random.Generator(np.random.PCG64(kids[i]))
        blk = out[i * _BLOCK:(i + 1) * _BLOCK]
        g.standard_normal(out=blk, dtype=np.float32)
        if scale != 1.0:
            blk *= np.float32(scale)

    if nb == 1:
        work(0)
    else:
        with ThreadPoolExecutor(min(nb, _threads())) as ex:
            list(ex.map(work, range(nb)))
    return out.reshape(shape)


def _round_bf16(a: np.ndarray):
    """Round an fp32 array to bf16 (RNE). Returns (bf16 torch tensor, fp32 numpy view of it)."""
    import torch
    t = torch.from_numpy(a).to(torch.bfloat16)
    return t, t.float().numpy()


@dataclass
class Inputs:
    """One workload's tensors. ``np`` holds fp32 arrays (bf16-rounded for bf16 presets);
    ``host`` holds the tensors in the path's storage dtype (torch, CPU)."""
    cfg: dict
    seed: int
    np: dict = field(default_factory=dict)
    host: dict = field(default_factory=dict)


def make_inputs(cfg: dict, seed: int | None = None, preset_number: int | None = None,
                names=None) -> Inputs:
    """Draw the tensors of a workload. ``seed`` defaults to 1000 + ``preset_number``.
    ``names`` restricts which tensors are drawn; the others keep their values (every
    tensor has its own child seed)."""
    import torch
    if seed is None:
        seed = 1000 + (preset_number or 0)
    S, E, M, H = cfg["S"], cfg["E"], cfg["M"], cfg["H"]
    ns, Hs = cfg.get("n_shared", 0), cfg.get("H_shared", 0)
    swiglu = cfg["act"] == "swiglu"
    plan = [
        ("x", (S, M), 1.0),
        ("W_g", (E, M), M ** -0.5),
        ("W_in", (E, H, M), M ** -0.5),
    ]
    if swiglu:
        plan.append(("W_up", (E, H, M), M ** -0.5))
    plan.append(("W_out", (E, M, H), H ** -0.5))
    if ns > 0:
        plan.append(("Ws_in", (ns, Hs, M), M ** -0.5))
        if swiglu:
            plan.append(("Ws_up", (ns, Hs, M), M ** -0.5))
        plan.append(("Ws_out", (ns, M, Hs), Hs ** -0.5))
    kids = np.random.SeedSequence(seed).spawn(len(plan) + 2)
    out = Inputs(cfg=cfg, seed=seed)
    for (name, shape, scale), kid in zip(plan, kids):
        if names is not None and name not in names:
            continue
        a = _fill_normal(kid, shape, scale)
        if cfg["dtype"] == "bf16":
            t, a = _round_bf16(a)
        else:
            t = torch.from_numpy(a)
        out.np[name] = a
        out.host[name] = t
    # uniform draws for random second-expert dispatch
    g_u = np.random.Generator(np.random.PCG64(kids[len(plan)]))
    u = g_u.random(S, dtype=np.float32)
    out.np["u"] = u
    out.host["u"] = torch.from_numpy(u)
    if cfg.get("bias", False):
        g_b = np.random.Generator(np.random.PCG64(kids[len(plan) + 1]))
        rank = g_b.permutation(E).astype(np.float64) + 1.0
        b = (-_BIAS_LAMBDA * _BIAS_S * np.log(rank)).astype(np.float32)
        out.np["bias"] = b
        out.host["bias"] = torch.from_numpy(b)
    return out
