"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and compare it
with the oracle.

Tolerances (element passes iff |gpu - ref| <= rtol * (|ref| + rms(ref row))):
  * layer outputs and expert GEMM outputs: 2e-2 for bf16 storage, 1e-5 for fp32;
  * router logits (fp32 accumulation of exact bf16 products over M terms): 1e-4 bf16 path,
    1e-5 fp32 path;
  * gates (fp32 exp and division, a few ulp): relative 2e-6;
  * aux / z losses (fp32 partial sums over <= 65536 tokens, fixed order): relative 2e-5.
Integer routing outputs are compared bit for bit.
"""

from __future__ import annotations

import numpy as np
import torch

from oracle import moe_oracle as O
from top_gating_expert_gb300 import _native as N
from top_gating_expert_gb300 import moe

RTOL = {"bf16": 2e-2, "f32": 1e-5}
LOGIT_RTOL = {"bf16": 1e-4, "f32": 1e-5}
GATE_RTOL = 2e-6
LOSS_RTOL = 2e-5


def tol_check(gpu, ref, rtol):
    """Returns (number of failing elements, max relative error where |ref| >= rms(row))."""
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    if r.size == 0:
        return 0, 0.0
    r2 = r.reshape(-1, r.shape[-1]) if r.ndim > 1 else r.reshape(1, -1)
    g2 = g.reshape(r2.shape)
    rms = np.sqrt(np.mean(r2 * r2, axis=1, keepdims=True))
    err = np.abs(g2 - r2)
    bad = int(np.count_nonzero(err > rtol * (np.abs(r2) + rms)))
    big = (np.abs(r2) >= rms) & (np.abs(r2) > 0)
    maxrel = float((err[big] / np.abs(r2[big])).max()) if big.any() else 0.0
    return bad, maxrel


def assert_close(gpu, ref, rtol, what=""):
    bad, maxrel = tol_check(gpu, ref, rtol)
    assert bad == 0, f"{what}: {bad} elements outside tolerance {rtol} (max rel err {maxrel:.3e})"
    return maxrel


def to_np(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


def oracle_cfg(cfg: dict) -> dict:
    """The oracle sees the capacity factor the C ABI sees (a float32)."""
    c = dict(cfg)
    c["capacity_factor"] = float(np.float32(cfg.get("capacity_factor", 0.0)))
    return c


def gpu_route(cfg, logits: np.ndarray, u: np.ndarray | None):
    dev = "cuda"
    lg = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).to(dev)
    uu = None if u is None else torch.from_numpy(np.ascontiguousarray(u, dtype=np.float32)).to(dev)
    out = moe.RouteOutputs.allocate(cfg, dev)
    ws = moe.workspace(cfg, N.MOE_WS_STEP, dev)
    moe.route(cfg, lg, uu, out, ws)
    status = moe.device_status(ws)
    return out, status


def route_np(out: moe.RouteOutputs) -> dict:
    return {f: to_np(getattr(out, f)) for f in N.ROUTE_FIELDS}


def gate_rtol(cfg: dict, logits=None) -> float:
    """Relative gate tolerance. Softmax over the k selected logits: 2e-6. The full-softmax
    probabilities (gate_norm "none") also carry the fp32 sum over E terms: each term within
    2 ulp, the sum within (E - 1) * 2^-24, the reciprocal and product within 1 ulp, and the
    argument l - m within |l - m| * 2^-24: (E + 16 + max|l - m|) * 2^-24. The p-norm adds
    powf over k terms: (8k + 32 + max|d|) * 2^-24 with d = l_j - l_1."""
    norm = cfg.get("gate_norm", "softmax_topk")
    spread = 0.0
    if logits is not None and norm != "softmax_topk":
        lg = np.asarray(logits, np.float64)
        lg = np.where(np.isfinite(lg), lg, 0.0)
        spread = float((lg.max(axis=1) - lg.min(axis=1)).max())
    if norm == "none":
        return max(GATE_RTOL, (cfg["E"] + 16 + spread) * 2.0 ** -24)
    if norm == "pnorm":
        return max(GATE_RTOL, (8 * cfg["k"] + 32 + spread) * 2.0 ** -24)
    return GATE_RTOL


def compare_route(g: dict, o: dict, what="", grtol: float = GATE_RTOL):
    """Bit-exact integer outputs; gates and losses within their tolerances."""
    for key in ("expert_id", "pos", "drop_reason", "row", "counts", "counts_routed",
                "expert_offsets"):
        a, b = np.asarray(g[key]).astype(np.int64), np.asarray(o[key]).astype(np.int64)
        if not np.array_equal(a, b):
            idx = np.argwhere(a != b)[:5]
            raise AssertionError(f"{what} {key} differs at {idx.tolist()}: gpu {a[tuple(idx.T)]} "
                                 f"oracle {b[tuple(idx.T)]}")
    R = int(o["expert_offsets"][-1])
    np.testing.assert_array_equal(g["token_of"][:R], o["token_of"], err_msg=f"{what} token_of")
    np.testing.assert_allclose(g["gate"], o["gate"], rtol=grtol, atol=1e-30, err_msg=f"{what} gate")
    np.testing.assert_allclose(g["w_perm"][:R], o["w_perm"], rtol=grtol, atol=1e-30,
                               err_msg=f"{what} w_perm")
    assert abs(float(g["aux_loss"][0]) - o["aux_loss"]) <= LOSS_RTOL * abs(o["aux_loss"]), \
        (what, float(g["aux_loss"][0]), o["aux_loss"])
    assert abs(float(g["z_loss"][0]) - o["z_loss"]) <= LOSS_RTOL * abs(o["z_loss"]) + 1e-7, \
        (what, float(g["z_loss"][0]), o["z_loss"])


def device_inputs(inp, cfg, dev="cuda") -> dict:
    return {k: v.to(dev) for k, v in inp.host.items()}


def near_tie_tokens(logits: np.ndarray, k: int, gap: float = 1e-6) -> np.ndarray:
    """Tokens whose top-(k+1) logits have a consecutive gap below `gap`."""
    s = -np.sort(-np.asarray(logits, np.float64), axis=1)[:, : k + 1]
    return np.nonzero((np.diff(-s, axis=1) < gap).any(axis=1))[0]


def relu_band(x_rows, W_in):
    """(row, unit) pairs whose fp64 pre-activation lies within the fp32-accumulation bound
    of zero, and that bound (module docstring)."""
    xr, W = np.asarray(x_rows, np.float64), np.asarray(W_in, np.float64)
    K = xr.shape[1]
    a = xr @ W.T
    bound = 2.0 * K * 2.0 ** -24 * (np.abs(xr) @ np.abs(W).T)
    return np.abs(a) <= bound, bound


def check_close(gpu, ref, rtol, dev, what):
    """R14 (|g - r| <= rtol (|r| + rms(r row))) plus the widening `dev` (0 where no ambiguous
    mask decision reaches the element). Returns how many elements the widening touched."""
    g = np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    r2 = r.reshape(-1, r.shape[-1])
    g2 = g.reshape(r2.shape)
    d2 = np.broadcast_to(np.asarray(dev, np.float64), r.shape).reshape(r2.shape)
    rms = np.sqrt(np.mean(r2 * r2, axis=1, keepdims=True))
    err = np.abs(g2 - r2)
    lim = rtol * (np.abs(r2) + rms)
    bad = err > lim + d2
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements outside tolerance "
                           f"(first at {np.argwhere(bad)[0].tolist()}, err "
                           f"{err[bad][0]:.3e}, limit {lim[bad][0]:.3e} + {d2[bad][0]:.3e})")
    return int(np.count_nonzero(d2 > 0))
