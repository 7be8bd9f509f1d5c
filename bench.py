#!/usr/bin/env python
"""Benchmark of the MoE layer forward on GB300: tokens/s plus per-kernel roofline figures.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config 3]
                  [--presets 1,2,4,5|none]

One step = one pass of the whole forward (router projection, routing, dispatch, expert
GEMM 1 + activation, expert GEMM 2 + gate, shared experts when present, combine) over one
batch of the workload, inputs resident in HBM. The headline workload (--config, default 3)
is the largest of the five presets by work: the MegaBlocks-style dropless top-2 SwiGLU
layer (8192 tokens, 8 experts, d_model 4096, d_ff 14336; 5.8 TFLOP of expert GEMMs a step).
The other presets are measured the same way into the line's "presets" object. L2 is
flushed before every timed step, outside the step's events: a 256 MiB write, then a
256 MiB read that writes the dirty lines back. N > 1 (torchrun): every rank runs an
independent replica on its own GPU (the forward has no exchange step on one GPU),
value = tokens of all ranks divided by the slowest rank's time.

--impl reference times the CPU oracle (plain numpy fp64, as it stands) on the host cores,
each step one bounded sample of the same workload; under torchrun only rank 0 runs it.
"""

from __future__ import annotations

import argparse
import faulthandler
import hashlib
import json
import os
import platform
import signal
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer fwd tokens/s"
UNIT = "tokens/s"
FLUSH_BYTES = 256 << 20
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.md")
HEADLINE = 3  # the largest preset by work
# steps in flight in the host-to-host leg: with two, a 134 MB input copy, the layer and the
# 134 MB output copy of one buffer set (≈ 0.65 + 1.1 + 0.7 ms at the ≈ 200 GB/s a pinned copy
# reaches over the host link, preset 5) bound a step at half their sum; three measured 11 %
# faster there (50.3 -> 55.7 M tokens/s), four no faster
E2E_DEPTH = 3
L2_POLICY = ("GPU: L2 flushed before every timed step, outside its events (256 MiB write, "
             "then 256 MiB read, so dirty lines are written back outside the step); "
             "host-to-host e2e: not flushed, inputs arrive from host memory")
# fp64 flops of the oracle per bench run: the headline's CPU baseline (10-30 s of host
# work), the other presets' (a few seconds each) and one reference-arm step
CPU_FLOPS_HEADLINE = 6.0e12
CPU_FLOPS_PRESET = 1.2e12
CPU_FLOPS_REFERENCE_STEP = 0.8e12


_T0 = time.perf_counter()


def log(msg: str):
    """A progress line on stderr (the JSON line alone goes to stdout)."""
    print(f"[bench {time.perf_counter() - _T0:7.1f} s] {msg}", file=sys.stderr, flush=True)


def parse(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", type=int, default=HEADLINE, help="headline workload preset (1..5)")
    p.add_argument("--presets", default="all",
                   help="other presets measured into the 'presets' object: a comma list, "
                        "'all' (every preset but the headline) or 'none'")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-backward", action="store_true",
                   help="skip the training-step (forward + backward) measurement")
    p.add_argument("--no-variants", action="store_true",
                   help="skip the routing-variant measurement")
    p.add_argument("--variants-preset", type=int, default=2,
                   help="the preset whose tokens the routing variants route")
    p.add_argument("--override", action="append", default=[], metavar="KEY=VALUE",
                   help="change a field of the headline preset (smaller cases for profiler "
                        "captures)")
    return p.parse_args(argv)


def preset_for(args, n=None) -> dict:
    """Preset n (default: the headline), with --override applied to the headline only."""
    from top_gating_expert_gb300.inputs import PRESETS
    n = args.config if n is None else n
    cfg = dict(PRESETS[n])
    if n != args.config:
        return cfg
    for kv in args.override:
        key, val = kv.split("=", 1)
        if key not in cfg:
            raise SystemExit(f"unknown preset field {key}")
        cfg[key] = type(cfg[key])(float(val)) if not isinstance(cfg[key], str) else val
    if args.override:
        cfg["name"] += " (" + ", ".join(args.override) + ")"
    return cfg


def other_presets(args) -> list:
    if args.presets == "none":
        return []
    if args.presets == "all":
        return [n for n in (1, 2, 3, 4, 5) if n != args.config]
    return [int(v) for v in args.presets.split(",") if v.strip() and int(v) != args.config]


def workload_desc(cfg: dict, n: int) -> dict:
    d = {"workload": f"preset {n} {cfg['name']}: S={cfg['S']} tokens, G={cfg['G']} groups, "
                     f"E={cfg['E']} experts, k={cfg['k']}, M={cfg['M']}, H={cfg['H']}, "
                     f"{cfg['act']}, {cfg['dtype']}"}
    if cfg["capacity_factor"] > 0:
        d["workload"] += f", capacity factor {cfg['capacity_factor']}"
    else:
        d["workload"] += ", dropless"
    if cfg["random_routing"]:
        d["workload"] += ", random 2nd-expert dispatch"
    if cfg["n_shared"]:
        d["workload"] += f", {cfg['n_shared']} shared experts H={cfg['H_shared']}"
    if cfg.get("bias"):
        d["workload"] += ", skewed router bias"
    if residual_for(n):
        d["workload"] += ", residual added"
    d.update(S=cfg["S"], G=cfg["G"], E=cfg["E"], k=cfg["k"], M=cfg["M"], H=cfg["H"])
    return d


def workload_config(cfg: dict, n: int) -> dict:
    """The line's `config`: the same dict in both arms (the workload, and the L2 policy)."""
    return dict(workload_desc(cfg, n), l2=L2_POLICY)


def residual_for(n: int) -> bool:
    """The overflow workload adds its input: dropped tokens pass through the residual."""
    return n == 5


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return dict(hbm=float(j["hbm_gbs"]), tc=float(j["bf16_tflops"]),
                    tc_sustained=float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm=6800.0, tc=1900.0, tc_sustained=1700.0, source="fallback")


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


def host_cores() -> int:
    return len(os.sched_getaffinity(0))


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        for r in rows:
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                "sw_power_cap"), r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "samples": len(rows),
                "reasons": sorted(reasons)}


def traffic_for(kernel: str, config: int):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, or None when the
    kernel source changed since the capture."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            lines = f.read().splitlines()
    except OSError:
        return None
    for line in lines:
        if line.startswith("|") and f"| {kernel} |" in line and f"| {config} |" in line:
            cells = [c.strip() for c in line.strip("|").split("|")]
            # | kernel | config | dram bytes per launch | source sha1 | files |
            try:
                sha = cells[3]
                h = hashlib.sha1()
                for name in cells[4].split("+"):  # the kernel's source files, in order
                    with open(os.path.join(ROOT, "top_gating_expert_gb300", "csrc", name.strip()), "rb") as f:
                        h.update(f.read())
                if h.hexdigest()[:12] != sha:
                    return None
                return float(cells[2])
            except Exception:
                return None
    return None


# ------------------------------------------------------------------ aggregation over ranks
def max_over_ranks(values, world: int, device=None) -> list:
    """Each rank's timings (ms); returns the maximum over the ranks of each: with one replica
    per GPU and a barrier on both sides of every timed region, the slowest replica bounds
    the whole job."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(units_per_rank_step: int, steps: int, world: int, total_ms: float) -> float:
    """Whole-job units/s: every replica processes its own units each step (weak scaling)."""
    return units_per_rank_step * steps * world / (total_ms * 1e-3)


# ------------------------------------------------------------------ roofline arithmetic
STEP_NAMES_FUSED = ["router_route", "dispatch", "expert_up", "expert_down"]
LAUNCHES = {"router_route": 3, "router": 1, "route": 3, "dispatch": 1, "expert_up": 1,
            "expert_down": 1, "shared_ffn": 2, "combine": 1}


def algorithmic(cfg: dict, R: int, used: int, has_bias: bool, has_u: bool, residual: bool) -> dict:
    """(bytes, flops) per launch of each step, algorithmic: every input read once and every
    output written once; flops of the contractions only."""
    eb = 2 if cfg["dtype"] == "bf16" else 4
    S, E, M, H, k = cfg["S"], cfg["E"], cfg["M"], cfg["H"], cfg["k"]
    f1 = 2 if cfg["act"] == "swiglu" else 1
    per_assign = S * k * (4 + 4 + 4 + 1 + 4)  # id, gate, pos, row (int32/fp32), drop (u8)
    algo = {
        "router": (S * M * eb + E * M * eb + S * E * 4 + (E * 4 if has_bias else 0),
                   2.0 * S * M * E),
        "route": (S * E * 4 + (S * 4 if has_u else 0) + per_assign + R * 8, 0.0),
        # x and W_g in; u in; per assignment outputs; the inverse map and gate per kept row
        # (the logits never leave the chip)
        "router_route": (S * M * eb + E * M * eb + (E * 4 if has_bias else 0)
                         + (S * 4 if has_u else 0) + per_assign + R * 8, 2.0 * S * M * E),
        "dispatch": (2 * R * M * eb + R * 4, 0.0),
        "expert_up": (used * f1 * H * M * eb + R * M * eb + R * H * eb, 2.0 * f1 * R * M * H),
        "expert_down": (used * M * H * eb + R * H * eb + R * M * eb + R * 4, 2.0 * R * M * H),
        "combine": (R * M * eb + S * M * eb + S * k * 4 + (S * M * eb if residual else 0)
                    + (S * M * eb if cfg.get("n_shared") else 0), 0.0),
    }
    if cfg.get("n_shared"):
        Hc = cfg["n_shared"] * cfg["H_shared"]
        algo["shared_ffn"] = ((f1 + 1) * Hc * M * eb + 2 * S * M * eb + 2 * S * Hc * eb,
                              2.0 * (f1 + 1) * S * M * Hc)
    return algo


def kernel_table(names, per_kernel: dict, algo: dict, P: dict) -> list:
    out = []
    for nm in names:
        ms = per_kernel[nm]
        b, fl = algo[nm]
        gbs = b / (ms * 1e-3) / 1e9
        ent = {"name": nm, "ms": round(ms, 5), "launches": LAUNCHES[nm], "bytes": int(b),
               "GB/s": round(gbs, 1), "hbm_frac": round(gbs / P["hbm"], 4)}
        if fl:
            tf = fl / (ms * 1e-3) / 1e12
            ent.update({"flops": fl, "TFLOP/s": round(tf, 2),
                        "tensor_frac_sustained": round(tf / P["tc_sustained"], 4),
                        "tensor_frac_burst": round(tf / P["tc"], 4)})
        out.append(ent)
    return out


def roofline_of(kernel: str, ms: float, algo: dict, P: dict, n: int) -> dict:
    """The roofline object of one kernel: the binding bound is the larger of its byte time
    (measured HBM copy rate) and flop time (sustained bf16 rate)."""
    b, fl = algo[kernel]
    byte_t, flop_t = b / (P["hbm"] * 1e9), fl / (P["tc_sustained"] * 1e12)
    if byte_t >= flop_t:
        achieved = b / (ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": P["hbm"], "unit": "GB/s",
                "frac": round(achieved / P["hbm"], 4)}
    else:
        achieved = fl / (ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": P["tc_sustained"],
                "unit": "TFLOP/s", "frac": round(achieved / P["tc_sustained"], 4),
                "frac_of_burst_peak": round(achieved / P["tc"], 4)}
    roof.update({"kernel": kernel, "ms": round(ms, 5),
                 "peak_source": P["source"] + (" (sustained bf16)" if roof["bound"] == "tensor"
                                               else " (copy)"),
                 "traffic": traffic_for(kernel, n), "algorithmic_bytes": int(b),
                 "algorithmic_flops": fl})
    return roof


def backward_summary(cfg, R, S, world, f_ms, b_ms, P) -> dict:
    M, H, E = cfg["M"], cfg["H"], cfg["E"]
    f1 = 2 if cfg["act"] == "swiglu" else 1
    F = f1 * H
    Hc = cfg.get("n_shared", 0) * cfg.get("H_shared", 0)

    # algorithmic flops: GEMM 2's and GEMM 1's data and weight gradients (and the SwiGLU
    # pre-activations recomputed) for the routed rows and the shared experts' S rows; the
    # router's dx and dW_g
    def ffn_bwd(rows, hidden):
        fh = f1 * hidden
        return 2.0 * rows * M * (2 * hidden + 2 * fh) + (4.0 * rows * M * hidden if f1 == 2 else 0.0)
    flops = ffn_bwd(R, H) + (ffn_bwd(S, Hc) if Hc else 0.0) + 4.0 * S * E * M
    grad_bytes = 4 * (E * (F + H) * M + ((f1 + 1) * Hc * M if Hc else 0) + E * M)
    # algorithmic bytes: every input read once (dy, x, the logits, W_g, the transposed weight
    # packs, the packed W_in again for the SwiGLU recompute, the stored h) and every output
    # written once (the fp32 weight gradients, dx)
    b2 = 2 if cfg["dtype"] == "bf16" else 4
    in_bytes = (b2 * (2 * S * M + E * M + E * (F + H) * M + (E * F * M if f1 == 2 else 0)
                      + R * H) + 4 * S * E)
    if Hc:
        in_bytes += b2 * ((f1 + 1) * Hc * M + (f1 * Hc * M if f1 == 2 else 0) + S * Hc)
    bwd_bytes = in_bytes + grad_bytes + b2 * S * M
    t_bytes = bwd_bytes / (P["hbm"] * 1e9) * 1e3
    t_flops = flops / (P["tc_sustained"] * 1e12) * 1e3
    if cfg["dtype"] != "bf16":  # the fp32 path: plain FMA on a tiny layer, no roofline
        return {
            "what": "moe_layer_backward (fp32, plain FMA): gradients of sum(dy*y) + 0.01 aux + "
                    "0.001 z w.r.t. x, W_g, every expert weight; forward = moe_layer_forward "
                    "keeping its logits; L2 flushed before each step",
            "ms_per_step": round(b_ms, 5), "forward_ms_per_step": round(f_ms, 5),
            "train_tokens_per_s": round(S * world / ((f_ms + b_ms) * 1e-3), 1),
            "algorithmic_flops": flops, "algorithmic_bytes": int(bwd_bytes),
            "bound": "latency", "roofline_frac": None,
        }
    return {
        "what": "moe_layer_backward: gradients of sum(dy*y) + 0.01 aux + 0.001 z w.r.t. x, "
                "W_g, every expert weight (fp32), routing fixed; forward = moe_layer_forward "
                "keeping its logits; L2 flushed before each step",
        "ms_per_step": round(b_ms, 5), "forward_ms_per_step": round(f_ms, 5),
        "train_tokens_per_s": round(S * world / ((f_ms + b_ms) * 1e-3), 1),
        "algorithmic_flops": flops, "TFLOP/s": round(flops / (b_ms * 1e-3) / 1e12, 2),
        "tensor_frac_sustained": round(flops / (b_ms * 1e-3) / 1e12 / P["tc_sustained"], 4),
        "fp32_weight_grad_bytes": int(grad_bytes),
        "algorithmic_bytes": int(bwd_bytes),
        "hbm_frac": round(bwd_bytes / (b_ms * 1e-3) / 1e9 / P["hbm"], 4),
        # the binding roofline: the larger of the byte time and the flop time, and the
        # step's fraction of it
        "bound": "hbm" if t_bytes >= t_flops else "tensor",
        "roofline_frac": round(max(t_bytes, t_flops) / b_ms, 4),
    }


# ------------------------------------------------------------------ our arm, one preset
class Flush:
    """Evicts L2 before a timed step: write 256 MiB (the cache then holds only dirty zeros),
    then read another 256 MiB, so those dirty lines are written back here, outside the
    step's events, instead of inside the next step."""

    def __init__(self, dev):
        import torch
        self.buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.read = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def __call__(self):
        import torch
        self.buf.zero_()
        self.read.sum(dtype=torch.int64)


def run_preset(args, n, cfg, rank, world, dev, flush, barrier, *, headline: bool,
               variants: bool):
    """Measures preset n; returns its figures (rank 0) or None."""
    import torch
    from top_gating_expert_gb300 import moe
    from top_gating_expert_gb300.inputs import make_inputs

    log(f"preset {n}: drawing inputs")
    inp = make_inputs(cfg, preset_number=n)
    # the layer's step output is y and the losses: the bf16 path never writes the logits
    layer = moe.MoeLayer(cfg, inp.host, device=dev, keep_logits=False)
    log(f"preset {n}: weights packed")
    c = layer.cfg
    x = inp.host["x"].to(dev)
    u = inp.host["u"].to(dev) if cfg["random_routing"] else None
    bias = layer.bias
    residual = x if residual_for(n) else None
    R_max = moe.rows_max(c)
    dt = moe.torch_dtype(c)
    ws, out = layer.ws, layer.route_out
    fused = cfg["dtype"] == "bf16"
    logits = None if fused else torch.empty((c.S, c.E), dtype=torch.float32, device=dev)
    x_perm = torch.empty((R_max, c.M), dtype=dt, device=dev)
    h_perm = torch.empty((R_max, c.H), dtype=dt, device=dev)
    y_perm = torch.empty((R_max, c.M), dtype=dt, device=dev)
    y = torch.empty((c.S, c.M), dtype=dt, device=dev)
    shared = c.n_shared > 0
    if shared:
        Hc = c.n_shared * c.H_shared
        h_sh = torch.empty((c.S, Hc), dtype=dt, device=dev)
        s_out = torch.empty((c.S, c.M), dtype=dt, device=dev)

    names = (["router_route"] if fused else ["router", "route"]) + \
            ["dispatch", "expert_up", "expert_down"] + (["shared_ffn"] if shared else []) + ["combine"]

    def step(evs=None):
        def mark(i):
            if evs is not None:
                evs[i].record()
        mark(0)
        i = 1
        if fused:
            moe.router_route(c, x, layer.W_g, bias, u, None, out, ws); mark(i)
            i += 1
        else:
            moe.router(c, x, layer.W_g, bias, logits, ws); mark(i)
            moe.route(c, logits, u, out, ws); mark(i + 1)
            i += 2
        moe.dispatch(c, x, out, x_perm); mark(i)
        moe.expert_up(c, x_perm, out.expert_offsets, layer.W_in_packed, h_perm, ws); mark(i + 1)
        moe.expert_down(c, h_perm, out.expert_offsets, out.w_perm, layer.W_out_packed, y_perm, ws)
        mark(i + 2)
        i += 3
        if shared:
            moe.shared_ffn(c, x, layer.Ws_in_packed, layer.Ws_out_packed, h_sh, s_out, ws); mark(i)
            i += 1
        moe.combine(c, y_perm, out, s_out if shared else None, residual, y); mark(i)

    def check(where):
        rc = moe.device_status(ws)
        if rc != 0:
            raise RuntimeError(f"preset {n}: device status {rc} {where}")

    for _ in range(args.warmup):
        flush()
        step()
    check("after warm-up")

    # ---- the whole forward (moe_layer_forward) captured once as a CUDA graph
    log(f"preset {n}: step-wise warm-up done; capturing the forward")
    graph_ok = True
    try:
        layer.capture(x, u, residual)
        for _ in range(args.warmup):
            flush()
            layer.replay()
    except Exception as exc:  # capture unavailable: time the eager call instead
        graph_ok = False
        print(f"preset {n}: graph capture failed ({exc}); timing eager moe_layer_forward",
              file=sys.stderr)
    check("after graph warm-up")
    clocks = ClockSampler(dev.index or 0)
    time.sleep(0.3)
    head_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    barrier()
    t_wall = time.perf_counter()
    for s in range(args.steps):
        flush()
        head_ev[s][0].record()
        if graph_ok:
            layer.replay()
        else:
            layer.forward(x, u, residual)
        head_ev[s][1].record()
    barrier()
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    check("in the timed region")
    total_ms, = max_over_ranks([sum(a.elapsed_time(b) for a, b in head_ev)], world, dev)

    # ---- the same replays back to back without the flush: reported beside, not as, the value
    warm_ms = None
    if graph_ok and headline:
        wev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        barrier()
        for s in range(args.steps):
            wev[s][0].record()
            layer.replay()
            wev[s][1].record()
        barrier()
        warm_ms, = max_over_ranks([sum(a.elapsed_time(b) for a, b in wev)], world, dev)

    # ---- per-kernel times: the same launches through the step-wise calls, an event between
    # consecutive calls (a second timed region of the same K steps)
    log(f"preset {n}: graph timed; per-kernel timing")
    nev = len(names) + 1
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(args.steps)]
    barrier()
    for s in range(args.steps):
        flush()
        step(events[s])
    barrier()
    check("in the per-kernel timed region")
    step_ms = [events[s][0].elapsed_time(events[s][-1]) for s in range(args.steps)]
    pk = [statistics.mean(events[s][i].elapsed_time(events[s][i + 1]) for s in range(args.steps))
          for i in range(len(names))]
    per_kernel = dict(zip(names, max_over_ranks(pk, world, dev)))

    # ---- e2e through the public API: pinned host buffers in and out, every step copying its
    # own inputs to the device and its result back (HostPipeline: E2E_DEPTH steps in flight,
    # so that a buffer set's input copy, layer and output copy together may take up to that
    # many steps' time)
    log(f"preset {n}: host-to-host timing")
    x_host = inp.host["x"].pin_memory()
    u_host = inp.host["u"].pin_memory() if u is not None else None
    y_host = torch.empty((c.S, c.M), dtype=dt).pin_memory()
    loss_host = torch.empty(2, dtype=torch.float32).pin_memory()
    pipe = moe.HostPipeline(layer, has_u=u is not None, residual=residual is not None,
                            depth=E2E_DEPTH)
    for i in range(args.warmup):
        pipe.submit(i, x_host, u_host, y_host, loss_host)
    barrier()
    e2e_start, e2e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_start.record(pipe.h2d)
    for i in range(args.steps):
        pipe.submit(i, x_host, u_host, y_host, loss_host)
    e2e_end.record(pipe.d2h)
    barrier()
    e2e_ms, = max_over_ranks([e2e_start.elapsed_time(e2e_end)], world, dev)
    check("in the e2e region")
    h2d = x_host.numel() * x_host.element_size() + (u_host.numel() * 4 if u_host is not None else 0)
    d2h = y_host.numel() * y_host.element_size() + 8
    del pipe, x_host, u_host, y_host

    # ---- the backward pass (a training step): a layer that keeps its logits, forward then
    # moe_layer_backward on the same inputs, L2 flushed before each step
    bwd = None
    if not args.no_backward:
        log(f"preset {n}: backward")
        del x_perm, h_perm, y_perm
        tl = moe.MoeLayer(cfg, inp.host, device=dev)
        tl.enable_backward(inp.host)
        dy = torch.randn((c.S, c.M), generator=torch.Generator().manual_seed(7)).to(dt).to(dev)

        def train_step(evs=None):
            if evs:
                evs[0].record()
            tl.forward(x, u, residual)
            if evs:
                evs[1].record()
            tl.backward(x, dy, residual=residual is not None, aux_coef=0.01, z_coef=0.001)
            if evs:
                evs[2].record()

        for _ in range(args.warmup):
            flush()
            train_step()
        tev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        barrier()
        for s_ in range(args.steps):
            flush()
            train_step(tev[s_])
        barrier()
        rc = moe.device_status(tl.ws_bwd)
        if rc != 0:
            raise RuntimeError(f"preset {n}: device status {rc} in the backward region")
        f_ms, b_ms = max_over_ranks([statistics.mean(a.elapsed_time(b) for a, b, _ in tev),
                                     statistics.mean(b.elapsed_time(e) for _, b, e in tev)],
                                    world, dev)
        bwd = (f_ms, b_ms, tl.route_out.expert_offsets[-1].item())
        del tl, dy

    var = None
    if variants and fused and not args.no_variants:
        log(f"preset {n}: routing variants")
        var = time_variants(args, cfg, c, x, layer, bias, u, flush, barrier, world, dev,
                            per_kernel["router_route"])
        var["preset"] = n

    offs = out.expert_offsets.cpu().numpy()
    R = int(offs[-1])
    used = int((offs[1:] > offs[:-1]).sum())
    del layer, x, u, residual, y, out, ws
    torch.cuda.empty_cache()
    if rank != 0:
        return None

    P = peaks()
    S, k = c.S, c.k
    algo = algorithmic(cfg, R, used, bias is not None, cfg["random_routing"] != 0,
                       residual_for(n))
    dom = max(("expert_up", "expert_down"), key=lambda nm: per_kernel[nm])
    res = {
        "workload": workload_desc(cfg, n)["workload"],
        "value": round(job_throughput(S, args.steps, world, total_ms), 1),
        "ms_per_step": round(total_ms / args.steps, 5),
        "rows": R, "kept_fraction": round(R / (S * k), 4),
        "roofline": roofline_of(dom, per_kernel[dom], algo, P, n),
        "kernels": kernel_table(names, per_kernel, algo, P),
        "e2e": {"value": round(job_throughput(S, args.steps, world, e2e_ms), 1), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": f"HostPipeline.submit (pinned host in/out, {E2E_DEPTH} steps in flight) -> "
                       "moe_layer_forward (CUDA graph); L2 not flushed: inputs arrive from host"},
        # moe_layer_forward runs the routing's last kernel and the dispatch as one launch
        "launches_per_step": sum(LAUNCHES[nm] for nm in names) - 1,
        "timing": {"headline": "CUDA graph of moe_layer_forward, one replay per step" if graph_ok
                   else "eager moe_layer_forward per step",
                   "ms_per_step_stepwise": round(statistics.mean(step_ms), 5),
                   "kernels": "step-wise ABI calls, a CUDA event between consecutive calls, "
                              "second timed region of the same K steps"},
        "clocks": clk,
        "wall_s_timed_region": round(t_wall, 4),
    }
    if warm_ms is not None:
        res["warm"] = {"ms_per_step": round(warm_ms / args.steps, 5),
                       "value": round(job_throughput(S, args.steps, world, warm_ms), 1),
                       "what": "the same CUDA-graph replays back to back, no L2 flush between steps"}
    if bwd is not None:
        f_ms, b_ms, Rb = bwd
        res["backward"] = backward_summary(cfg, Rb, S, world, f_ms, b_ms, P)
    if var is not None:
        res["variants"] = var
    if world == 1 and not args.no_cpu_baseline:
        log(f"preset {n}: oracle on the host")
        res["cpu_baseline"] = cpu_baseline(cfg, n, inp,
                                           CPU_FLOPS_HEADLINE if headline else CPU_FLOPS_PRESET)
    log(f"preset {n}: done")
    return res


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    flush = Flush(dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    n = args.config
    cfg = preset_for(args)
    head = run_preset(args, n, cfg, rank, world, dev, flush, barrier, headline=True,
                      variants=(args.variants_preset == n))
    others = {}
    for m in other_presets(args):
        others[m] = run_preset(args, m, preset_for(args, m), rank, world, dev, flush, barrier,
                               headline=False, variants=(args.variants_preset == m))
    if rank != 0:
        return None

    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cfg["dtype"],
        "data": "synthetic", "config": workload_config(cfg, n),
        "parallelism": f"replicas x{world}",
        "routing": {"rows": head["rows"], "kept_fraction": head["kept_fraction"]},
        "roofline": head["roofline"],
        "kernels": head["kernels"],
        "e2e": head["e2e"],
        "gpu_launches": args.steps * head["launches_per_step"],
        "timing": head["timing"],
        "clocks": head["clocks"],
        "wall_s_timed_region": head["wall_s_timed_region"],
    }
    for key in ("warm", "backward", "cpu_baseline"):
        if key in head:
            line[key] = head[key]
    var = head.get("variants")
    presets = {}
    for m, r in others.items():
        var = var or r.pop("variants", None)
        presets[str(m)] = r
    if presets:
        line["presets"] = presets
    if var is not None:
        line["variants"] = var
    return line


# ------------------------------------------------------------------ routing variants
# Each entry: the preset's fields it changes. Group-limited routing and the gate
# normalisations: Lec16 "DeepSeek V3 MoE" (8 expert groups, 4 kept, TopK(Softmax) gates),
# MegaBlocks router chapter §2 (p-norm of the top-k weights, the uniform-assignment switch).
VARIANTS = {
    "group_limited_8x4": dict(n_expert_groups=8, topk_groups=4),
    "gates_unnormalised": dict(gate_norm="none"),
    "gates_pnorm2": dict(gate_norm="pnorm", gate_p=2.0),
    "uniform_assignment": dict(uniform_assignment=1, random_routing=0),
    "top4": dict(k=4, random_routing=0),
    # DeepSeek-V3's routing over the preset's tokens: 256 experts in 8 groups, 4 kept, top-8,
    # un-normalised gates, no capacity (a seeded random router of 256 rows)
    "deepseek_v3_routing": dict(E=256, k=8, n_expert_groups=8, topk_groups=4, gate_norm="none",
                                capacity_factor=0.0, random_routing=0, G=1),
}


def variant_router_weights(E: int, M: int):
    """The seeded router of a variant whose expert count differs from the preset's (fp32,
    N(0, 1/M)); callers cast it to the layer's dtype."""
    import torch
    g = torch.Generator().manual_seed(31)
    return torch.randn((E, M), generator=g) / M ** 0.5


def variant_cfg(cfg: dict, kw: dict):
    """The preset with a variant's fields, or None where the variant does not apply."""
    vc = dict(cfg, **kw)
    if vc["S"] % vc["G"] or vc["E"] % vc.get("n_expert_groups", 1) or vc["k"] > vc["E"]:
        return None
    return vc


def time_variants(args, cfg, c, x, layer, bias, u, flush, barrier, world, dev, default_ms):
    """moe_router_route under each routing variant on the preset's tokens (x and, where E is
    unchanged, W_g), L2 flushed before each call, CUDA events around it; bytes as for the
    default routing (x and W_g in, per-assignment outputs, the inverse map)."""
    import torch
    from top_gating_expert_gb300 import moe

    P = peaks()
    res = {"what": "moe_router_route (router GEMM + softmax + variant top-k + slots + rows), "
                   "L2 flushed before each call; default routing for comparison",
           "default_ms": round(default_ms, 5)}
    for name, kw in VARIANTS.items():
        vc = variant_cfg(cfg, kw)
        if vc is None:
            continue
        cv = moe.make_config(vc)
        if moe.validate(cv) != 0:
            res[name] = {"skipped": "configuration not valid for this preset"}
            continue
        if vc["E"] != cfg["E"]:
            W_g = variant_router_weights(vc["E"], vc["M"]).to(x.dtype).to(dev)
            b = None
        else:
            W_g, b = layer.W_g, bias
        uv = u if vc["random_routing"] else None
        outv = moe.RouteOutputs.allocate(cv, dev)
        wsv = moe.workspace(cv, moe.N.MOE_WS_STEP, device=dev)
        for _ in range(max(3, args.warmup)):
            flush()
            moe.router_route(cv, x, W_g, b, uv, None, outv, wsv)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        barrier()
        for s in range(args.steps):
            flush()
            evs[s][0].record()
            moe.router_route(cv, x, W_g, b, uv, None, outv, wsv)
            evs[s][1].record()
        barrier()
        rc = moe.device_status(wsv)
        if rc != 0:
            raise RuntimeError(f"device status {rc} in the {name} variant")
        ms, = max_over_ranks([sum(a.elapsed_time(e) for a, e in evs) / args.steps], world, dev)
        R = int(outv.expert_offsets[-1].item())
        S, E, M, k = vc["S"], vc["E"], vc["M"], vc["k"]
        nb = (S * M * 2 + E * M * 2 + (E * 4 if b is not None else 0) + (S * 4 if uv is not None else 0)
              + S * k * (4 + 4 + 4 + 1 + 4) + R * 8)
        gbs = nb / (ms * 1e-3) / 1e9
        res[name] = {"fields": {kk: vv for kk, vv in kw.items()}, "ms": round(ms, 5),
                     "vs_default": round(ms / default_ms, 3), "rows": R,
                     "kept_fraction": round(R / (S * k), 4), "bytes": int(nb),
                     "GB/s": round(gbs, 1), "hbm_frac": round(gbs / P["hbm"], 4),
                     "TFLOP/s": round(2.0 * S * M * E / (ms * 1e-3) / 1e12, 2)}
        del outv, wsv
    return res


# ------------------------------------------------------------------ the oracle on the host
def _sample_cfg(cfg: dict, tokens: int) -> dict:
    """A bounded sample of the workload: whole groups when grouped, else a token prefix."""
    s = dict(cfg)
    if cfg["G"] > 1:
        g = max(1, tokens // (cfg["S"] // cfg["G"]))
        s["G"] = g
        s["S"] = g * (cfg["S"] // cfg["G"])
    else:
        s["S"] = min(cfg["S"], tokens)
    return s


def sample_tokens(cfg: dict, target_flops: float) -> int:
    """Tokens whose oracle layer forward takes about `target_flops` fp64 flops of expert
    FFNs (at least 256, at most the workload)."""
    f1 = 3 if cfg["act"] == "swiglu" else 2
    per_token = 2.0 * f1 * cfg["M"] * cfg["H"] * cfg["k"] + \
        2.0 * f1 * cfg["M"] * cfg.get("n_shared", 0) * cfg.get("H_shared", 0)
    return int(max(256, min(cfg["S"], target_flops / per_token)))


def oracle_arrays(inp_np: dict, S: int) -> dict:
    """The oracle's inputs upcast to fp64 once, outside any timed region (the oracle's own
    upcast then costs nothing): x and u cut to the sample's first S tokens."""
    import numpy as np
    a = {}
    for key, v in inp_np.items():
        v = v[:S] if key in ("x", "u") else v
        a[key] = np.asarray(v, dtype=np.float64)
    return a


def _oracle_step(sample_cfg, arrays, residual: bool):
    from oracle import moe_oracle as O
    y, _, _ = O.layer_forward(arrays, sample_cfg, residual=arrays["x"] if residual else None)
    return y


def cpu_baseline(cfg, n, inp, target_flops=CPU_FLOPS_PRESET):
    """The oracle on a bounded sample: about `target_flops` of fp64 expert-FFN work."""
    sc = _sample_cfg(cfg, sample_tokens(cfg, target_flops))
    t = time.perf_counter()
    arrays = oracle_arrays(inp.np, sc["S"])
    t_up = time.perf_counter() - t
    t = time.perf_counter()
    _oracle_step(sc, arrays, residual_for(n))
    dt = time.perf_counter() - t
    # the routing stage alone on the same sample (router projection, softmax, top-k, slots,
    # rows, losses); the rest of the step is the experts' FFNs and the combine
    from oracle import moe_oracle as O
    t = time.perf_counter()
    O.route(O.router_logits(arrays["x"], arrays["W_g"], arrays.get("bias")), sc, arrays["u"])
    dt_route = time.perf_counter() - t
    del arrays
    return {"value": round(sc["S"] / dt, 2), "unit": UNIT, "cores": host_cores(),
            "cpu": cpu_model(), "kind": "oracle",
            "sample": f"{sc['S']} tokens ({sc['G']} group(s)) of preset {n}, one oracle layer "
                      f"forward (numpy fp64, inputs upcast to fp64 beforehand: {t_up:.2f} s, "
                      f"untimed), {dt:.2f} s",
            "stages_s": {"layer": round(dt, 3), "router_and_routing": round(dt_route, 3),
                         "experts_and_combine": round(max(dt - dt_route, 0.0), 3)}}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    from top_gating_expert_gb300.inputs import make_inputs
    n = args.config
    cfg = preset_for(args)
    inp = make_inputs(cfg, preset_number=n)
    sc = _sample_cfg(cfg, sample_tokens(cfg, CPU_FLOPS_REFERENCE_STEP))
    arrays = oracle_arrays(inp.np, sc["S"])  # fp64 once, before timing
    del inp
    res = residual_for(n)
    for _ in range(args.warmup):
        _oracle_step(sc, arrays, res)
    t = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(sc, arrays, res)
    dt = time.perf_counter() - t
    value = sc["S"] * args.steps / dt
    cores = host_cores()
    sample = (f"each step: {sc['S']} tokens ({sc['G']} group(s)) of preset {n} (a bounded sample "
              f"of the workload), one oracle layer forward (numpy fp64, inputs upcast to fp64 "
              f"before timing) on {cores} host cores")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(cfg, n),
        "parallelism": "host cores (oracle), rank 0 only",
        "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores, "cpu": cpu_model(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    # a run that should take minutes: after 15 minutes, every thread's Python stack goes to
    # stderr (every 5 minutes), so that a stalled phase can be located afterwards
    faulthandler.dump_traceback_later(900, repeat=True, file=sys.stderr)
    if hasattr(signal, "SIGUSR1"):  # and on demand (kill -USR1)
        faulthandler.register(signal.SIGUSR1, file=sys.stderr, all_threads=True)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        line = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
