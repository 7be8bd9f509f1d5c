"""Python binding of the MoE C ABI (include/moe.h): argument marshalling only.

Every step of the forward runs in the library's CUDA kernels; torch supplies device
memory and the current stream. Importing this module does not need a GPU; calling a
compute function does, and raises if the library is missing.
"""

from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _native as N


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = N.lib().moe_status_string(status)
        super().__init__(f"{where}: {msg.decode() if msg else status}")


def _check(rc: int, where: str):
    if rc != N.MOE_OK:
        raise MoeError(rc, where)


def make_config(cfg: dict) -> N.MoeConfig:
    """A moe_config_t from a workload dict (keys as in top_gating_expert_gb300.inputs)."""
    return N.MoeConfig(
        S=cfg["S"], G=cfg["G"], E=cfg["E"], M=cfg["M"], H=cfg["H"], k=cfg["k"],
        capacity_factor=float(cfg.get("capacity_factor", 0.0)),
        random_routing=int(cfg.get("random_routing", 0)),
        n_shared=int(cfg.get("n_shared", 0)), H_shared=int(cfg.get("H_shared", 0)),
        act=N.MOE_ACT_SWIGLU if cfg["act"] == "swiglu" else N.MOE_ACT_RELU,
        dtype=N.MOE_BF16 if cfg["dtype"] == "bf16" else N.MOE_F32,
        gate_norm=N.GATE_NORMS[cfg.get("gate_norm", "softmax_topk")],
        gate_p=float(cfg.get("gate_p", 1.0)),
        n_expert_groups=int(cfg.get("n_expert_groups", 0) or 0),
        topk_groups=int(cfg.get("topk_groups", 0) or 0),
        uniform_assignment=int(cfg.get("uniform_assignment", 0)))


def _cfg(c) -> N.MoeConfig:
    return c if isinstance(c, N.MoeConfig) else make_config(c)


def torch_dtype(cfg) -> torch.dtype:
    return torch.bfloat16 if _cfg(cfg).dtype == N.MOE_BF16 else torch.float32


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


# ------------------------------------------------------------------ host-only queries
def validate(cfg) -> int:
    return N.lib().moe_validate_config(ctypes.byref(_cfg(cfg)))


def capacity(cfg):
    C = N.c_int32()
    _check(N.lib().moe_capacity(ctypes.byref(_cfg(cfg)), ctypes.byref(C)), "moe_capacity")
    return None if C.value < 0 else C.value


def rows_max(cfg) -> int:
    R = N.c_int64()
    _check(N.lib().moe_rows_max(ctypes.byref(_cfg(cfg)), ctypes.byref(R)), "moe_rows_max")
    return R.value


def workspace_bytes(cfg, kind: int = N.MOE_WS_LAYER) -> int:
    b = N.c_size_t()
    _check(N.lib().moe_workspace_bytes(ctypes.byref(_cfg(cfg)), kind, ctypes.byref(b)),
           "moe_workspace_bytes")
    return b.value


def packed_sizes(cfg):
    """(W_in_packed, W_out_packed, Ws_in_packed, Ws_out_packed) element counts."""
    a, b, c, d = N.c_int64(), N.c_int64(), N.c_int64(), N.c_int64()
    _check(N.lib().moe_packed_sizes(ctypes.byref(_cfg(cfg)), ctypes.byref(a), ctypes.byref(b),
                                    ctypes.byref(c), ctypes.byref(d)), "moe_packed_sizes")
    return a.value, b.value, c.value, d.value


def workspace(cfg, kind: int = N.MOE_WS_LAYER, device="cuda") -> torch.Tensor:
    """A zero-filled workspace (torch allocations are 512-byte aligned)."""
    return torch.zeros(workspace_bytes(cfg, kind), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ routing outputs
@dataclass
class RouteOutputs:
    expert_id: torch.Tensor
    gate: torch.Tensor
    pos: torch.Tensor
    drop_reason: torch.Tensor
    row: torch.Tensor
    counts: torch.Tensor
    counts_routed: torch.Tensor
    expert_offsets: torch.Tensor
    token_of: torch.Tensor
    w_perm: torch.Tensor
    aux_loss: torch.Tensor
    z_loss: torch.Tensor

    @classmethod
    def allocate(cls, cfg, device="cuda") -> "RouteOutputs":
        c = _cfg(cfg)
        R = rows_max(c)
        z = lambda shape, dt: torch.zeros(shape, dtype=dt, device=device)
        return cls(expert_id=z((c.S, c.k), torch.int32), gate=z((c.S, c.k), torch.float32),
                   pos=z((c.S, c.k), torch.int32), drop_reason=z((c.S, c.k), torch.uint8),
                   row=z((c.S, c.k), torch.int32), counts=z((c.G, c.E), torch.int32),
                   counts_routed=z((c.G, c.E), torch.int32),
                   expert_offsets=z((c.E + 1,), torch.int32), token_of=z((R,), torch.int32),
                   w_perm=z((R,), torch.float32), aux_loss=z((1,), torch.float32),
                   z_loss=z((1,), torch.float32))

    def struct(self) -> N.MoeRouteOut:
        return N.MoeRouteOut(**{f: getattr(self, f).data_ptr() for f in N.ROUTE_FIELDS})


# ------------------------------------------------------------------ weight packing
def pack_weights(cfg, W_in, W_up, W_out, stream=None):
    """Returns (W_in_packed, W_out_packed) in the layout the expert GEMMs stream."""
    c = _cfg(cfg)
    n_in, n_out, _, _ = packed_sizes(c)
    p_in = torch.empty(n_in, dtype=W_in.dtype, device=W_in.device)
    p_out = torch.empty(n_out, dtype=W_in.dtype, device=W_in.device)
    _check(N.lib().moe_pack_weights(ctypes.byref(c), _ptr(W_in), _ptr(W_up), _ptr(W_out),
                                    _ptr(p_in), _ptr(p_out), _stream(stream)), "moe_pack_weights")
    return p_in, p_out


def pack_shared_weights(cfg, Ws_in, Ws_up, Ws_out, stream=None):
    c = _cfg(cfg)
    _, _, n_in, n_out = packed_sizes(c)
    p_in = torch.empty(n_in, dtype=Ws_in.dtype, device=Ws_in.device)
    p_out = torch.empty(n_out, dtype=Ws_in.dtype, device=Ws_in.device)
    _check(N.lib().moe_pack_shared_weights(ctypes.byref(c), _ptr(Ws_in), _ptr(Ws_up), _ptr(Ws_out),
                                           _ptr(p_in), _ptr(p_out), _stream(stream)),
           "moe_pack_shared_weights")
    return p_in, p_out


# ------------------------------------------------------------------ forward steps
def router(cfg, x, W_g, bias, logits, ws, stream=None):
    _check(N.lib().moe_router(ctypes.byref(_cfg(cfg)), _ptr(x), _ptr(W_g), _ptr(bias), _ptr(logits),
                              _ptr(ws), ws.numel(), _stream(stream)), "moe_router")


def route(cfg, logits, u, out: RouteOutputs, ws, stream=None):
    s = out.struct()
    _check(N.lib().moe_route(ctypes.byref(_cfg(cfg)), _ptr(logits), _ptr(u), ctypes.byref(s),
                             _ptr(ws), ws.numel(), _stream(stream)), "moe_route")


def router_route(cfg, x, W_g, bias, u, logits_out, out: RouteOutputs, ws, stream=None):
    """moe_router + moe_route in one pass (bf16: the logits stay on chip unless logits_out
    is given; fp32 needs logits_out)."""
    s = out.struct()
    _check(N.lib().moe_router_route(ctypes.byref(_cfg(cfg)), _ptr(x), _ptr(W_g), _ptr(bias), _ptr(u),
                                    _ptr(logits_out), ctypes.byref(s), _ptr(ws), ws.numel(),
                                    _stream(stream)), "moe_router_route")


def route_noalloc(cfg, logits, u, out: RouteOutputs, device_status=None, stream=None):
    """moe_route without a workspace (scratch in the library's fixed 4 MiB device array),
    for callers that cannot allocate device memory; see include/moe.h."""
    s = out.struct()
    _check(N.lib().moe_route_noalloc(ctypes.byref(_cfg(cfg)), _ptr(logits), _ptr(u), ctypes.byref(s),
                                     _ptr(device_status), _stream(stream)), "moe_route_noalloc")


def dispatch(cfg, x, out: RouteOutputs, x_perm, stream=None):
    s = out.struct()
    _check(N.lib().moe_dispatch(ctypes.byref(_cfg(cfg)), _ptr(x), ctypes.byref(s), _ptr(x_perm),
                                _stream(stream)), "moe_dispatch")


def expert_up(cfg, x_perm, expert_offsets, W_in_packed, h_perm, ws, stream=None):
    _check(N.lib().moe_expert_up(ctypes.byref(_cfg(cfg)), _ptr(x_perm), _ptr(expert_offsets),
                                 _ptr(W_in_packed), _ptr(h_perm), _ptr(ws), ws.numel(),
                                 _stream(stream)), "moe_expert_up")


def expert_down(cfg, h_perm, expert_offsets, w_perm, W_out_packed, y_perm, ws, stream=None):
    _check(N.lib().moe_expert_down(ctypes.byref(_cfg(cfg)), _ptr(h_perm), _ptr(expert_offsets),
                                   _ptr(w_perm), _ptr(W_out_packed), _ptr(y_perm), _ptr(ws),
                                   ws.numel(), _stream(stream)), "moe_expert_down")


def expert_ffn(cfg, x_perm, expert_offsets, w_perm, W_in_packed, W_out_packed, h_perm, y_perm, ws,
               stream=None):
    _check(N.lib().moe_expert_ffn(ctypes.byref(_cfg(cfg)), _ptr(x_perm), _ptr(expert_offsets),
                                  _ptr(w_perm), _ptr(W_in_packed), _ptr(W_out_packed), _ptr(h_perm),
                                  _ptr(y_perm), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_expert_ffn")


def shared_ffn(cfg, x, Ws_in_packed, Ws_out_packed, h_shared, shared_out, ws, stream=None):
    _check(N.lib().moe_shared_ffn(ctypes.byref(_cfg(cfg)), _ptr(x), _ptr(Ws_in_packed),
                                  _ptr(Ws_out_packed), _ptr(h_shared), _ptr(shared_out), _ptr(ws),
                                  ws.numel(), _stream(stream)), "moe_shared_ffn")


def combine(cfg, y_perm, out: RouteOutputs, shared_out, residual, y, stream=None):
    s = out.struct()
    _check(N.lib().moe_combine(ctypes.byref(_cfg(cfg)), _ptr(y_perm), ctypes.byref(s),
                               _ptr(shared_out), _ptr(residual), _ptr(y), _stream(stream)),
           "moe_combine")


def layer_forward(cfg, x, W_g, bias, W_in_packed, W_out_packed, Ws_in_packed, Ws_out_packed, u,
                  residual, y, logits_out, out: RouteOutputs, ws, stream=None):
    s = out.struct()
    _check(N.lib().moe_layer_forward(
        ctypes.byref(_cfg(cfg)), _ptr(x), _ptr(W_g), _ptr(bias), _ptr(W_in_packed), _ptr(W_out_packed),
        _ptr(Ws_in_packed), _ptr(Ws_out_packed), _ptr(u), _ptr(residual), _ptr(y), _ptr(logits_out),
        ctypes.byref(s), _ptr(ws), ws.numel(), _stream(stream)), "moe_layer_forward")


def pack_weights_backward(cfg, W_in, W_up, W_out, stream=None):
    """Transposed packs for the backward's data-gradient GEMMs: (Wt_in_packed, Wt_out_packed)."""
    c = _cfg(cfg)
    n_in, n_out, _, _ = packed_sizes(c)
    p_in = torch.empty(n_in, dtype=W_in.dtype, device=W_in.device)
    p_out = torch.empty(n_out, dtype=W_in.dtype, device=W_in.device)
    _check(N.lib().moe_pack_weights_backward(ctypes.byref(c), _ptr(W_in), _ptr(W_up), _ptr(W_out),
                                             _ptr(p_in), _ptr(p_out), _stream(stream)),
           "moe_pack_weights_backward")
    return p_in, p_out


def pack_shared_weights_backward(cfg, Ws_in, Ws_up, Ws_out, stream=None):
    c = _cfg(cfg)
    _, _, n_in, n_out = packed_sizes(c)
    p_in = torch.empty(n_in, dtype=Ws_in.dtype, device=Ws_in.device)
    p_out = torch.empty(n_out, dtype=Ws_in.dtype, device=Ws_in.device)
    _check(N.lib().moe_pack_shared_weights_backward(ctypes.byref(c), _ptr(Ws_in), _ptr(Ws_up),
                                                    _ptr(Ws_out), _ptr(p_in), _ptr(p_out),
                                                    _stream(stream)),
           "moe_pack_shared_weights_backward")
    return p_in, p_out


class Grads:
    """Device buffers for moe_layer_backward's outputs (fp32 weight gradients)."""

    def __init__(self, cfg, device="cuda", bias=False):
        c = _cfg(cfg)
        sw = c.act == N.MOE_ACT_SWIGLU
        f32 = lambda *shape: torch.zeros(shape, dtype=torch.float32, device=device)
        Hc = c.n_shared * c.H_shared
        self.dx = torch.zeros((c.S, c.M), dtype=torch_dtype(c), device=device)
        self.dW_g = f32(c.E, c.M)
        self.dbias = f32(c.E) if bias else None
        self.dW_in = f32(c.E, c.H, c.M)
        self.dW_up = f32(c.E, c.H, c.M) if sw else None
        self.dW_out = f32(c.E, c.M, c.H)
        self.dWs_in = f32(Hc, c.M) if Hc else None
        self.dWs_up = f32(Hc, c.M) if (Hc and sw) else None
        self.dWs_out = f32(c.M, Hc) if Hc else None

    def struct(self) -> N.MoeGrads:
        return N.MoeGrads(**{f: (getattr(self, f).data_ptr() if getattr(self, f) is not None else None)
                             for f in N.GRAD_FIELDS})


def layer_backward(cfg, x, dy, W_g, W_in_packed, Wt_in_packed, Wt_out_packed, Ws_in_packed,
                   Wst_in_packed, Wst_out_packed, logits, out: RouteOutputs, fwd_ws, residual,
                   aux_coef, z_coef, grads: Grads, ws, stream=None):
    s = out.struct()
    g = grads.struct()
    _check(N.lib().moe_layer_backward(
        ctypes.byref(_cfg(cfg)), _ptr(x), _ptr(dy), _ptr(W_g), _ptr(W_in_packed), _ptr(Wt_in_packed),
        _ptr(Wt_out_packed), _ptr(Ws_in_packed), _ptr(Wst_in_packed), _ptr(Wst_out_packed),
        _ptr(logits), ctypes.byref(s), _ptr(fwd_ws), fwd_ws.numel(), int(bool(residual)),
        float(aux_coef), float(z_coef), ctypes.byref(g), _ptr(ws), ws.numel(), _stream(stream)),
        "moe_layer_backward")


def device_status(ws, stream=None) -> int:
    """Synchronises the stream; returns (and clears) the device status recorded in ws."""
    return N.lib().moe_get_device_status(_ptr(ws), _stream(stream))


def set_wait_limit(ws, limit_ns: int, stream=None):
    """How long the kernels using workspace ws wait on their own pipeline before giving up
    (0 = the default of 2 s)."""
    _check(N.lib().moe_set_wait_limit(_ptr(ws), int(limit_ns), _stream(stream)),
           "moe_set_wait_limit")


# ------------------------------------------------------------------ a layer object
class MoeLayer:
    """Weights resident on one GPU (packed once), a workspace and routing outputs.

    ``forward`` runs moe_layer_forward on device tensors; ``forward_from_host`` copies
    the step's inputs from (pinned) host tensors, runs the layer and copies y and the two
    losses back."""

    def __init__(self, cfg: dict, weights: dict, device="cuda", keep_logits: bool = True):
        """keep_logits: also store the router logits in ``self.logits`` on every forward
        (for inspection and tests); without it the bf16 path never writes them."""
        self.cfg_dict = cfg
        self.cfg = make_config(cfg)
        _check(validate(self.cfg), "moe_validate_config")
        dt = torch_dtype(self.cfg)
        dev = torch.device(device)
        to = lambda t: None if t is None else t.to(device=dev, dtype=dt).contiguous()
        self.W_g = to(weights["W_g"])
        W_in, W_up, W_out = to(weights["W_in"]), to(weights.get("W_up")), to(weights["W_out"])
        self.W_in_packed, self.W_out_packed = pack_weights(self.cfg, W_in, W_up, W_out)
        del W_in, W_up, W_out
        self.bias = None if weights.get("bias") is None else weights["bias"].to(dev, torch.float32)
        self.Ws_in_packed = self.Ws_out_packed = None
        if self.cfg.n_shared > 0:
            self.Ws_in_packed, self.Ws_out_packed = pack_shared_weights(
                self.cfg, to(weights["Ws_in"]), to(weights.get("Ws_up")), to(weights["Ws_out"]))
        self.ws = workspace(self.cfg, N.MOE_WS_LAYER, dev)
        self.route_out = RouteOutputs.allocate(self.cfg, dev)
        self.logits = (torch.zeros((self.cfg.S, self.cfg.E), dtype=torch.float32, device=dev)
                       if keep_logits else None)
        self.y = torch.empty((self.cfg.S, self.cfg.M), dtype=dt, device=dev)
        self.device = dev

    def forward(self, x, u=None, residual=None, stream=None, out=None, route_out=None):
        """y (self.y unless `out` is given); the routing outputs go to self.route_out unless
        `route_out` (a RouteOutputs of this config) is given."""
        y = self.y if out is None else out
        layer_forward(self.cfg, x, self.W_g, self.bias, self.W_in_packed, self.W_out_packed,
                      self.Ws_in_packed, self.Ws_out_packed, u, residual, y, self.logits,
                      self.route_out if route_out is None else route_out, self.ws, stream)
        return y

    def enable_backward(self, weights: dict):
        """Pack the transposed weights the backward needs and allocate its workspace and
        gradient buffers (self.grads)."""
        dt = torch_dtype(self.cfg)
        to = lambda t: None if t is None else t.to(device=self.device, dtype=dt).contiguous()
        self.Wt_in_packed, self.Wt_out_packed = pack_weights_backward(
            self.cfg, to(weights["W_in"]), to(weights.get("W_up")), to(weights["W_out"]))
        self.Wst_in_packed = self.Wst_out_packed = None
        if self.cfg.n_shared > 0:
            self.Wst_in_packed, self.Wst_out_packed = pack_shared_weights_backward(
                self.cfg, to(weights["Ws_in"]), to(weights.get("Ws_up")), to(weights["Ws_out"]))
        self.ws_bwd = workspace(self.cfg, N.MOE_WS_BACKWARD, self.device)
        self.grads = Grads(self.cfg, self.device, bias=self.bias is not None)

    def backward(self, x, dy, residual=False, aux_coef=0.0, z_coef=0.0, stream=None):
        """Gradients of sum(dy * y) + aux_coef * aux + z_coef * z for the last forward on x
        (which must have kept its logits), into self.grads."""
        if self.logits is None:
            raise RuntimeError("the backward needs the forward's logits (keep_logits=True)")
        layer_backward(self.cfg, x, dy, self.W_g, self.W_in_packed, self.Wt_in_packed,
                       self.Wt_out_packed, self.Ws_in_packed, self.Wst_in_packed,
                       self.Wst_out_packed, self.logits, self.route_out, self.ws, residual,
                       aux_coef, z_coef, self.grads, self.ws_bwd, stream)
        return self.grads

    def capture(self, x, u=None, residual=None, warmup: int = 1) -> torch.cuda.CUDAGraph:
        """Capture forward(x, u, residual) into a CUDA graph (one launch per replay). x, u,
        residual and the layer's outputs stay the graph's fixed buffers: write new inputs
        into them and call replay()."""
        side = torch.cuda.Stream(device=self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            for _ in range(warmup):
                self.forward(x, u, residual)
        torch.cuda.current_stream(self.device).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self.forward(x, u, residual)
        self._graph = graph
        return graph

    def replay(self):
        self._graph.replay()
        return self.y

    def forward_from_host(self, x_host, u_host=None, y_host=None, losses_host=None, stream=None):
        """x_host (and u_host) pinned CPU tensors; y_host / losses_host pinned outputs."""
        if not hasattr(self, "_x_dev"):
            self._x_dev = torch.empty_like(x_host, device=self.device)
            self._u_dev = None if u_host is None else torch.empty_like(u_host, device=self.device)
            self._loss_dev = torch.empty(2, dtype=torch.float32, device=self.device)
        self._x_dev.copy_(x_host, non_blocking=True)
        if u_host is not None:
            self._u_dev.copy_(u_host, non_blocking=True)
        self.forward(self._x_dev, self._u_dev if u_host is not None else None, stream=stream)
        if y_host is not None:
            y_host.copy_(self.y, non_blocking=True)
        if losses_host is not None:
            self._loss_dev[0:1].copy_(self.route_out.aux_loss)
            self._loss_dev[1:2].copy_(self.route_out.z_loss)
            losses_host.copy_(self._loss_dev, non_blocking=True)
        return y_host


class HostPipeline:
    """Pinned-host in, pinned-host out, `depth` steps in flight.

    Step i copies its inputs host->device on a copy stream, runs the layer (a CUDA graph per
    buffer set) on the compute stream, and copies y and the two losses device->host on a
    second copy stream, so step i's input copy and step i-1's output copy overlap the
    compute of the steps around them. Buffer set i % depth is reused only after step
    i - depth's output copy has finished. Each buffer set has its own routing outputs
    (``route[i % depth]`` holds step i's), so the output copy reads the two losses from
    them directly."""

    def __init__(self, layer: MoeLayer, has_u: bool, depth: int = 2, residual: bool = False):
        """residual: the layer adds its input x to the expert output (y = x + MoE(x))."""
        dev = layer.device
        c = layer.cfg
        dt = torch_dtype(c)
        self.layer, self.depth = layer, depth
        self.x = [torch.empty((c.S, c.M), dtype=dt, device=dev) for _ in range(depth)]
        self.u = [torch.empty(c.S, dtype=torch.float32, device=dev) if has_u else None
                  for _ in range(depth)]
        self.y = [torch.empty((c.S, c.M), dtype=dt, device=dev) for _ in range(depth)]
        self.route = [RouteOutputs.allocate(c, dev) for _ in range(depth)]
        self.compute = torch.cuda.current_stream(dev)
        self.h2d = torch.cuda.Stream(device=dev)
        self.d2h = torch.cuda.Stream(device=dev)
        self.ev_in = [torch.cuda.Event() for _ in range(depth)]
        self.ev_done = [torch.cuda.Event() for _ in range(depth)]
        self.ev_free = [torch.cuda.Event() for _ in range(depth)]
        self.graphs = []
        for b in range(depth):
            self.x[b].zero_()
            if has_u:
                self.u[b].fill_(0.5)
            side = torch.cuda.Stream(device=dev)
            side.wait_stream(self.compute)
            res = self.x[b] if residual else None
            with torch.cuda.stream(side):
                layer.forward(self.x[b], self.u[b], res, out=self.y[b], route_out=self.route[b])
            self.compute.wait_stream(side)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                layer.forward(self.x[b], self.u[b], res, out=self.y[b], route_out=self.route[b])
            self.graphs.append(g)
        torch.cuda.synchronize(dev)

    def submit(self, i: int, x_host, u_host=None, y_host=None, loss_host=None):
        b = i % self.depth
        self.h2d.wait_event(self.ev_free[b])
        with torch.cuda.stream(self.h2d):
            self.x[b].copy_(x_host, non_blocking=True)
            if u_host is not None:
                self.u[b].copy_(u_host, non_blocking=True)
            self.ev_in[b].record(self.h2d)
        self.compute.wait_event(self.ev_in[b])
        self.graphs[b].replay()
        self.ev_done[b].record(self.compute)
        self.d2h.wait_event(self.ev_done[b])
        with torch.cuda.stream(self.d2h):
            if y_host is not None:
                y_host.copy_(self.y[b], non_blocking=True)
            if loss_host is not None:
                loss_host[0:1].copy_(self.route[b].aux_loss, non_blocking=True)
                loss_host[1:2].copy_(self.route[b].z_loss, non_blocking=True)
            self.ev_free[b].record(self.d2h)
