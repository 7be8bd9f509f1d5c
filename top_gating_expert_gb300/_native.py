"""ctypes declarations of the C ABI in include/moe.h (argument marshalling only)."""

from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

c_int32, c_int64, c_float, c_size_t, c_void_p = (ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                                 ctypes.c_size_t, ctypes.c_void_p)

MOE_F32, MOE_BF16 = 0, 1
MOE_ACT_RELU, MOE_ACT_SWIGLU = 0, 1
GATE_NORMS = {"softmax_topk": 0, "none": 1, "pnorm": 2}
MOE_WS_STEP, MOE_WS_LAYER, MOE_WS_BACKWARD = 0, 1, 2
MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED",
                -3: "MOE_ERR_WORKSPACE", -4: "MOE_ERR_CUDA", -5: "MOE_ERR_TIMEOUT",
                -6: "MOE_ERR_NONFINITE", -7: "MOE_ERR_DEVICE_DATA"}


class MoeConfig(ctypes.Structure):
    _fields_ = [("S", c_int32), ("G", c_int32), ("E", c_int32), ("M", c_int32), ("H", c_int32),
                ("k", c_int32), ("capacity_factor", c_float), ("random_routing", c_int32),
                ("n_shared", c_int32), ("H_shared", c_int32), ("act", c_int32), ("dtype", c_int32),
                ("gate_norm", c_int32), ("gate_p", c_float), ("n_expert_groups", c_int32),
                ("topk_groups", c_int32), ("uniform_assignment", c_int32)]


ROUTE_FIELDS = ("expert_id", "gate", "pos", "drop_reason", "row", "counts", "counts_routed",
                "expert_offsets", "token_of", "w_perm", "aux_loss", "z_loss")


class MoeRouteOut(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ROUTE_FIELDS]


GRAD_FIELDS = ("dx", "dW_g", "dbias", "dW_in", "dW_up", "dW_out", "dWs_in", "dWs_up", "dWs_out")


class MoeGrads(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in GRAD_FIELDS]


_P = ctypes.POINTER
# name -> argtypes (restype c_int unless listed in _RESTYPES)
_PROTOTYPES = {
    "moe_status_string": [ctypes.c_int],
    "moe_abi_version": [],
    "moe_validate_config": [_P(MoeConfig)],
    "moe_capacity": [_P(MoeConfig), _P(c_int32)],
    "moe_rows_max": [_P(MoeConfig), _P(c_int64)],
    "moe_workspace_bytes": [_P(MoeConfig), ctypes.c_int, _P(c_size_t)],
    "moe_packed_sizes": [_P(MoeConfig), _P(c_int64), _P(c_int64), _P(c_int64), _P(c_int64)],
    "moe_pack_weights": [_P(MoeConfig), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                         c_void_p],
    "moe_pack_shared_weights": [_P(MoeConfig), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                c_void_p],
    "moe_router": [_P(MoeConfig), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                   c_void_p],
    "moe_route": [_P(MoeConfig), c_void_p, c_void_p, _P(MoeRouteOut), c_void_p, c_size_t, c_void_p],
    "moe_router_route": [_P(MoeConfig), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                         _P(MoeRouteOut), c_void_p, c_size_t, c_void_p],
    "moe_route_noalloc": [_P(MoeConfig), c_void_p, c_void_p, _P(MoeRouteOut), c_void_p, c_void_p],
    "moe_dispatch": [_P(MoeConfig), c_void_p, _P(MoeRouteOut), c_void_p, c_void_p],
    "moe_expert_up": [_P(MoeConfig), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                      c_void_p],
    "moe_expert_down": [_P(MoeConfig), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                        c_size_t, c_void_p],
    "moe_expert_ffn": [_P(MoeConfig), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                       c_void_p, c_void_p, c_size_t, c_void_p],
    "moe_shared_ffn": [_P(MoeConfig), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                       c_size_t, c_void_p],
    "moe_combine": [_P(MoeConfig), c_void_p, _P(MoeRouteOut), c_void_p, c_void_p, c_void_p,
                    c_void_p],
    "moe_layer_forward": [_P(MoeConfig), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                          c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, _P(MoeRouteOut),
                          c_void_p, c_size_t, c_void_p],
    "moe_pack_weights_backward": [_P(MoeConfig), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                  c_void_p],
    "moe_pack_shared_weights_backward": [_P(MoeConfig), c_void_p, c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_void_p],
    "moe_layer_backward": [_P(MoeConfig), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                           c_void_p, c_void_p, c_void_p, c_void_p, _P(MoeRouteOut), c_void_p,
                           c_size_t, ctypes.c_int, c_float, c_float, _P(MoeGrads), c_void_p,
                           c_size_t, c_void_p],
    "moe_get_device_status": [c_void_p, c_void_p],
    "moe_set_wait_limit": [c_void_p, ctypes.c_uint64, c_void_p],
}
_RESTYPES = {"moe_status_string": ctypes.c_char_p}

_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library. Raises if it has not been built: there is no fallback."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"the CUDA MoE library {path} is not built; run "
                    "`python -m top_gating_expert_gb300.build` (or __graft_entry__.build())")
            L = ctypes.CDLL(path)
            for name, args in _PROTOTYPES.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = _RESTYPES.get(name, ctypes.c_int)
            _lib = L
    return _lib


def declared_symbols(header: str | None = None) -> list[str]:
    """Names of the functions declared in include/moe.h."""
    import re
    header = header or os.path.join(_build.INCLUDE, "moe.h")
    with open(header) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))
