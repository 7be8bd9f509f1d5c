"""Host-side checks of the C ABI: the library loads without a GPU, exports every function
include/moe.h declares, and its host-only queries and argument checks behave."""

import ctypes
import math

import pytest

from top_gating_expert_gb300 import _native as N
from top_gating_expert_gb300.inputs import PRESETS, preset


def test_exports_every_declared_symbol(native_lib):
    declared = N.declared_symbols()
    assert len(declared) >= 19
    missing = [s for s in declared if not hasattr(native_lib, s)]
    assert not missing, missing
    # and the binding declares a prototype for each
    assert set(declared) == set(N._PROTOTYPES), set(declared) ^ set(N._PROTOTYPES)


def test_status_strings(native_lib):
    for code, name in N.STATUS_NAMES.items():
        assert native_lib.moe_status_string(code).decode().startswith(name)
    assert native_lib.moe_abi_version() == 102


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_presets_validate_and_capacity(native_lib, n):
    from top_gating_expert_gb300 import moe
    cfg = PRESETS[n]
    assert moe.validate(cfg) == 0
    want_C = None if cfg["capacity_factor"] <= 0 else math.ceil(
        cfg["capacity_factor"] * cfg["k"] * (cfg["S"] // cfg["G"]) / cfg["E"])
    assert moe.capacity(cfg) == want_C
    sk = cfg["S"] * cfg["k"]
    assert moe.rows_max(cfg) == (sk if want_C is None else min(sk, cfg["G"] * cfg["E"] * want_C))
    step = moe.workspace_bytes(cfg, N.MOE_WS_STEP)
    layer = moe.workspace_bytes(cfg, N.MOE_WS_LAYER)
    assert 0 < step < layer
    R = moe.rows_max(cfg)
    eb = 2 if cfg["dtype"] == "bf16" else 4
    assert layer >= step + R * (2 * cfg["M"] + cfg["H"]) * eb


def test_capacity_values(native_lib):
    from top_gating_expert_gb300 import moe
    assert moe.capacity(PRESETS[1]) == 64
    assert moe.capacity(PRESETS[2]) == 16
    assert moe.capacity(PRESETS[5]) == 2560
    assert moe.capacity(PRESETS[3]) is None


BAD = [
    dict(S=100, G=3),             # S % G != 0
    dict(S=0, G=1),               # no tokens: an empty batch is rejected, not launched
    dict(E=0), dict(E=300),       # expert count
    dict(k=0), dict(k=9),         # k range
    dict(k=3, random_routing=1),  # random routing needs k == 2
    dict(random_routing=2),
    dict(n_shared=1, H_shared=0),
    dict(gate_norm="pnorm", gate_p=0.0), dict(gate_norm="pnorm", gate_p=float("inf")),
    dict(n_expert_groups=3),                        # does not divide E = 128
    dict(n_expert_groups=32, topk_groups=4),        # more than 16 groups
    dict(n_expert_groups=8, topk_groups=0), dict(n_expert_groups=8, topk_groups=9),
    dict(E=16, n_expert_groups=8, topk_groups=1, k=3, random_routing=0),  # 1 group of 2 < k
    dict(uniform_assignment=1),                     # preset 2 has random routing
    dict(uniform_assignment=2, random_routing=0),
]


@pytest.mark.parametrize("over", BAD)
def test_invalid_configs_rejected(native_lib, over):
    from top_gating_expert_gb300 import moe
    cfg = preset(2, **over)
    assert moe.validate(cfg) == -1


def test_valid_variant_configs(native_lib):
    from top_gating_expert_gb300 import moe
    for over in (dict(gate_norm="none"), dict(gate_norm="pnorm", gate_p=2.0),
                 dict(n_expert_groups=8, topk_groups=4), dict(n_expert_groups=16, topk_groups=1),
                 dict(uniform_assignment=1, random_routing=0)):
        assert moe.validate(preset(2, **over)) == 0, over


@pytest.mark.parametrize("n", [2, 3, 4, 5])
def test_bench_routing_variants_validate(native_lib, n):
    """Every routing variant the benchmark times is a valid configuration of each bf16 preset."""
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    from top_gating_expert_gb300 import moe
    for name, over in bench.VARIANTS.items():
        assert moe.validate(preset(n, **over)) == 0, (n, name)


def test_group_index_by_multiply_shift():
    """The variant top-k filter finds an expert's group as (e * ceil(2^24 / gsz)) >> 24 in
    32-bit arithmetic; exact for every expert index and group size up to 256."""
    for gsz in range(1, 257):
        m = ((1 << 24) + gsz - 1) // gsz
        for e in range(256):
            assert ((e * m) & 0xFFFFFFFF) >> 24 == e // gsz


@pytest.mark.parametrize("over", [dict(M=1000), dict(H=4000), dict(act="swiglu", H=4160)])
def test_unsupported_shapes(native_lib, over):
    from top_gating_expert_gb300 import moe
    assert moe.validate(preset(2, **over)) == -2


def test_compute_entry_points_check_arguments_on_host(native_lib):
    """Null pointers and short workspaces fail before any launch (no GPU needed)."""
    from top_gating_expert_gb300 import moe
    c = moe.make_config(PRESETS[2])
    L = native_lib
    out = N.MoeRouteOut()
    assert L.moe_route(ctypes.byref(c), None, None, ctypes.byref(out), None, 0, None) == -1
    fake = ctypes.c_void_p(1 << 20)
    out2 = N.MoeRouteOut(**{f: (1 << 20) for f in N.ROUTE_FIELDS})
    # workspace too small
    assert L.moe_route(ctypes.byref(c), fake, fake, ctypes.byref(out2), fake, 16, None) == -3
    # misaligned workspace
    need = moe.workspace_bytes(c, N.MOE_WS_STEP)
    assert L.moe_route(ctypes.byref(c), fake, fake, ctypes.byref(out2), ctypes.c_void_p((1 << 20) + 8),
                       need, None) == -3
    assert L.moe_router(ctypes.byref(c), None, fake, None, fake, fake, need, None) == -1
    assert L.moe_dispatch(ctypes.byref(c), fake, None, fake, None) == -1
    assert L.moe_combine(ctypes.byref(c), fake, ctypes.byref(out2), None, None, None, None) == -1
    assert L.moe_expert_ffn(ctypes.byref(c), None, fake, fake, fake, fake, fake, fake, fake, need,
                            None) == -1
    assert L.moe_layer_forward(ctypes.byref(c), fake, fake, None, fake, fake, None, None, fake, None,
                               fake, None, ctypes.byref(out2), fake, 16, None) == -3
    assert L.moe_router_route(ctypes.byref(c), None, fake, None, fake, None, ctypes.byref(out2), fake,
                              need, None) == -1
    assert L.moe_router_route(ctypes.byref(c), fake, fake, None, None, None, ctypes.byref(out2), fake,
                              need, None) == -1  # random routing needs u
    assert L.moe_router_route(ctypes.byref(c), fake, fake, None, fake, None, ctypes.byref(out2), fake,
                              16, None) == -3
    c32 = moe.make_config(PRESETS[1])
    assert L.moe_router_route(ctypes.byref(c32), fake, fake, None, fake, None, ctypes.byref(out2),
                              fake, moe.workspace_bytes(c32, N.MOE_WS_STEP), None) == -1  # fp32 needs logits_out
    assert L.moe_get_device_status(None, None) == -1
    # the wait limit lives in a workspace header: null or misaligned workspaces are refused
    assert L.moe_set_wait_limit(None, 1000, None) == -1
    assert L.moe_set_wait_limit(ctypes.c_void_p((1 << 20) + 8), 1000, None) == -1
    # shared-expert calls need shared experts
    assert L.moe_shared_ffn(ctypes.byref(c), fake, fake, fake, fake, fake, fake, need, None) == -1


def test_backward_host_checks(native_lib):
    """The backward's workspace kind and its argument checks, before any launch."""
    from top_gating_expert_gb300 import moe
    L = native_lib
    c = moe.make_config(PRESETS[2])
    step = moe.workspace_bytes(c, N.MOE_WS_STEP)
    bwd = moe.workspace_bytes(c, N.MOE_WS_BACKWARD)
    assert bwd > step
    fake = ctypes.c_void_p(1 << 20)
    out = N.MoeRouteOut(**{f: (1 << 20) for f in N.ROUTE_FIELDS})
    g = N.MoeGrads(**{f: (1 << 20) for f in N.GRAD_FIELDS})
    lay = moe.workspace_bytes(c, N.MOE_WS_LAYER)
    args = lambda **kw: [kw.get(n, v) for n, v in (
        ("x", fake), ("dy", fake), ("W_g", fake), ("W_in_p", fake), ("Wt_in", fake), ("Wt_out", fake),
        ("Ws_in", None), ("Wst_in", None), ("Wst_out", None), ("logits", fake))]
    tail = lambda fwd=fake, fwd_bytes=lay, ws=fake, ws_bytes=bwd, grads=g: (
        ctypes.byref(out), fwd, fwd_bytes, 0, ctypes.c_float(0.0), ctypes.c_float(0.0),
        ctypes.byref(grads), ws, ws_bytes, None)
    assert L.moe_layer_backward(ctypes.byref(c), *args(dy=None), *tail()) == -1
    assert L.moe_layer_backward(ctypes.byref(c), *args(logits=None), *tail()) == -1
    assert L.moe_layer_backward(ctypes.byref(c), *args(), *tail(ws_bytes=16)) == -3
    assert L.moe_layer_backward(ctypes.byref(c), *args(), *tail(fwd_bytes=16)) == -3
    g0 = N.MoeGrads(**{f: (1 << 20) for f in N.GRAD_FIELDS}); g0.dW_in = None
    assert L.moe_layer_backward(ctypes.byref(c), *args(), *tail(grads=g0)) == -1
    # fp32 layers have a backward too (plain FMA); its checks come before any launch as well
    c32 = moe.make_config(PRESETS[1])
    b32 = moe.workspace_bytes(c32, N.MOE_WS_BACKWARD)
    assert L.moe_layer_backward(ctypes.byref(c32), *args(), *tail(ws_bytes=b32 - 256)) == -3
    assert L.moe_layer_backward(ctypes.byref(c32), *args(dy=None), *tail(ws_bytes=b32)) == -1
    cu = moe.make_config(preset(2, uniform_assignment=1, random_routing=0))
    assert L.moe_layer_backward(ctypes.byref(cu), *args(), *tail()) == -2    # forward-only ids
    assert L.moe_pack_weights_backward(ctypes.byref(c32), None, fake, fake, fake, fake, None) == -1
