"""moe_route_noalloc: routing for callers that cannot allocate device memory (a plugin
inside a framework that owns all device memory, a loop that must not allocate after
start-up). Its scratch is a fixed array inside the library, so the caller passes only
inputs and outputs. Checked through the C ABI on two calls in a row: against moe_route (the
entry point with a caller workspace) and against the oracle's routing; and the second call
allocates nothing (device free memory and the torch allocator's counters are unchanged
across it).

This file is collected last on purpose: a run that stops at the first failure has run
every other test before this one."""

import ctypes

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from gpu_util import GATE_RTOL, LOSS_RTOL, compare_route, oracle_cfg, route_np
from top_gating_expert_gb300 import _native as N
from top_gating_expert_gb300 import moe

pytestmark = pytest.mark.gpu

CFG = dict(S=6000, G=3, E=64, M=64, H=128, k=2, capacity_factor=1.0, random_routing=1,
           n_shared=0, H_shared=0, act="relu", dtype="bf16")


def _inputs(seed):
    rng = np.random.default_rng(seed)
    logits = (rng.standard_normal((CFG["S"], CFG["E"])) * 2).astype(np.float32)
    if seed % 2:  # exact ties in the second call
        logits = np.round(logits * 2) / 2
    u = rng.random(CFG["S"], dtype=np.float32)
    return logits, u


def _alloc_state():
    torch.cuda.synchronize()
    free, _ = torch.cuda.mem_get_info()
    st = torch.cuda.memory_stats()
    return free, {k: st.get(k, 0) for k in ("allocated_bytes.all.current",
                                            "reserved_bytes.all.current",
                                            "allocation.all.allocated",
                                            "segment.all.allocated")}


def test_route_noalloc_matches_route(native_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = native_lib
    c = moe.make_config(CFG)
    need = moe.workspace_bytes(c, N.MOE_WS_STEP)
    assert need <= 4 << 20
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # everything either call touches is allocated before the first one
    host = [_inputs(seed) for seed in (1, 2)]
    dev = [(torch.from_numpy(lg).cuda(), torch.from_numpy(uu).cuda()) for lg, uu in host]
    got = [moe.RouteOutputs.allocate(c) for _ in host]
    status = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    structs = [g.struct() for g in got]

    states = []
    for i, (logits, u) in enumerate(dev):  # two calls in a row into separate outputs
        states.append(_alloc_state())
        rc = lib.moe_route_noalloc(ctypes.byref(c), ctypes.c_void_p(logits.data_ptr()),
                                   ctypes.c_void_p(u.data_ptr()), ctypes.byref(structs[i]),
                                   ctypes.c_void_p(status.data_ptr() + 4 * i), stream)
        assert rc == 0
    states.append(_alloc_state())
    # the second call (after the first has set up its device address) allocated nothing
    assert states[2] == states[1], (states[1], states[2])
    assert status.tolist() == [0, 0]

    for i, (logits, u) in enumerate(dev):
        # the entry point with a caller workspace, on the same inputs
        ref = moe.RouteOutputs.allocate(c)
        ws = moe.workspace(c, N.MOE_WS_STEP)
        moe.route(c, logits, u, ref, ws)
        assert moe.device_status(ws) == 0
        a, b = route_np(got[i]), route_np(ref)
        for key in ("expert_id", "pos", "drop_reason", "row", "counts", "counts_routed",
                    "expert_offsets"):
            assert np.array_equal(a[key], b[key]), key
        R = int(b["expert_offsets"][-1])
        assert np.array_equal(a["token_of"][:R], b["token_of"][:R])
        np.testing.assert_allclose(a["gate"], b["gate"], rtol=GATE_RTOL, atol=1e-30)
        np.testing.assert_allclose(a["w_perm"][:R], b["w_perm"][:R], rtol=GATE_RTOL, atol=1e-30)
        np.testing.assert_allclose(a["aux_loss"], b["aux_loss"], rtol=LOSS_RTOL)
        np.testing.assert_allclose(a["z_loss"], b["z_loss"], rtol=LOSS_RTOL)
        # and the oracle's routing of the same logits and uniform draws
        compare_route(a, O.route(host[i][0], oracle_cfg(CFG), host[i][1]), f"noalloc call {i + 1}")


def test_route_noalloc_rejects_sizes_beyond_its_array(native_lib):
    big = moe.make_config(dict(CFG, S=2 ** 20, G=1, E=256, k=8, random_routing=0))
    assert moe.workspace_bytes(big, N.MOE_WS_STEP) > 4 << 20
    out = N.MoeRouteOut(**{f: 1 << 20 for f in N.ROUTE_FIELDS})
    rc = native_lib.moe_route_noalloc(ctypes.byref(big), ctypes.c_void_p(1 << 20), None,
                                      ctypes.byref(out), None, None)
    assert rc == -3  # MOE_ERR_WORKSPACE, before any launch
