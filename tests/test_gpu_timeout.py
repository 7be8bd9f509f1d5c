"""The bounded waits' timeout path, on a real launch: with a one-microsecond wait limit set in
its workspace header, the router's single-CTA tcgen05 GEMM (moe_router, bf16) gives up
(every CTA's epilogue waits tens of microseconds for its first accumulator), drains what it
issued, frees its tensor memory and returns early; moe_get_device_status reports
MOE_ERR_TIMEOUT. With the default limit restored, the next call on the same workspace and
context succeeds and its logits match the oracle's fp64 projection."""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from gpu_util import LOGIT_RTOL, assert_close, to_np
from top_gating_expert_gb300 import _native as N
from top_gating_expert_gb300 import moe
from top_gating_expert_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

MOE_ERR_TIMEOUT = -5
# 128 tiles of 128 rows, each a K loop of 128 k-blocks (M = 8192): the first accumulator of
# a CTA takes far longer than the limit below
CFG = dict(S=16384, G=1, E=64, M=8192, H=128, k=2, capacity_factor=0.0, random_routing=0,
           n_shared=0, H_shared=0, act="relu", dtype="bf16", bias=False)


def test_wait_limit_times_out_then_recovers(native_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    inp = make_inputs(CFG, seed=4242, names=("x", "W_g"))
    x = inp.host["x"].cuda()
    W_g = inp.host["W_g"].cuda()
    ws = moe.workspace(CFG, N.MOE_WS_STEP)
    logits = torch.empty((CFG["S"], CFG["E"]), dtype=torch.float32, device="cuda")

    moe.set_wait_limit(ws, 1000)  # 1 microsecond
    moe.router(CFG, x, W_g, None, logits, ws)
    assert moe.device_status(ws) == MOE_ERR_TIMEOUT

    moe.set_wait_limit(ws, 0)  # back to the default
    for _ in range(2):
        logits.fill_(float("nan"))
        moe.router(CFG, x, W_g, None, logits, ws)
        assert moe.device_status(ws) == 0
    got = to_np(logits)
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([rng.choice(CFG["S"], 96, replace=False), [0, CFG["S"] - 1]]))
    ref = O.router_logits(inp.np["x"][rows], inp.np["W_g"])
    assert_close(got[rows], ref, LOGIT_RTOL["bf16"], "logits after the timeout")
    assert np.isfinite(got).all()
