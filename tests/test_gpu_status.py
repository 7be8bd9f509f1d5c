"""Failure detection without a GPU fault: status words injected into the workspace, and
invalid device offsets caught by the GEMM before it touches memory. No kernel here traps,
faults or waits on something that never happens."""

import ctypes

import numpy as np
import pytest
import torch

from top_gating_expert_gb300 import _native as N
from top_gating_expert_gb300 import moe

pytestmark = pytest.mark.gpu

CFG = dict(S=512, G=1, E=8, M=256, H=512, k=2, capacity_factor=0.0, random_routing=0,
           n_shared=0, H_shared=0, act="relu", dtype="bf16")


@pytest.fixture
def ws(native_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return moe.workspace(CFG, N.MOE_WS_STEP)


@pytest.mark.parametrize("bits,code", [(1, -5), (2, -6), (4, -7), (1 | 2, -5), (2 | 4, -6)])
def test_injected_status_word_is_reported_and_cleared(ws, bits, code):
    ws[:4].copy_(torch.tensor([bits], dtype=torch.int32).view(torch.uint8))
    assert moe.device_status(ws) == code
    assert moe.device_status(ws) == 0  # read-and-clear


def test_gemm_rejects_invalid_device_offsets(ws):
    """expert_offsets beyond the row buffer: the GEMM records MOE_ERR_DEVICE_DATA, runs no
    tile, and leaves its output untouched."""
    c = moe.make_config(CFG)
    R = moe.rows_max(c)
    dev = "cuda"
    x_perm = torch.randn(R, CFG["M"], device=dev).to(torch.bfloat16)
    W_in = torch.randn(CFG["E"], CFG["H"], CFG["M"], device=dev).to(torch.bfloat16)
    W_out = torch.randn(CFG["E"], CFG["M"], CFG["H"], device=dev).to(torch.bfloat16)
    W_in_p, _ = moe.pack_weights(c, W_in, None, W_out)
    offsets = torch.arange(CFG["E"] + 1, dtype=torch.int32, device=dev) * (R // CFG["E"])
    offsets[-1] = R + 1000  # past the end of the row buffer
    h = torch.full((R, CFG["H"]), 7.0, dtype=torch.bfloat16, device=dev)
    moe.expert_up(c, x_perm, offsets, W_in_p, h, ws)
    assert moe.device_status(ws) == -7
    assert torch.all(h == 7.0)
    offsets[-1] = R  # valid again: the same call succeeds and the context is usable
    moe.expert_up(c, x_perm, offsets, W_in_p, h, ws)
    assert moe.device_status(ws) == 0
    assert not torch.all(h == 7.0)
