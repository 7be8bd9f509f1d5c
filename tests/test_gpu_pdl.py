"""Programmatic dependent launch changes when kernels start, never what they compute: several
kernels do work before their `griddepcontrol.wait` (weight prefetches into L2, the GEMM's
guess of its first tile), and all of it must be free of results. The switch (MOE_PDL=0) is
read once per process, so a child process computes the same layer — forward and backward —
without it, and every output must equal this process's bit for bit."""

import os
import subprocess
import sys
import tempfile

import numpy as np
import pytest
import torch

from gpu_util import to_np
from top_gating_expert_gb300 import moe
from top_gating_expert_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CFG = dict(S=3000, G=2, E=64, M=512, H=512, k=2, capacity_factor=1.0, random_routing=1,
           n_shared=0, H_shared=0, act="relu", dtype="bf16", bias=False)
FIELDS = ("y", "dx", "dW_g", "dW_in", "dW_out")


def _run_layer(cfg):
    inp = make_inputs(cfg, seed=11)
    layer = moe.MoeLayer(cfg, inp.host)
    layer.enable_backward(inp.host)
    x, u = inp.host["x"].cuda(), inp.host["u"].cuda()
    y = to_np(layer.forward(x, u))
    dy = torch.randn((cfg["S"], cfg["M"]), generator=torch.Generator().manual_seed(12))
    g = layer.backward(x, dy.to(torch.bfloat16).cuda(), aux_coef=0.5, z_coef=0.25)
    assert moe.device_status(layer.ws) == 0 and moe.device_status(layer.ws_bwd) == 0
    out = {f: to_np(getattr(g, f)) for f in FIELDS[1:]}
    out["y"] = y
    out["expert_offsets"] = to_np(layer.route_out.expert_offsets)
    return out


def test_layer_without_pdl_is_bit_identical(native_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    here = _run_layer(CFG)
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "nopdl.npz")
        code = ("import sys, numpy as np; sys.path.insert(0, %r); sys.path.insert(0, %r)\n"
                "from test_gpu_pdl import _run_layer, CFG\n"
                "np.savez(%r, **_run_layer(CFG))\n") % (ROOT, os.path.join(ROOT, "tests"), path)
        env = dict(os.environ, MOE_PDL="0")
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                           timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        other = dict(np.load(path))
    for f in here:
        assert np.array_equal(here[f], other[f]), f"{f} differs without programmatic dependent launch"
