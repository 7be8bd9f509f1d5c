"""Host-side pieces of bench.py that need no GPU: workload overrides, the bounded oracle
sample, the workload description, the routing variants it times and the roofline traffic
lookup."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from top_gating_expert_gb300.inputs import PRESETS  # noqa: E402


def _args(*argv):
    old = sys.argv
    try:
        sys.argv = ["bench.py", *argv]
        return bench.parse()
    finally:
        sys.argv = old


def test_defaults_are_one_gpu_headline_on_the_largest_preset():
    a = _args()
    assert (a.gpus, a.config, a.impl) == (1, bench.HEADLINE, "ours")
    assert a.warmup >= 3 and a.steps >= 1
    # the headline is the preset with the most expert-GEMM work
    def work(c):
        f = 3 if c["act"] == "swiglu" else 2
        return 2 * f * c["S"] * c["k"] * c["M"] * c["H"] + \
            2 * f * c["S"] * c["M"] * c["n_shared"] * c["H_shared"]
    assert bench.HEADLINE == max(PRESETS, key=lambda n: work(PRESETS[n]))
    # every other preset is measured into the line's "presets" object by default
    assert bench.other_presets(a) == [n for n in sorted(PRESETS) if n != bench.HEADLINE]
    assert bench.other_presets(_args("--presets", "none")) == []
    assert bench.other_presets(_args("--config", "2", "--presets", "2,5")) == [5]


def test_override_changes_fields_and_names_them():
    a = _args("--config", "2", "--override", "S=4096", "--override", "G=4", "--override", "E=32")
    cfg = bench.preset_for(a)
    assert (cfg["S"], cfg["G"], cfg["E"]) == (4096, 4, 32)
    assert isinstance(cfg["S"], int) and "S=4096" in cfg["name"]
    assert cfg["M"] == PRESETS[2]["M"]
    # overrides apply to the headline preset only
    assert bench.preset_for(a, 5) == PRESETS[5]


def test_both_arms_print_the_same_config():
    cfg = PRESETS[3]
    c = bench.workload_config(cfg, 3)
    assert c == bench.workload_config(dict(cfg), 3)
    assert c["workload"].startswith("preset 3 ") and "l2" in c
    assert "residual added" in bench.workload_config(PRESETS[5], 5)["workload"]


def test_oracle_arrays_are_fp64_and_cut_to_the_sample():
    import numpy as np
    a = {"x": np.ones((10, 4), np.float32), "u": np.ones(10, np.float32),
         "W_g": np.ones((3, 4), np.float32)}
    o = bench.oracle_arrays(a, 6)
    assert o["x"].shape == (6, 4) and o["u"].shape == (6,) and o["W_g"].shape == (3, 4)
    assert all(v.dtype == np.float64 for v in o.values())


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_cpu_sample_is_bounded(n):
    cfg = PRESETS[n]
    t = bench.sample_tokens(cfg, bench.CPU_FLOPS_REFERENCE_STEP)
    assert min(256, cfg["S"]) <= t <= cfg["S"]


def test_roofline_picks_the_binding_bound():
    P = {"hbm": 6000.0, "tc": 2000.0, "tc_sustained": 1800.0, "source": "test"}
    algo = {"a": (6e9, 1e9), "b": (1e6, 1.8e12)}
    ra = bench.roofline_of("a", 2.0, algo, P, 9)
    assert ra["bound"] == "hbm" and ra["frac"] == pytest.approx(0.5)
    rb = bench.roofline_of("b", 2.0, algo, P, 9)
    assert rb["bound"] == "tensor" and rb["frac"] == pytest.approx(0.5)
    assert rb["frac_of_burst_peak"] == pytest.approx(0.45)


def test_override_rejects_unknown_fields():
    with pytest.raises(SystemExit):
        bench.preset_for(_args("--override", "not_a_field=1"))


@pytest.mark.parametrize("n", [2, 5])
def test_oracle_sample_is_whole_groups_or_a_prefix(n):
    cfg = PRESETS[n]
    sc = bench._sample_cfg(cfg, 3000)
    if cfg["G"] > 1:
        Sg = cfg["S"] // cfg["G"]
        assert sc["S"] % Sg == 0 and sc["S"] // sc["G"] == Sg
    else:
        assert sc["S"] == 3000 and sc["G"] == 1


def test_workload_description_names_the_shape():
    d = bench.workload_desc(PRESETS[2], 2)
    for key in ("S", "G", "E", "k", "M", "H"):
        assert d[key] == PRESETS[2][key]
    assert "capacity factor" in d["workload"] and "random 2nd-expert" in d["workload"]


def test_variants_are_routing_fields_only():
    # every variant changes routing fields, never the expert FFN's shape or dtype
    for name, kw in bench.VARIANTS.items():
        assert not set(kw) & {"M", "H", "act", "dtype", "n_shared", "H_shared"}, name


def test_traffic_lookup_is_null_once_the_source_changes(tmp_path, monkeypatch):
    import hashlib
    files = "gemm_tcgen05.cu+sm100_ptx.cuh"
    h = hashlib.sha1()
    for name in files.split("+"):
        with open(os.path.join(ROOT, "top_gating_expert_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    good = h.hexdigest()[:12]
    table = tmp_path / "traffic.md"
    table.write_text("| kernel | preset | bytes | sha | files |\n|---|---|---|---|---|\n"
                     f"| expert_up | 2 | 123456 | {good} | {files} |\n"
                     f"| expert_down | 2 | 654321 | 000000000000 | {files} |\n")
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(table))
    assert bench.traffic_for("expert_up", 2) == 123456.0
    assert bench.traffic_for("expert_down", 2) is None  # taken on another source
    assert bench.traffic_for("expert_up", 3) is None    # no row for that preset
    assert bench.traffic_for("no_such_kernel", 2) is None


def test_backward_summary_bounds():
    """bf16 backwards take the larger of their byte and flop times as their roofline; the
    fp32 path's (plain FMA on a tiny layer) reports its latency and no roofline fraction."""
    from top_gating_expert_gb300.inputs import PRESETS
    P = {"hbm": 6000.0, "tc": 2000.0, "tc_sustained": 1800.0, "source": "test"}
    b2 = bench.backward_summary(PRESETS[2], 27000, 16384, 1, 0.45, 1.4, P)
    assert b2["bound"] == "hbm" and 0 < b2["roofline_frac"] < 1
    b3 = bench.backward_summary(PRESETS[3], 16384, 8192, 1, 3.2, 9.9, P)
    assert b3["bound"] == "tensor" and 0 < b3["roofline_frac"] < 1
    b1 = bench.backward_summary(PRESETS[1], 512, 256, 1, 0.05, 0.1, P)
    assert b1["bound"] == "latency" and b1["roofline_frac"] is None
    assert b1["train_tokens_per_s"] == round(256 / 0.15e-3, 1)
