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


def test_defaults_are_one_gpu_preset_2():
    a = _args()
    assert (a.gpus, a.config, a.impl) == (1, 2, "ours")
    assert a.warmup >= 3 and a.steps >= 1


def test_override_changes_fields_and_names_them():
    cfg = bench.preset_for(_args("--override", "S=4096", "--override", "G=4", "--override", "E=32"))
    assert (cfg["S"], cfg["G"], cfg["E"]) == (4096, 4, 32)
    assert isinstance(cfg["S"], int) and "S=4096" in cfg["name"]
    assert cfg["M"] == PRESETS[2]["M"]


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
