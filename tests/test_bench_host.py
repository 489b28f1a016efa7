"""bench.py's host logic (no GPU): the per-launch DRAM traffic it reports comes
from the committed capture only while the kernel sources still hash to the
captured tree, and the clock record's reasons are read as nvidia-smi prints them."""
import json
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _bench(monkeypatch, root):
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    import bench

    monkeypatch.setattr(bench, "ROOT", root)
    return bench


def _tree(tmp_path):
    """A copy of the kernel sources and an empty profiles folder."""
    csrc = tmp_path / "bwd_gn3d_stats_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in os.listdir(os.path.join(ROOT, "bwd_gn3d_stats_gb300", "csrc")):
        if f.endswith((".cuh", ".cu")):
            shutil.copy(os.path.join(ROOT, "bwd_gn3d_stats_gb300", "csrc", f), csrc / f)
    (tmp_path / "profiles").mkdir()
    return str(tmp_path)


def test_traffic_only_for_the_captured_sources(tmp_path, monkeypatch):
    root = _tree(tmp_path)
    bench = _bench(monkeypatch, root)
    assert bench.traffic_for("k_bwd_reduce", "w") is None  # no capture at all
    sha = bench.source_sha()
    entry = {"dram_bytes_per_launch": 123, "source_sha": sha, "sources": bench.KERNEL_SOURCES}
    with open(os.path.join(root, "profiles", "traffic.json"), "w") as f:
        json.dump({"k_bwd_reduce": {"w": entry}}, f)
    assert bench.traffic_for("k_bwd_reduce", "w") == 123
    assert bench.traffic_for("k_bwd_reduce", "other") is None
    assert bench.traffic_for("k_bwd_dx", "w") is None
    # a kernel source edited after the capture: the figure no longer applies
    p = os.path.join(root, "bwd_gn3d_stats_gb300", "csrc", "gn3d_kernels.cuh")
    with open(p, "a") as f:
        f.write("\n// edited\n")
    assert bench.source_sha() != sha
    assert bench.traffic_for("k_bwd_reduce", "w") is None


def test_committed_traffic_entries_are_complete(monkeypatch):
    """Every committed per-launch figure has its bytes, the sources it was taken
    on and the capture it came from."""
    bench = _bench(monkeypatch, ROOT)
    d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for kernel, by_workload in d.items():
        assert kernel in bench.KERNEL_TENSORS
        for workload, e in by_workload.items():
            assert e["dram_bytes_per_launch"] > 0 and e["sources"] and e["from"] and len(e["source_sha"]) == 16


def test_clock_reasons_parsed(tmp_path, monkeypatch):
    bench = _bench(monkeypatch, ROOT)
    cs = bench.ClockSampler(0)
    cs.path = str(tmp_path / "clocks.csv")
    with open(cs.path, "w") as f:
        f.write("0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active\n")
        f.write("0, 2070, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active\n")
        f.write("0, 345, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")  # idle sample
    s = cs.summary()
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]
