"""Host logic: the launch plans' index arithmetic, replayed on the CPU.

tests/plan_walk.cpp includes the real plan headers (csrc/gn3d_plan.cuh and
csrc/gn3d_ndhwc_plan.cuh, host-compilable) and walks, for a few thousand
shapes, every vector and scalar the kernels read, every workspace entry they
write and read, the channels-last rings' bulk-copy parts, and the NCDHW
streaming kernels' work shares in both layouts (strided blocks, unit shares
with cut blocks); it fails on the first element read twice or never, any
access outside its tensor, unit, range or slot, or a merge block completed
other than exactly once."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_plans_cover_every_element_once(tmp_path):
    exe = tmp_path / "plan_walk"
    subprocess.run(["g++", "-O2", "-std=c++17", "-o", str(exe), os.path.join(HERE, "plan_walk.cpp")], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.startswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]
