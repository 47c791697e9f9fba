"""Host checks of the workspace layout (csrc/layout.h): the zeroed / tagged
regions of the single-launch decode sit at the same offsets for every T, every
region is aligned and inside the workspace, the launch's split factors never
exceed the ones the layout sized, the slot bound holds for random (skewed)
routings, and the 16-token shapes fit the no-alloc scratch.  The checks are a
small C++ program compiled with the host compiler."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "block_scaled_fp4_router_gb300", "csrc")


def test_workspace_layout_properties():
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "layout_check")
        r = subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, os.path.join(ROOT, "tests", "layout_check.cpp"),
                            "-o", exe], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
        r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
        assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
