"""The range predicate of the bounds-checked build, compiled for the host with g++
and run (CPU only)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_range_predicate(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no g++")
    exe = tmp_path / "bounds_range_test"
    subprocess.run([gxx, "-std=c++17", "-O2", "-Wall", "-Werror",
                    "-I", os.path.join(ROOT, "kv_norm_rope_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "c", "bounds_range_test.cpp"), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip().endswith("OK"), out.stdout
