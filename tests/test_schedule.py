"""The GEMM kernels' work schedule (bit_gemm_gb300/csrc/mx_schedule.h), checked
on the host: the header is host-compilable, and tests/schedule_check.cpp walks
every worker's units for a set of shapes (whole tiles, slices of (tile, K
stage), and whole tiles with the last partial round in slices)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "bit_gemm_gb300", "csrc")


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_schedule_covers_every_unit_once(tmp_path):
    exe = str(tmp_path / "schedule_check")
    subprocess.run(["g++", "-std=c++17", "-O2", "-Wall", "-Werror", "-I", CSRC,
                    os.path.join(HERE, "schedule_check.cpp"), "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
