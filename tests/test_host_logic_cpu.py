"""Host logic checked without a GPU.  tests/c/stage_jobs.cu expands 20,000
random operand geometries with the staging kernel's own address arithmetic and checks that
every source byte lands once, in dense order, with aligned vectors."""

from __future__ import annotations

import shutil
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent


def test_stage_jobs_cover_each_byte_once(tmp_path):
    from selective_state_update_02_gb300 import _build
    nvcc = _build.nvcc_path()
    if shutil.which(nvcc) is None and not Path(nvcc).exists():
        pytest.skip("nvcc not available")
    exe = tmp_path / "stage_jobs"
    subprocess.run([nvcc, *_build.ARCH, "-O1", "-std=c++17",
                    "-I", str(ROOT / "selective_state_update_02_gb300" / "csrc"),
                    str(ROOT / "tests" / "c" / "stage_jobs.cu"), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


def test_group_index_without_division(tmp_path):
    """group_of(h, group_magic(d)) == h // d for every d < 2^16 at and around every multiple
    of d (tests/c/group_magic.cu)."""
    from selective_state_update_02_gb300 import _build
    nvcc = _build.nvcc_path()
    exe = tmp_path / "group_magic"
    subprocess.run([nvcc, *_build.ARCH, "-O2", "-std=c++17",
                    "-I", str(ROOT / "selective_state_update_02_gb300" / "csrc"),
                    str(ROOT / "tests" / "c" / "group_magic.cu"), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr

