"""The boundary from plain C99: tests/c/abi_step.c includes only include/ssu.h, links
libssu.so and the CUDA runtime's C API, and runs the hand-computed step (y = 2 exactly)."""

from __future__ import annotations

import shutil
import subprocess
from pathlib import Path

import pytest
import torch

ROOT = Path(__file__).resolve().parent.parent
SRC = ROOT / "tests" / "c" / "abi_step.c"
PKG = ROOT / "selective_state_update_02_gb300"
CUDA = Path("/usr/local/cuda")


def _build(tmp_path: Path) -> Path:
    from selective_state_update_02_gb300 import _build
    _build.build()
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    exe = tmp_path / "abi_step"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-O1",
                    "-I", str(ROOT / "include"), "-isystem", str(CUDA / "include"), str(SRC),
                    "-o", str(exe), "-L", str(PKG), "-l:libssu.so", "-L", str(CUDA / "lib64"),
                    "-lcudart", "-lm", f"-Wl,-rpath,{PKG}", f"-Wl,-rpath,{CUDA / 'lib64'}"],
                   check=True)
    return exe


@pytest.mark.parametrize("lang,std", [("c", "c99"), ("c", "c11"), ("c++", "c++11")])
def test_header_is_strict_c_and_cxx(lang, std):
    compiler = "gcc" if lang == "c" else "g++"
    if shutil.which(compiler) is None:
        pytest.skip(f"{compiler} not available")
    subprocess.run([compiler, "-x", lang, f"-std={std}", "-pedantic", "-Wall", "-Wextra",
                    "-Werror", "-fsyntax-only", str(ROOT / "include" / "ssu.h")], check=True)


def test_c_program_builds_and_checks_the_host_side(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() in ("ok", "no-device")


@pytest.mark.gpu
def test_c_program_runs_the_step_on_the_gpu(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = _build(tmp_path)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
