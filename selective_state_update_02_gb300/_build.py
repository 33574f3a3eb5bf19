"""Builds libssu.so in-tree with nvcc for sm_103a (one translation unit, one -gencode)."""

from __future__ import annotations

import os
import shutil
import subprocess
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
SOURCES = [PKG / "csrc" / "ssu.cu"]
HEADERS = [ROOT / "include" / "ssu.h"]
LIB = PKG / "libssu.so"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libssu.so")


def nvcc_command(out: Path, extra: list[str] | None = None) -> list[str]:
    return [nvcc_path(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
            "-shared", "-I", str(ROOT / "include"), *(extra or []),
            *[str(s) for s in SOURCES], "-o", str(out)]


def stale() -> bool:
    if not LIB.exists():
        return True
    built = LIB.stat().st_mtime
    return any(p.stat().st_mtime > built for p in SOURCES + HEADERS)


def build(force: bool = False, extra: list[str] | None = None) -> Path:
    """Compile libssu.so next to this file unless it is up to date."""
    if force or stale():
        tmp = LIB.with_name(f"libssu.so.tmp{os.getpid()}")
        subprocess.run(nvcc_command(tmp, extra), check=True)
        os.replace(tmp, LIB)
    return LIB
