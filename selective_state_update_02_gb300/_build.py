"""Builds libssu.so in-tree with nvcc for sm_103a (one -gencode; the translation units are
compiled in parallel, then linked into one shared library)."""

from __future__ import annotations

import os
import shutil
import subprocess
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
SOURCES = [CSRC / "ssu.cu", CSRC / "ssu_tokens.cu", CSRC / "ssu_copy.cu",
           CSRC / "ssu_host.cpp"]
HEADERS = [ROOT / "include" / "ssu.h", CSRC / "ssu_device.cuh", CSRC / "ssu_host.h",
           CSRC / "ssu_vec.cuh", CSRC / "ssu_stage.cuh",
           CSRC / "ssu_tokens.cuh", CSRC / "ssu_tokens_mma.cuh"]
OBJDIR = PKG / "_build"
LIB = PKG / "libssu.so"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libssu.so")


def compile_command(src: Path, obj: Path, extra: list[str] | None = None) -> list[str]:
    return [nvcc_path(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
            "-I", str(ROOT / "include"), "-I", str(CSRC), *(extra or []), "-c", str(src),
            "-o", str(obj)]


def link_command(objs: list[Path], out: Path) -> list[str]:
    return [nvcc_path(), *ARCH, "-shared", *[str(o) for o in objs], "-o", str(out)]


def stale() -> bool:
    if not LIB.exists():
        return True
    built = LIB.stat().st_mtime
    return any(p.stat().st_mtime > built for p in SOURCES + HEADERS)


def build(force: bool = False, extra: list[str] | None = None) -> Path:
    """Compile libssu.so next to this file unless it is up to date."""
    if not (force or stale()):
        return LIB
    OBJDIR.mkdir(exist_ok=True)
    objs = [OBJDIR / (src.name + ".o") for src in SOURCES]
    procs = [subprocess.Popen(compile_command(src, obj, extra))
             for src, obj in zip(SOURCES, objs)]
    codes = [p.wait() for p in procs]
    if any(codes):
        raise subprocess.CalledProcessError(max(codes), "nvcc (libssu sources)")
    tmp = LIB.with_name(f"libssu.so.tmp{os.getpid()}")
    subprocess.run(link_command(objs, tmp), check=True)
    os.replace(tmp, LIB)
    return LIB
