"""Register use of the kernels the launch tables pick, from ptxas's own report (no GPU).

The decode-step kernel's residency (32 warps per SM at 64 registers for 8 rows per warp,
fp32, dstate 128) and the multi-token kernel's 128-register cap (16 warps per SM) are what
their measured times rest on; a change that spills or grows past those counts fails here
before it reaches a GPU.  ptxas prints, per kernel, "Used N registers" and the spill bytes;
nothing of the compiled code itself is read.
"""

from __future__ import annotations

import re
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
CSRC = ROOT / "selective_state_update_02_gb300" / "csrc"

# (rows per warp, dstate, state type) -> most registers it may use: the shapes the built-in
# tables pick for a small and a large call.
VEC_TABLE = {
    (8, 128, "f32"): 64,    # batch >= 16: 32 warps per SM
    (2, 128, "f32"): 64,    # batch 8
    (4, 256, "f32"): 72,
    (2, 256, "f32"): 64,
    (16, 64, "f32"): 64,    # 8 vector rows of 2 rows each
    (8, 64, "f32"): 64,
    (16, 128, "bf16"): 96,
    (8, 128, "bf16"): 72,
    (32, 64, "bf16"): 96,
    (16, 64, "bf16"): 72,
    (8, 64, "bf16"): 64,
    (8, 256, "bf16"): 96,
    (2, 256, "bf16"): 64,
}
TOKENS_TABLE = {           # the multi-token table's tiles: (cap, spill bytes allowed)
    (8, 128, "f32"): (96, 8),     # 32 fp32 values per lane, 20 warps per SM
    (16, 64, "f32"): (96, 40),
    (4, 256, "f32"): (96, 0),
    (32, 64, "bf16"): (128, 0),   # 64 values per lane
    (16, 128, "bf16"): (128, 0),
    (8, 256, "bf16"): (128, 0),
}

# The chunked multi-token kernel (dstate -> (cap, spill bytes allowed)): 4 CTAs of 4 warps per
# SM at 128 registers; the state takes 64 of them at dstate 128.
MMA_TABLE = {
    (128, "f32"): (128, 0),
    (128, "bf16"): (128, 8),
    (64, "f32"): (128, 0),
}


def _ptxas_report(tmp_path: Path, unit: str) -> dict:
    from selective_state_update_02_gb300 import _build
    out = subprocess.run(
        [_build.nvcc_path(), *_build.ARCH, "-O3", "-std=c++17", "-I", str(ROOT / "include"),
         "-I", str(CSRC), "-Xptxas", "-v", "-cubin", "-c", str(CSRC / unit), "-o",
         str(tmp_path / (unit + ".cubin"))],
        capture_output=True, text=True, timeout=600, check=True).stderr
    kernels = {}
    for block in out.split("ptxas info    : Compiling entry function '")[1:]:
        name = block.split("'")[0]
        m = re.search(r"(ssu_vec_kernel|ssu_tokens_kernel)(?:_capped)?ILi(\d+)ELi(\d+)E(\w+?)"
                      r"Lb([01])E", name)
        mm = re.search(r"ssu_tokens_mma_kernelILi(\d+)E(\w+?)Lb([01])E", name)
        regs = re.search(r"Used (\d+) registers", block)
        spill = re.search(r"(\d+) bytes spill stores", block)
        if m and regs and spill:
            st = "bf16" if "nv_bfloat16" in m.group(4) else "f32"
            key = (m.group(1), int(m.group(2)), int(m.group(3)), st, m.group(5) == "1")
            kernels[key] = (int(regs.group(1)), int(spill.group(1)))
        elif mm and regs and spill:
            st = "bf16" if "nv_bfloat16" in mm.group(2) else "f32"
            key = ("ssu_tokens_mma_kernel", int(mm.group(1)), st, mm.group(3) == "1")
            kernels[key] = (int(regs.group(1)), int(spill.group(1)))
    return kernels


@pytest.mark.parametrize("unit,kernel,table", [
    ("ssu.cu", "ssu_vec_kernel", VEC_TABLE),
    ("ssu_tokens.cu", "ssu_tokens_kernel", TOKENS_TABLE),
])
def test_table_kernels_fit_their_registers(tmp_path, unit, kernel, table):
    report = _ptxas_report(tmp_path, unit)
    for (rpw, n, st), budget in table.items():
        cap, spill_ok = budget if isinstance(budget, tuple) else (budget, 0)
        for i64 in (False, True):
            key = (kernel, rpw, n, st, i64)
            assert key in report, f"{key} not compiled"
            regs, spill = report[key]
            assert spill <= spill_ok, f"{key} spills {spill} bytes (at most {spill_ok})"
            assert regs <= cap, f"{key} uses {regs} registers (at most {cap})"


def test_chunked_token_kernel_fits_its_registers(tmp_path):
    report = _ptxas_report(tmp_path, "ssu_tokens.cu")
    for (n, st), (cap, spill_ok) in MMA_TABLE.items():
        for i64 in (False, True):
            key = ("ssu_tokens_mma_kernel", n, st, i64)
            assert key in report, f"{key} not compiled"
            regs, spill = report[key]
            assert spill <= spill_ok, f"{key} spills {spill} bytes (at most {spill_ok})"
            assert regs <= cap, f"{key} uses {regs} registers (at most {cap})"
