"""Register use of the kernels the launch tables pick, from ptxas's own report (no GPU).

The decode-step kernel's residency (32 warps per SM at 64 registers for 8 rows per warp,
fp32, dstate 128) and the multi-token kernel's 96-register cap (20 warps per SM) are what
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

# (kernel, rows per warp, columns per lane, state type) -> most registers it may use.
VEC_TABLE = {
    (8, 4, "f32"): 64,   # dstate 128, batch >= 32: 32 warps per SM
    (2, 4, "f32"): 64,   # dstate 128, batch 8
    (4, 8, "f32"): 128,  # dstate 256
    (8, 2, "f32"): 128,  # dstate 64
    (8, 4, "bf16"): 128,
    (8, 8, "bf16"): 128,
    (8, 2, "bf16"): 128,
}
TOKENS_TABLE = {
    (8, 4, "f32"): 96,   # the table's shape up to dstate 128: 20 warps per SM
    (8, 4, "bf16"): 96,
    (8, 2, "f32"): 96,
    (8, 2, "bf16"): 96,
    (4, 8, "f32"): 128,  # dstate 256
    (4, 8, "bf16"): 128,
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
        m = re.search(r"(ssu_vec_kernel|ssu_tokens_kernel)ILi(\d+)ELi(\d+)E(\w+?)Lb([01])E",
                      name)
        regs = re.search(r"Used (\d+) registers", block)
        spill = re.search(r"(\d+) bytes spill stores", block)
        if m and regs and spill:
            st = "bf16" if "nv_bfloat16" in m.group(4) else "f32"
            key = (m.group(1), int(m.group(2)), int(m.group(3)), st, m.group(5) == "1")
            kernels[key] = (int(regs.group(1)), int(spill.group(1)))
    return kernels


@pytest.mark.parametrize("unit,kernel,table", [
    ("ssu.cu", "ssu_vec_kernel", VEC_TABLE),
    ("ssu_tokens.cu", "ssu_tokens_kernel", TOKENS_TABLE),
])
def test_table_kernels_fit_their_registers(tmp_path, unit, kernel, table):
    report = _ptxas_report(tmp_path, unit)
    for (rpw, nc, st), cap in table.items():
        for i64 in (False, True):
            key = (kernel, rpw, nc, st, i64)
            assert key in report, f"{key} not compiled"
            regs, spill = report[key]
            assert spill == 0, f"{key} spills {spill} bytes"
            assert regs <= cap, f"{key} uses {regs} registers (at most {cap})"
