"""The README's Python example runs as written (on a GPU) and gives what the library's own
tests expect: the host-operand call reproduces the device call's readout bit for bit."""

from __future__ import annotations

import re
from pathlib import Path

import pytest
import torch

ROOT = Path(__file__).resolve().parent.parent

pytestmark = pytest.mark.gpu


def test_readme_example_runs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    code = re.findall(r"```python\n(.*?)```", (ROOT / "README.md").read_text(), re.S)[0]
    scope: dict = {}
    exec(compile(code, "README.md", "exec"), scope)
    torch.cuda.synchronize()
    assert scope["skipped"] == 0 and scope["first_bad"] == -1
    # the second call updated the same slots again from the same inputs: its readout is the
    # step applied to the already-updated state, so compare it against a device call on a copy
    import selective_state_update_02_gb300 as ssu
    op, pool = scope["op"], scope["pool"]
    before = pool.clone()
    out_dev = torch.empty_like(scope["out"])
    op(pool, scope["idx"], scope["x"], scope["dt"], scope["dt_bias"], scope["A"], scope["B"],
       scope["C"], scope["D"], out_dev)
    after_dev = pool.clone()
    pool.copy_(before)
    h = scope["h"]
    ssu.ssu_update_from_host(op.handle, pool, h["idx"], h["x"], h["dt"], scope["dt_bias"],
                             scope["A"], h["B"], h["C"], scope["D"], scope["h_out"], scope["ws"])
    torch.cuda.synchronize()
    assert torch.equal(pool, after_dev)
    assert torch.equal(scope["h_out"].view(torch.int16), out_dev.cpu().view(torch.int16))
    op.close()
