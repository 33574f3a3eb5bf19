"""The 920-point sweep: heads {8, 16, 32, 64, 128} x batch 1..64 then every 8 up to 1024.

This is the grid of the bitwise check in sglang PR #41223 (Correctness Verification, last
row; Details / Kernel measurement).  At each point:

* the default launch shape and an alternative one run on two copies of the same pool and
  must agree bit for bit (state and output, every request), as the page's launch configs do;
* every request is compared with the oracle where the point holds at most 2048 (request,
  head) units (every batch at 8 heads up to 256, at 128 heads up to 16), and beyond that a
  random 2048 units' worth of requests (always the first and the last): 1.54 million of the
  sweep's 16.8 million units, the rest covered by the bit-for-bit agreement above;
* the 16 slots no request names stay bit-identical.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import selective_state_update_02_gb300 as ssu
import workloads as wl
from parity_util import bf16_tensor, bits_of, compare_every_request

pytestmark = pytest.mark.gpu

HEADS = [8, 16, 32, 64, 128]
BATCHES = list(range(1, 65)) + list(range(72, 1025, 8))
GUARD = 16
UNITS_PER_POINT = 2048  # (request, head) units compared with the oracle at each point
ALT_SHAPES = [(ssu.SSU_MODE_VEC, 16, 4, 0), (ssu.SSU_MODE_VEC, 4, 4, 0),
              (ssu.SSU_MODE_VEC, 4, 1, 0), (ssu.SSU_MODE_VEC, 2, 2, 0),
              (ssu.SSU_MODE_VEC, 1, 16, 0), (ssu.SSU_MODE_VEC, 16, 2, 0),
              (ssu.SSU_MODE_VEC, 8, 2, 0), (ssu.SSU_MODE_VEC, 2, 8, 0)]


def test_grid_has_920_points():
    assert len(HEADS) * len(BATCHES) == 920


@pytest.mark.parametrize("H", HEADS)
def test_sweep(H):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    op = ssu.SelectiveStateUpdate(0)
    alt = ssu.SelectiveStateUpdate(0)
    try:
        rng = np.random.default_rng(1000 + H)
        max_slots = BATCHES[-1] + GUARD
        master_host = wl.state_pool(rng, max_slots, H)
        master = torch.from_numpy(master_host).to("cuda")
        dt_bias, A, D = wl.head_params(rng, H)
        bias_d, A_d, D_d = (torch.from_numpy(v).cuda() for v in (dt_bias, A, D))
        worst_ulp = 0
        checked = 0
        for i, bs in enumerate(BATCHES):
            n = bs + GUARD
            idx = rng.permutation(n)[:bs].astype(np.int64)
            x, dt, B, C = wl.request_inputs(rng, bs, H)
            xd, dtd, Bd, Cd = (bf16_tensor(v, "cuda") for v in (x, dt, B, C))
            idx_d = torch.from_numpy(idx).to(torch.int32).cuda()
            pa = master[:n].clone()
            pb = master[:n].clone()
            oa = torch.zeros(bs, H, 64, dtype=torch.bfloat16, device="cuda")
            ob = torch.zeros_like(oa)
            shape = ALT_SHAPES[i % len(ALT_SHAPES)]
            alt.set_launch(*shape)
            op(pa, idx_d, xd, dtd, bias_d, A_d, Bd, Cd, D_d, oa)
            alt(pb, idx_d, xd, dtd, bias_d, A_d, Bd, Cd, D_d, ob)
            assert torch.equal(pa, pb), (H, bs, shape)
            assert torch.equal(oa.view(torch.int16), ob.view(torch.int16)), (H, bs, shape)
            untouched = np.setdiff1d(np.arange(n), idx)
            ut = torch.from_numpy(untouched).cuda()
            assert torch.equal(pa[ut], master[:n][ut]), (H, bs)
            if bs * H <= UNITS_PER_POINT:
                rows = np.arange(bs)
            else:
                k = max(2, UNITS_PER_POINT // H)
                rows = np.unique(np.concatenate([[0, bs - 1],
                                                 rng.choice(bs, size=k - 2, replace=False)]))
            st = compare_every_request(master_host, idx, x, dt, dt_bias, A, B, C, D, pa,
                                       bits_of(oa), rows=rows, chunk=max(1, 1024 // H))
            worst_ulp = max(worst_ulp, st["max_ulp"])
            checked += len(rows) * H
        assert op.get_error() == (0, -1) and alt.get_error() == (0, -1)
        print(f"sweep H={H}: {checked} (request, head) units against the oracle, worst "
              f"readout {worst_ulp} bf16 steps")
    finally:
        op.close()
        alt.close()
