"""The 920-point sweep: heads {8, 16, 32, 64, 128} x batch 1..64 then every 8 up to 1024.

This is the grid of the bitwise check in sglang PR #41223 (Correctness Verification, last
row; Details / Kernel measurement).  At each point:

* the default launch shape and an alternative one run on two copies of the same pool and
  must agree bit for bit (state and output), as the page's launch configs do;
* sampled requests (first, last and one at random) are compared with the oracle;
* the 16 slots no request names stay bit-identical.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import selective_state_update_02_gb300 as ssu
import workloads as wl
from parity_util import bf16_tensor, bits_of, check_state, check_y, expected_terms, \
    oracle_on_requests

pytestmark = pytest.mark.gpu

HEADS = [8, 16, 32, 64, 128]
BATCHES = list(range(1, 65)) + list(range(72, 1025, 8))
GUARD = 16
ALT_SHAPES = [(ssu.SSU_MODE_VEC, 16, 4, 0), (ssu.SSU_MODE_BULK, 8, 4, 4),
              (ssu.SSU_MODE_VEC, 4, 1, 0), (ssu.SSU_MODE_BULK, 4, 2, 3),
              (ssu.SSU_MODE_VEC, 1, 16, 0), (ssu.SSU_MODE_BULK, 16, 4, 2),
              (ssu.SSU_MODE_VEC, 8, 2, 0), (ssu.SSU_MODE_BULK, 2, 8, 5)]


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
            rows = np.unique([0, bs - 1, int(rng.integers(bs))])
            ref_states, ref_y = oracle_on_requests(master_host, idx, rows, x, dt, dt_bias, A, B,
                                                   C, D)
            got = pa[torch.from_numpy(idx[rows]).cuda()].cpu().numpy()
            check_state(got, ref_states, f"state H={H} bs={bs}")
            Ch, Dx = expected_terms(x[rows], D, C[rows], 1, H)
            st = check_y(bits_of(oa)[rows], ref_y, ref_states, Ch, Dx, 128, f"y H={H} bs={bs}")
            worst_ulp = max(worst_ulp, st["max_ulp"])
        assert op.get_error() == (0, -1) and alt.get_error() == (0, -1)
    finally:
        op.close()
        alt.close()
