"""The allocation-free entry point, ssu_update_static, against ssu_update.

ssu_update_static is for callers that cannot allocate device memory (for example code running
under an allocator that must not be re-entered, or a runtime that only hands out memory it
owns), so they cannot create a handle.  Its kernel keeps its skipped-request counters in a
fixed array inside the library instead.  This file is collected last on purpose: if it fails,
a run that stops at the first failure has already run every other test.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import selective_state_update_02_gb300 as ssu
import workloads as wl
from parity_util import STATE_RTOL, bf16_tensor, ordered_bf16, to_device

pytestmark = pytest.mark.gpu


def _close(a_state, b_state, a_out, b_out):
    """The tolerance the parity tests use: state within 1e-5 (1 + |ref|), out within 2 bf16 ulp."""
    ref = b_state.double()
    err = ((a_state.double() - ref).abs() / (1.0 + ref.abs())).max().item()
    assert err <= STATE_RTOL, err
    ua = ordered_bf16(a_out.view(torch.int16).cpu().numpy().view(np.uint16))
    ub = ordered_bf16(b_out.view(torch.int16).cpu().numpy().view(np.uint16))
    assert np.abs(ua - ub).max() <= 2


def test_static_entry_point_matches_ssu_update_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    bs, H, pool_size = 48, 16, 64
    pr = wl.make_problem(bs, H, pool_size=pool_size, seed=31)
    idx = pr.idx.copy()
    idx[[4, 17]] = [pool_size, -2]            # two requests name no slot: skipped, counted
    ref = to_device(pr, "cuda")               # the handle-based entry point runs here
    new = to_device(pr, "cuda")               # the allocation-free one runs here
    for t in (ref, new):
        t["state_batch_indices"] = torch.from_numpy(idx).to(torch.int32).cuda()
    counters = torch.full((3,), -7, dtype=torch.int32, device="cuda")
    op = ssu.SelectiveStateUpdate(0)
    rng = np.random.default_rng(99)
    try:
        for step in range(2):
            if step:
                x, dt, B, C = wl.request_inputs(rng, bs, H)
                for t in (ref, new):
                    t["x"], t["dt"] = bf16_tensor(x, "cuda"), bf16_tensor(dt, "cuda")
                    t["B"], t["C"] = bf16_tensor(B, "cuda"), bf16_tensor(C, "cuda")
            op(ref["state_pool"], ref["state_batch_indices"], ref["x"], ref["dt"],
               ref["dt_bias"], ref["A"], ref["B"], ref["C"], ref["D"], ref["out"])
            ssu.ssu_update_static(new["state_pool"], new["state_batch_indices"], new["x"],
                                  new["dt"], new["dt_bias"], new["A"], new["B"], new["C"],
                                  new["D"], new["out"], counters_out=counters)
            torch.cuda.synchronize()
            _close(new["state_pool"], ref["state_pool"], new["out"], ref["out"])
            assert op.get_error() == (2, 4)
            got = counters.cpu().numpy().view(np.uint32).tolist()
            assert got == [2, 4, 0], got       # cleared at the start of every call
    finally:
        op.close()


def test_static_entry_point_rejects_batches_beyond_its_maximum():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    shape = ssu.ssu_shape_t(ssu.SSU_STATIC_MAX_BATCH + 1, 16, 64, 128, 1, 8, 0, 0)
    strides = ssu.ssu_strides_t()
    fake = [1 << 32] * 10                     # never dereferenced: rejected on the host
    st = ssu.lib().ssu_update_static(*fake, shape, strides, None, None)
    assert st == ssu.SSU_ERR_UNSUPPORTED
    assert "SSU_STATIC_MAX_BATCH" in ssu.last_error()
