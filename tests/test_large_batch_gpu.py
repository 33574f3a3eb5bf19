"""Batches past the 65,535 CTAs the grid's third dimension holds: every per-request kernel
then loops over requests (request b, b + 65535, ...).  70,000 requests of one head (headdim
16, dstate 64, fp32 state, a pool with 16 spare slots): the single step and the multi-token
step (2 tokens: the general kernel; 5: the chunked kernel) on requests sampled at both ends
and around the 65,535 boundary against the oracle, and the spare slots left alone."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import selective_state_update_02_gb300 as ssu
import workloads as wl
from parity_util import (bf16_tensor, bits_of, check_state, check_y, compare_every_request,
                         expected_terms, to_device)

pytestmark = pytest.mark.gpu

BS, H, P, N = 70_000, 1, 16, 64
SAMPLE = np.r_[0:6, 65_530:65_542, BS - 6:BS]


@pytest.fixture(scope="module")
def op():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    o = ssu.SelectiveStateUpdate(0)
    yield o
    o.close()


def _spare_slots_untouched(pr, got_pool):
    spare = np.setdiff1d(np.arange(pr.pool.shape[0]), pr.idx)
    assert len(spare) == 16
    assert np.array_equal(got_pool[spare], pr.pool[spare])


def test_decode_step_past_the_grid_limit(op):
    pr = wl.make_problem(BS, H, P, N, pool_size=BS + 16, seed=91)
    dev = to_device(pr)
    op(**dev)
    torch.cuda.synchronize()
    assert op.get_error() == (0, -1)
    compare_every_request(pr.pool, pr.idx, pr.x, pr.dt, pr.dt_bias, pr.A, pr.B, pr.C, pr.D,
                          dev["state_pool"], bits_of(dev["out"]), rows=SAMPLE)
    _spare_slots_untouched(pr, dev["state_pool"].cpu().numpy())


@pytest.mark.parametrize("T", [2, 5])
def test_tokens_past_the_grid_limit(op, T):
    pr = wl.make_problem(BS, H, P, N, pool_size=BS + 16, seed=92 + T)
    rng = np.random.default_rng(93 + T)
    steps = [wl.request_inputs(rng, BS, H, P, N) for _ in range(T)]
    x, dt, B, C = (np.stack([s[k] for s in steps], 1) for k in range(4))
    dev = to_device(pr)
    out = torch.zeros(BS, T, H, P, dtype=torch.bfloat16, device="cuda")
    op.tokens(dev["state_pool"], dev["state_batch_indices"], bf16_tensor(x, "cuda"),
              bf16_tensor(dt, "cuda"), dev["dt_bias"], dev["A"], bf16_tensor(B, "cuda"),
              bf16_tensor(C, "cuda"), dev["D"], out)
    torch.cuda.synchronize()
    assert op.get_error() == (0, -1)
    got_pool = dev["state_pool"].cpu().numpy()
    got_out = bits_of(out)
    # the oracle on the sampled requests alone (their slots as a small pool of their own)
    ref_pool, ref_y, ref_inter, _ = oracle.ssu_tokens(
        pr.pool[pr.idx[SAMPLE]], np.arange(len(SAMPLE)), x[SAMPLE], dt[SAMPLE], pr.dt_bias,
        pr.A, B[SAMPLE], C[SAMPLE], pr.D)
    check_state(got_pool[pr.idx[SAMPLE]], ref_pool)
    for t in range(T):
        Ch, Dx = expected_terms(x[SAMPLE, t], pr.D, C[SAMPLE, t], 1, H)
        check_y(got_out[SAMPLE, t], ref_y[:, t], ref_inter[:, t], Ch, Dx, N, f"y token {t}")
    _spare_slots_untouched(pr, got_pool)
