"""GPU parity for the other dstate buckets (64, 256) and for a bf16 state pool, against the
double-precision oracle: single step, every VEC launch shape bit for bit, the multi-token
step, skipped requests, and a sampled serving-size batch."""

from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
import selective_state_update_02_gb300 as ssu
import workloads as wl
from parity_util import (bf16_tensor, bits_of, check_state, check_y, expected_terms,
                         oracle_on_requests, pool_host, pool_tensor, to_device, widen)

pytestmark = pytest.mark.gpu

COMBOS = [(64, "f32"), (256, "f32"), (64, "bf16"), (128, "bf16"), (256, "bf16")]


@pytest.fixture(scope="module")
def op():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    o = ssu.SelectiveStateUpdate(0)
    yield o
    o.close()


def _run(op, t):
    op(t["state_pool"], t["state_batch_indices"], t["x"], t["dt"], t["dt_bias"], t["A"], t["B"],
       t["C"], t["D"], t["out"])


def _compare_all(pr, t, idx=None):
    idx = pr.idx if idx is None else idx
    ok = (idx >= 0) & (idx < pr.pool_size)
    rows = np.nonzero(ok)[0]
    ref_states, ref_y = oracle_on_requests(pr.pool, idx, rows, pr.x, pr.dt, pr.dt_bias, pr.A,
                                           pr.B, pr.C, pr.D, pr.ngroups)
    got = pool_host(t["state_pool"])
    check_state(got[idx[rows]], ref_states)
    Ch, Dx = expected_terms(pr.x[rows], pr.D, pr.C[rows], pr.ngroups, pr.nheads)
    check_y(bits_of(t["out"])[rows], ref_y, ref_states, Ch, Dx, pr.pool.shape[-1])
    untouched = np.setdiff1d(np.arange(pr.pool_size), idx[rows])
    assert np.array_equal(got[untouched], pr.pool[untouched])


@pytest.mark.parametrize("N,dtype", COMBOS)
@pytest.mark.parametrize("P", [64, 40, 3])
def test_single_step(op, N, dtype, P):
    pr = wl.make_problem(9, 8, P=P, N=N, G=2, pool_size=20, seed=N + P, state_dtype=dtype)
    t = to_device(pr)
    _run(op, t)
    assert op.get_error() == (0, -1)
    _compare_all(pr, t)


def rows_per_instruction(N: int, dtype: str) -> int:
    """Rows one warp-wide 16-byte vector instruction covers: 512 bytes of state."""
    return max(1, 512 // (N * (2 if dtype == "bf16" else 4)))


@pytest.mark.parametrize("N,dtype", COMBOS)
def test_every_vec_shape_is_bitwise_identical(op, N, dtype):
    pr = wl.make_problem(6, 16, P=40, N=N, pool_size=14, seed=7, state_dtype=dtype)
    ref = to_device(pr)
    _run(op, ref)
    _compare_all(pr, ref)
    rpi = rows_per_instruction(N, dtype)
    try:
        for rpw in (rpi, 2 * rpi, 4 * rpi, 8 * rpi):
            for wpc in (1, 2, 3, 4, 8):
                t = to_device(pr)
                op.set_launch(ssu.SSU_MODE_VEC, rpw, wpc)
                _run(op, t)
                assert torch.equal(t["state_pool"].view(torch.int16) if dtype == "bf16"
                                   else t["state_pool"],
                                   ref["state_pool"].view(torch.int16) if dtype == "bf16"
                                   else ref["state_pool"]), (rpw, wpc)
                assert torch.equal(t["out"].view(torch.int16), ref["out"].view(torch.int16))
    finally:
        op.set_launch(ssu.SSU_MODE_AUTO)


@pytest.mark.parametrize("N,dtype", COMBOS)
def test_rows_per_warp_outside_the_bucket_are_refused(op, N, dtype):
    # A warp's rows come in whole vector instructions (rows_per_instruction of them) and at
    # most 8 instructions per warp (16 rows only for an fp32 state of dstate 128).
    pr = wl.make_problem(4, 8, N=N, pool_size=8, seed=2, state_dtype=dtype)
    t = to_device(pr)
    rpi = rows_per_instruction(N, dtype)
    bad = [16 * rpi] + ([rpi // 2] if rpi > 1 else [])
    for rpw in bad:
        try:
            # refused when set (more than 32 rows per warp) or at the call (not a shape of
            # this bucket)
            with pytest.raises(ssu.SsuError) as e:
                op.set_launch(ssu.SSU_MODE_VEC, rpw, 2)
                _run(op, t)
            assert e.value.status == ssu.SSU_ERR_UNSUPPORTED
        finally:
            op.set_launch(ssu.SSU_MODE_AUTO)


@pytest.mark.parametrize("N,dtype", COMBOS + [(128, "f32")])
def test_every_token_shape_is_bitwise_identical(op, N, dtype):
    # The general multi-token kernel's tiles (rows per warp, warps per CTA) change which warp
    # updates which rows, never the arithmetic: every shape gives the same bits.
    bs, T, H, P = 9, 3, 8, 40
    pr = wl.make_problem(bs, H, P=P, N=N, pool_size=12, seed=19, state_dtype=dtype)
    rng = np.random.default_rng(20)
    steps = [wl.request_inputs(rng, bs, H, P, N) for _ in range(T)]
    x, dt, B, C = (bf16_tensor(np.stack([s[k] for s in steps], 1), "cuda") for k in range(4))

    def run():
        dev = to_device(pr)
        out = torch.zeros(bs, T, H, P, dtype=torch.bfloat16, device="cuda")
        op.tokens(dev["state_pool"], dev["state_batch_indices"], x, dt, dev["dt_bias"],
                  dev["A"], B, C, dev["D"], out)
        torch.cuda.synchronize()
        return dev["state_pool"].view(torch.int16).clone() if dtype == "bf16" else \
            dev["state_pool"].clone(), out.view(torch.int16).clone()

    rpi = rows_per_instruction(N, dtype)
    nc = 8 if (dtype == "bf16" or N == 256) else 4
    try:
        # the reference: one slot per lane, one warp per CTA (a forced shape runs the general
        # kernel; without one, dstate 64 and 128 run the chunked kernel, which sums otherwise)
        op.set_launch(ssu.SSU_MODE_VEC, rpi, 1)
        ref_pool, ref_out = run()
        for slots in (1, 2, 4, 8):
            if slots * nc > 32:
                continue
            for wpc in (1, 2, 4):
                op.set_launch(ssu.SSU_MODE_VEC, slots * rpi, wpc)
                got_pool, got_out = run()
                assert torch.equal(got_pool, ref_pool), (slots * rpi, wpc)
                assert torch.equal(got_out, ref_out), (slots * rpi, wpc)
    finally:
        op.set_launch(ssu.SSU_MODE_AUTO)
    assert op.get_error() == (0, -1)


@pytest.mark.parametrize("N,dtype", COMBOS)
def test_skipped_requests(op, N, dtype):
    pr = wl.make_problem(8, 8, N=N, pool_size=10, seed=3, state_dtype=dtype)
    idx = pr.idx.copy()
    idx[[1, 5]] = [10, -1]
    t = to_device(pr)
    t["state_batch_indices"] = torch.from_numpy(idx).to(torch.int32).cuda()
    _run(op, t)
    assert op.get_error() == (2, 1)
    _compare_all(pr, t, idx)


@pytest.mark.parametrize("N,dtype", COMBOS + [(128, "f32")])
@pytest.mark.parametrize("with_inter,T", [(True, 5), (False, 5), (False, 16)],
                         ids=["inter", "no_inter", "no_inter-16"])
def test_tokens(op, N, dtype, with_inter, T):
    # with intermediate states the general kernel runs; without them, the chunked kernel for
    # an fp32 state from 5 tokens and a bf16 state of dstate 128 from 16
    bs, H, P = 7, 8, 40
    pr = wl.make_problem(bs, H, P=P, N=N, pool_size=12, seed=11, state_dtype=dtype)
    rng = np.random.default_rng(12)
    steps = [wl.request_inputs(rng, bs, H, P, N) for _ in range(T)]
    x, dt, B, C = (np.stack([s[k] for s in steps], 1) for k in range(4))
    dev = to_device(pr)
    out = torch.zeros(bs, T, H, P, dtype=torch.bfloat16, device="cuda")
    inter = (torch.zeros(bs, T, H, P, N, dtype=dev["state_pool"].dtype, device="cuda")
             if with_inter else None)
    op.tokens(dev["state_pool"], dev["state_batch_indices"], bf16_tensor(x, "cuda"),
              bf16_tensor(dt, "cuda"), dev["dt_bias"], dev["A"], bf16_tensor(B, "cuda"),
              bf16_tensor(C, "cuda"), dev["D"], out, inter)
    torch.cuda.synchronize()
    ref_pool, ref_y, ref_inter, _ = oracle.ssu_tokens(widen(pr.pool), pr.idx, x, dt, pr.dt_bias,
                                                     pr.A, B, C, pr.D)
    got = pool_host(dev["state_pool"])
    check_state(got[pr.idx], ref_pool[pr.idx])
    got_inter = (pool_host(inter.view(bs, T * H, P, N)).reshape(bs, T, H, P, N)
                 if with_inter else None)
    outb = bits_of(out)
    for t in range(T):
        if with_inter:
            check_state(got_inter[:, t], ref_inter[:, t], f"intermediate {t}")
        Ch, Dx = expected_terms(x[:, t], pr.D, C[:, t], 1, H)
        check_y(outb[:, t], ref_y[:, t], ref_inter[:, t], Ch, Dx, N, f"y token {t}")


@pytest.mark.parametrize("N,dtype", [(128, "bf16"), (64, "f32"), (256, "f32"), (256, "bf16"),
                                     (64, "bf16")])
def test_serving_batch_128_sampled(op, N, dtype):
    """Each bucket at the batch the bench times it (128 requests, 16 heads, the built-in
    launch table), slots scattered over a 384-slot pool; every request against the oracle,
    every other slot unchanged."""
    bs, H, slots = 128, 16, 384
    rng = np.random.default_rng(5 + N)
    pool = wl.state_pool(rng, slots, H, N=N, dtype=dtype)
    idx = wl.rotation_sets(bs, 3, seed=5)[1]
    dt_bias, A, D = wl.head_params(rng, H)
    x, dt, B, C = wl.request_inputs(rng, bs, H, N=N)
    pool_d = pool_tensor(pool, "cuda")
    out = torch.zeros(bs, H, 64, dtype=torch.bfloat16, device="cuda")
    op(pool_d, torch.from_numpy(idx).cuda(), bf16_tensor(x, "cuda"), bf16_tensor(dt, "cuda"),
       torch.from_numpy(dt_bias).cuda(), torch.from_numpy(A).cuda(), bf16_tensor(B, "cuda"),
       bf16_tensor(C, "cuda"), torch.from_numpy(D).cuda(), out)
    torch.cuda.synchronize()
    rows = np.arange(bs)  # every request against the oracle
    ref_states, ref_y = oracle_on_requests(pool, idx, rows, x, dt, dt_bias, A, B, C, D,
                                           threads=os.cpu_count() or 1)
    got = pool_host(pool_d)
    check_state(got[idx[rows]], ref_states)
    Ch, Dx = expected_terms(x[rows], D, C[rows], 1, H)
    check_y(bits_of(out)[rows], ref_y, ref_states, Ch, Dx, N)
    mask = np.ones(slots, bool)
    mask[idx] = False
    assert np.array_equal(got[mask], pool[mask])


@pytest.mark.parametrize("N,dtype", COMBOS)
def test_one_token_kernel_equals_ssu_update_bitwise(op, N, dtype):
    """T = 1 with an intermediate buffer runs the multi-token kernel; it gives the bits of
    ssu_update in every bucket (one element mapping, one summation order)."""
    bs, H, P = 11, 8, 40
    pr = wl.make_problem(bs, H, P=P, N=N, pool_size=15, seed=23, state_dtype=dtype)
    a, b = to_device(pr), to_device(pr)
    _run(op, a)
    out = torch.zeros(bs, 1, H, P, dtype=torch.bfloat16, device="cuda")
    inter = torch.zeros(bs, 1, H, P, N, dtype=b["state_pool"].dtype, device="cuda")
    op.tokens(b["state_pool"], b["state_batch_indices"], b["x"].unsqueeze(1),
              b["dt"].unsqueeze(1), b["dt_bias"], b["A"], b["B"].unsqueeze(1),
              b["C"].unsqueeze(1), b["D"], out, inter)
    torch.cuda.synchronize()
    as_bits = (lambda t: t.view(torch.int16)) if dtype == "bf16" else (lambda t: t)
    assert torch.equal(as_bits(a["state_pool"]), as_bits(b["state_pool"]))
    assert torch.equal(a["out"].view(torch.int16), out[:, 0].view(torch.int16))
    idx = torch.from_numpy(pr.idx).cuda()
    assert torch.equal(as_bits(inter[:, 0]), as_bits(b["state_pool"][idx]))
