"""A long decode: 128 consecutive steps on the same slots, new inputs each step, against the
oracle's double-precision trajectory.

A per-call tolerance does not carry over to a chain of calls: every step's fp32 rounding is
carried into the next state, scaled by that step's decay dA.  To first order the state error
obeys, per element,

    E_t = dA_t E_{t-1} + |S_{t-1}| dA_t r_dA + |dtv x B| r_k + |S_t| u,      u = 2^-24,

where the relative errors come from the fp32 arithmetic of one step: z = dt + dt_bias is
rounded once (u), softplus amplifies a relative error of z by |z| sigmoid(z) / softplus(z) and
adds its own (taken as 4u for log1pf of expf), so r_dtv = (|z| sigmoid(z)/softplus(z) + 5) u;
dA = exp(dtv A) turns the argument's relative error into |dtv A| (r_dtv + u) and adds 2u for
expf, r_dA = |dtv A| (r_dtv + u) + 2u; the input term is two more rounded products,
r_k = r_dtv + 2u; the fused multiply-add rounds once (u).  The test doubles that bound,
accumulates it along the oracle's trajectory, checks the GPU state after every 32 steps and
every readout against 2 bf16 ulp + the dot product's bound + the state bound carried through
C."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import selective_state_update_02_gb300 as ssu
import workloads as wl
from parity_util import bf16_tensor, bits_of, ordered_bf16, ulp_bf16

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


def test_128_steps_stay_within_the_accumulated_rounding_bound():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bs, H, P, N, steps = 8, 16, 64, 128, 128
    pr = wl.make_problem(bs, H, pool_size=16, seed=90)
    rng = np.random.default_rng(91)
    op = ssu.SelectiveStateUpdate(0)
    pool_d = torch.from_numpy(pr.pool).cuda()
    idx_d = torch.from_numpy(pr.idx.astype(np.int32)).cuda()
    dt_bias, A, D = (torch.from_numpy(v).cuda() for v in (pr.dt_bias, pr.A, pr.D))
    out = torch.empty(bs, H, P, dtype=torch.bfloat16, device="cuda")
    ref = np.ascontiguousarray(pr.pool[pr.idx].astype(np.float64))   # [bs, H, P, N]
    local = np.arange(bs)
    bound = np.zeros_like(ref)
    worst_state, worst_y = 0.0, 0
    try:
        for t in range(steps):
            x, dt, B, C = wl.request_inputs(rng, bs, H)
            op(pool_d, idx_d, bf16_tensor(x, "cuda"), bf16_tensor(dt, "cuda"), dt_bias, A,
               bf16_tensor(B, "cuda"), bf16_tensor(C, "cuda"), D, out)
            prev = ref.copy()
            y_ref, skipped = oracle.ssu_step_inplace(ref, local, x, dt, pr.dt_bias, pr.A, B, C,
                                                     pr.D)
            assert skipped == 0
            # the bound's own terms, in double, from the step's inputs
            z = oracle.bf16_to_f64(dt) + pr.dt_bias[None, :]
            dtv = np.where(z > 20.0, z, np.log1p(np.exp(z)))                 # [bs, H]
            r_dtv = (np.abs(z) / (1.0 + np.exp(-z)) / dtv + 5.0) * U
            r_dA = (np.abs(dtv * pr.A[None, :]) * (r_dtv + U) + 2.0 * U)[:, :, None, None]
            r_k = (r_dtv + 2.0 * U)[:, :, None, None]
            dA = np.exp(dtv * pr.A[None, :])[:, :, None, None]
            xin = oracle.bf16_to_f64(x)                                      # [bs, H, P]
            Bf = oracle.bf16_to_f64(B)[:, 0]                                 # [bs, N]
            kb = np.abs(dtv[:, :, None, None] * xin[:, :, :, None] * Bf[:, None, None, :])
            bound = dA * bound + 2.0 * (np.abs(prev) * dA * r_dA + kb * r_k + np.abs(ref) * U)
            torch.cuda.synchronize()
            # every readout: 2 ulp, or the dot product's bound plus the carried state error
            Cf = oracle.bf16_to_f64(C)[:, 0]                                 # [bs, N]
            got_bits = bits_of(out)
            got_y = oracle.bf16_to_f64(got_bits)
            ref_bits = oracle.bf16_rne(y_ref)
            mag = np.abs(ref * Cf[:, None, None, :]).sum(-1)
            carried = (bound * np.abs(Cf)[:, None, None, :]).sum(-1)
            dx = np.abs(pr.D[None, :, None] * xin)
            tol = 2 * ulp_bf16(y_ref) + (N + 4) * 2.0 ** -24 * mag + carried + dx * 2.0 ** -23
            ok = (got_bits == ref_bits) | (np.abs(got_y - y_ref) <= tol)
            assert ok.all(), f"step {t}: readout outside the accumulated bound"
            worst_y = max(worst_y, int(np.abs(ordered_bf16(got_bits) -
                                              ordered_bf16(ref_bits)).max()))
            if t % 32 == 31:
                got = pool_d.cpu().numpy()[pr.idx].astype(np.float64)
                err = np.abs(got - ref)
                assert (err <= bound + 1e-30).all(), \
                    f"step {t}: state error {err.max():.3e} above its bound"
                worst_state = max(worst_state, float((err / (1.0 + np.abs(ref))).max()))
        assert op.get_error() == (0, -1)
    finally:
        op.close()
    # untouched slots never changed
    others = np.setdiff1d(np.arange(16), pr.idx)
    assert np.array_equal(pool_d.cpu().numpy()[others], pr.pool[others])
    print(f"128 steps: worst state error {worst_state:.2e} relative, worst readout "
          f"{worst_y} bf16 ulp apart")
