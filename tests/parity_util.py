"""Helpers shared by the GPU parity tests: moving problems to the device, running the oracle
on sampled requests, and the tolerance rules.

Tolerances (written here once, used by every parity test):

* updated state: ``|S_gpu - S_ref| <= 1e-5 * (1 + |S_ref|)`` per element; for a bf16 state
  pool half a bf16 spacing of ``S_ref`` is allowed on top (the storage rounding);
* readout ``y`` (bf16): within 2 bf16 ulp of the oracle's correctly rounded value, or, where
  ``y`` is small against the terms it sums (cancellation), within
  ``2 * ulp_bf16(y_ref) + gamma * sum_n |S'_n C_n| + |D x| * 2^-23`` with
  ``gamma = (N + 4) * 2^-24``, the classical forward error bound of an fp32 dot product of
  length N plus the skip term;
* indexing: bit-exact (untouched slots bit-identical, touched slots compared as above).
"""

from __future__ import annotations

import numpy as np
import torch

import oracle

STATE_RTOL = 1e-5
Y_ULPS = 2


def bf16_tensor(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def pool_tensor(pool: np.ndarray, dev) -> torch.Tensor:
    """Device tensor of a host pool: fp32 values or bf16 patterns (uint16)."""
    if pool.dtype == np.uint16:
        return bf16_tensor(pool, dev)
    return torch.from_numpy(pool).to(dev)


def pool_host(t: torch.Tensor) -> np.ndarray:
    """Host copy of a device pool in the same representation (fp32 or uint16 patterns)."""
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def widen(a: np.ndarray) -> np.ndarray:
    """float64 values of an fp32 array or of bf16 patterns."""
    return oracle.bf16_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def to_device(pr, dev="cuda", idx_dtype=torch.int32):
    """Contiguous device tensors for a workloads.Problem."""
    return dict(
        state_pool=pool_tensor(pr.pool, dev),
        state_batch_indices=torch.from_numpy(pr.idx).to(dev).to(idx_dtype),
        x=bf16_tensor(pr.x, dev), dt=bf16_tensor(pr.dt, dev),
        dt_bias=torch.from_numpy(pr.dt_bias).to(dev), A=torch.from_numpy(pr.A).to(dev),
        B=bf16_tensor(pr.B, dev), C=bf16_tensor(pr.C, dev), D=torch.from_numpy(pr.D).to(dev),
        out=torch.zeros(pr.x.shape, dtype=torch.bfloat16, device=dev))


def ordered_bf16(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def ulp_bf16(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126)
    return np.where(a > 0, np.exp2(e - 7), 2.0 ** -133)


def check_state(got: np.ndarray, ref: np.ndarray, what: str = "state") -> float:
    """fp32 state: |err| <= 1e-5 (1 + |ref|).  bf16 state (uint16 patterns): the stored value
    is the fp32 update rounded to nearest bf16, so |err| <= 0.5 ulp_bf16(ref) + 1e-5 (1 + |ref|)
    (half a bf16 spacing for the storage rounding plus the fp32 arithmetic's share)."""
    if got.dtype == np.uint16:
        g = oracle.bf16_to_f64(got)
        excess = np.abs(g - ref) - 0.5 * ulp_bf16(ref)
        err = np.maximum(excess, 0.0) / (1.0 + np.abs(ref))
    else:
        g = got.astype(np.float64)
        err = np.abs(g - ref) / (1.0 + np.abs(ref))
    worst = float(err.max()) if err.size else 0.0
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    assert worst <= STATE_RTOL, f"{what}: max |err|/(1+|ref|) = {worst:.3e} > {STATE_RTOL}"
    return worst


# Running totals of the readout checks of this test session (printed at the end of the run
# by conftest.py): how many readouts were compared, how many passed only by the cancellation
# rule (ii), and how close those came to the bound.
READOUT_REPORT = {"readouts": 0, "rule_ii": 0, "rule_ii_worst_frac": 0.0,
                  "rule_ii_least_cancellation": 0.0, "worst_ulp": 0}


def check_y(got_bits: np.ndarray, y_ref: np.ndarray, new_state_ref: np.ndarray,
            C_ref: np.ndarray, Dx_ref: np.ndarray, N: int, what: str = "y") -> dict:
    """got_bits [..., P] bf16 patterns; y_ref [..., P] float64; new_state_ref [..., P, N];
    C_ref [..., N] broadcastable against new_state_ref's leading dims; Dx_ref like y_ref.

    A readout passes by rule (i), within 2 bf16 steps of the oracle's correctly rounded value,
    or by rule (ii), within 2 ulp(y_ref) + gamma * sum_n |S'_n C_n| + 2^-23 |D x|.  Rule (ii)
    is only sound where the fp32 sum can be that far off, so every readout that passes by it
    alone must sit where the fp32 forward-error bound is at least one bf16 ulp of y_ref (the
    sum cancels); one that does not is reported as a failure.  Returns the counts."""
    ref_bits = oracle.bf16_rne(y_ref)
    dist = np.abs(ordered_bf16(got_bits) - ordered_bf16(ref_bits))
    gamma = (N + 4) * 2.0 ** -24
    mag = np.abs(new_state_ref * C_ref[..., None, :]).sum(axis=-1)
    got = oracle.bf16_to_f64(got_bits)
    fp32_bound = gamma * mag + np.abs(Dx_ref) * 2.0 ** -23
    ulp = ulp_bf16(y_ref)
    bound = Y_ULPS * ulp + fp32_bound
    ok_ulp = dist <= Y_ULPS
    err = np.abs(got - y_ref)
    ok_abs = err <= bound
    bad = ~(ok_ulp | ok_abs)
    assert not bad.any(), (f"{what}: {int(bad.sum())} readouts out of tolerance; worst ulp "
                           f"distance {int(dist.max())}")
    rule_ii = ~ok_ulp & ok_abs
    n_ii = int(rule_ii.sum())
    worst_frac = float((err / bound)[rule_ii].max()) if n_ii else 0.0
    # |y_ref| / sum |S'C|: the smaller, the more the sum cancels
    least_cancel = float((np.abs(y_ref) / np.maximum(mag, 1e-300))[rule_ii].max()) if n_ii \
        else 0.0
    if n_ii:
        unsound = rule_ii & (fp32_bound < ulp)
        assert not unsound.any(), (f"{what}: {int(unsound.sum())} readouts pass only by the "
                                   f"cancellation rule where the sum does not cancel")
    R = READOUT_REPORT
    R["readouts"] += int(dist.size)
    R["rule_ii"] += n_ii
    R["rule_ii_worst_frac"] = max(R["rule_ii_worst_frac"], worst_frac)
    R["rule_ii_least_cancellation"] = max(R["rule_ii_least_cancellation"], least_cancel)
    R["worst_ulp"] = max(R["worst_ulp"], int(dist.max()) if dist.size else 0)
    return {"max_ulp": int(dist.max()) if dist.size else 0, "abs_rule_used": n_ii,
            "abs_rule_worst_frac": worst_frac}


def oracle_on_requests(pool_host: np.ndarray, idx: np.ndarray, rows: np.ndarray, x, dt,
                       dt_bias, A, B, C, D, ngroups: int = 1, threads: int = 1):
    """Run the oracle on requests ``rows`` only (split over ``threads`` host threads).

    The sampled requests' slots are gathered from the (pre-step) host pool into a small pool
    whose slot j holds request rows[j]'s state, so the oracle's own slot lookup still runs.
    Returns (new_states [k,H,P,N] float64, y [k,H,P] float64).
    """
    rows = np.asarray(rows, dtype=np.int64)
    slots = idx[rows]
    sub = np.ascontiguousarray(widen(pool_host[slots]))
    local = np.arange(len(rows), dtype=np.int64)
    y, skipped = oracle.ssu_step_inplace(sub, local, x[rows], dt[rows], dt_bias, A, B[rows],
                                         C[rows], D, ngroups, threads=threads)
    assert skipped == 0
    return sub, y


def expected_terms(x_bits, D, C_bits, ngroups: int, H: int):
    """(C per head [k,H,N] float64, D*x [k,H,P] float64) for the readout tolerance."""
    Cf = oracle.bf16_to_f64(C_bits)                 # [k, G, N]
    g = np.arange(H) // (H // ngroups)
    Ch = Cf[:, g, :]                                 # [k, H, N]
    Dx = np.asarray(D, dtype=np.float64)[None, :, None] * oracle.bf16_to_f64(x_bits)
    return Ch, Dx


def compare_every_request(pool_before: np.ndarray, idx: np.ndarray, x, dt, dt_bias, A, B, C, D,
                          got_pool_dev: torch.Tensor, got_out_bits: np.ndarray, ngroups: int = 1,
                          rows=None, chunk: int = 32, threads: int | None = None) -> dict:
    """Every request in ``rows`` (default: all) against the oracle, ``chunk`` requests at a
    time so host memory stays bounded: the updated state of its slot (read back from
    ``got_pool_dev``) and its readout.  ``pool_before`` is the host pool before the call."""
    import os
    rows = np.arange(len(idx)) if rows is None else np.asarray(rows)
    threads = threads or os.cpu_count() or 1
    H = x.shape[1]
    N = pool_before.shape[-1]
    worst = {"max_ulp": 0, "abs_rule_used": 0, "state_err": 0.0, "requests": 0}
    for lo in range(0, len(rows), chunk):
        r = rows[lo:lo + chunk]
        ref_states, ref_y = oracle_on_requests(pool_before, idx, r, x, dt, dt_bias, A, B, C, D,
                                               ngroups, threads=threads)
        sel = torch.from_numpy(idx[r].astype(np.int64)).to(got_pool_dev.device)
        got = pool_host(got_pool_dev[sel])
        worst["state_err"] = max(worst["state_err"], check_state(got, ref_states))
        Ch, Dx = expected_terms(x[r], D, C[r], ngroups, H)
        st = check_y(got_out_bits[r], ref_y, ref_states, Ch, Dx, N)
        worst["max_ulp"] = max(worst["max_ulp"], st["max_ulp"])
        worst["abs_rule_used"] += st["abs_rule_used"]
        worst["requests"] += len(r)
    return worst
