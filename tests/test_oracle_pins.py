"""Pins for the CPU oracle: checks against what the definition and the mathematics fix.

None of these retypes the oracle's loop.  Each one is a hand-computed value, a special case
with a closed form, an invariant (linearity, the unrolled T-step recurrence), or a library
routine on a case where it must agree.  A dropped term, a swapped operand, a wrong sign or a
wrong head-to-group map each fails at least one of them (see the comments per test).
"""

import json
import math
from pathlib import Path

import numpy as np
import pytest

import oracle
import workloads as wl

GOLDEN = Path(__file__).resolve().parent / "golden"
LN2 = math.log(2.0)


def _bits(v):
    return wl.f32_to_bf16_bits(np.asarray(v, dtype=np.float32))


def _unit_case(S, x, dt, dt_bias, A, B, C, D):
    """Run the oracle on one request, one head, P=1, N=len(S), a one-slot pool."""
    N = len(S)
    pool = np.asarray(S, dtype=np.float64).reshape(1, 1, 1, N)
    xb = _bits([x]).reshape(1, 1, 1)
    dtb = _bits([dt]).reshape(1, 1)
    Bb = _bits(B).reshape(1, 1, N)
    Cb = _bits(C).reshape(1, 1, N)
    new_pool, y, skipped = oracle.ssu_step(pool, np.array([0]), xb, dtb, [dt_bias], [A], Bb,
                                           Cb, [D])
    assert skipped == 0
    return new_pool.reshape(N), float(y.reshape(()))


@pytest.mark.parametrize("case", json.loads((GOLDEN / "hand_cases.json").read_text())["cases"],
                         ids=lambda c: c["name"])
def test_hand_cases(case):
    # base: catches y read from the old state (3.5), a missing D*x (1.5), a missing softplus
    # (dA = 1), the sign of A (dA = 2) and B/C swapped (2 ln 2).  bias_carries_dt: dt_bias
    # dropped.  decay_only: the input term.  selector: the column a C = e_k picks, and bf16.
    S_new, y = _unit_case(case["S"], case["x"], case["dt"], case["dt_bias"], case["A"],
                          case["B"], case["C"], case["D"])
    np.testing.assert_allclose(S_new, case["S_new"], rtol=0, atol=1e-15)
    assert y == pytest.approx(case["y"], abs=1e-15)
    assert int(oracle.bf16_rne([y])[0]) == int(case["y_bf16_bits"], 16)


def test_hand_case_values_follow_from_ln2():
    # The fixture's decimals are 0.5 + ln 2 and 1 - ln 2.
    case = json.loads((GOLDEN / "hand_cases.json").read_text())["cases"][0]
    assert case["S_new"][0] == pytest.approx(0.5 + LN2, abs=1e-16)
    assert case["S_new"][1] == pytest.approx(1.0 - LN2, abs=1e-16)


def test_softplus_large_argument():
    # z = 25: softplus(z) = z + log1p(e^-z) = 25 + 1.4e-11, so S' = S e^{25 A} + 25 x B.
    A = -0.04
    S_new, y = _unit_case([1.0, 2.0], 1.0, 20.0, 5.0, A, [1.0, -1.0], [1.0, 1.0], 0.0)
    dA = math.exp(25.0 * A)
    np.testing.assert_allclose(S_new, [dA + 25.0, 2 * dA - 25.0], rtol=1e-9)
    assert y == pytest.approx(3 * dA, rel=1e-9)


def test_softplus_small_argument():
    # z = -30: softplus(z) = e^z (1 - e^z/2 + ...) to double precision.
    A = -1.0
    S_new, _ = _unit_case([1.0, 1.0], 1.0, -32.0, 2.0, A, [1.0, 0.0], [0.0, 0.0], 0.0)
    dtv = math.exp(-30.0)
    assert S_new[0] == pytest.approx(math.exp(-dtv) + dtv, rel=1e-15)


def _random_problem(bs=3, H=4, P=5, N=6, G=1, pool_size=7, seed=11):
    return wl.make_problem(bs, H, P, N, G, pool_size=pool_size, seed=seed)


def _run(pr, **over):
    args = dict(pool=pr.pool, idx=pr.idx, x=pr.x, dt=pr.dt, dt_bias=pr.dt_bias, A=pr.A, B=pr.B,
                C=pr.C, D=pr.D, ngroups=pr.ngroups)
    args.update(over)
    return oracle.ssu_step(**args)


def _softplus_lib(z):
    return np.logaddexp(0.0, z)  # numpy's log(e^0 + e^z)


def test_zero_input_is_pure_decay():
    # x = 0: S' = S * exp(softplus(dt + dt_bias) * A) and y = S' C (the D x term vanishes).
    pr = _random_problem()
    x0 = np.zeros_like(pr.x)
    new_pool, y, _ = _run(pr, x=x0)
    z = oracle.bf16_to_f64(pr.dt) + pr.dt_bias.astype(np.float64)[None, :]
    dA = np.exp(_softplus_lib(z) * pr.A.astype(np.float64)[None, :])           # [bs, H]
    S0 = pr.pool.astype(np.float64)[pr.idx]                                     # [bs,H,P,N]
    expect = S0 * dA[:, :, None, None]
    np.testing.assert_allclose(new_pool[pr.idx], expect, rtol=1e-14, atol=0)
    Cv = oracle.bf16_to_f64(pr.C)[:, 0, :]                                      # G = 1
    np.testing.assert_allclose(y, np.einsum("bhpn,bn->bhp", expect, Cv), rtol=1e-12,
                               atol=1e-12)


@pytest.mark.parametrize("k", [0, 3, 5])
def test_unit_vector_C_selects_a_state_column(k):
    # C = e_k: y[p] = S'[p, k] + D x[p].  A wrong p/n index or an off-by-one fails.
    pr = _random_problem()
    N = pr.C.shape[-1]
    ek = np.zeros((pr.batch, 1, N), dtype=np.float32)
    ek[:, :, k] = 1.0
    new_pool, y, _ = _run(pr, C=_bits(ek))
    x = oracle.bf16_to_f64(pr.x)
    expect = new_pool[pr.idx][:, :, :, k] + pr.D.astype(np.float64)[None, :, None] * x
    np.testing.assert_allclose(y, expect, rtol=0, atol=1e-13)


def _zero_state(pr):
    pool = np.zeros_like(pr.pool)
    return pool


def test_linearity_in_x_and_B():
    # From a zero state, S' and y - D x are linear in x (B fixed) and in B (x fixed).
    pr = _random_problem(seed=5)
    pool0 = _zero_state(pr)
    x = oracle.bf16_to_f64(pr.x)
    D = pr.D.astype(np.float64)[None, :, None]
    rng = np.random.default_rng(99)
    u = wl.f32_to_bf16_bits(rng.standard_normal(pr.x.shape, dtype=np.float32))
    v = wl.f32_to_bf16_bits(rng.standard_normal(pr.x.shape, dtype=np.float32))
    a = -0.5  # a power of two, so a * B is exact in bf16 (checked below)
    uf, vf = oracle.bf16_to_f64(u), oracle.bf16_to_f64(v)

    def f(xbits):
        P1, y1, _ = _run(pr, pool=pool0, x=xbits)
        return P1[pr.idx], y1 - D * oracle.bf16_to_f64(xbits)

    Su, yu = f(u)
    Sv, yv = f(v)
    # a*u + b*v is not in general a bf16 value; use bf16 inputs whose combination is exact:
    # scale by powers of two only (u -> 2u is exact), then add separately-run results.
    S2u, y2u = f(wl.f32_to_bf16_bits((2.0 * uf).astype(np.float32)))
    np.testing.assert_allclose(S2u, 2.0 * Su, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(y2u, 2.0 * yu, rtol=1e-13, atol=1e-13)
    # additivity: run x = u + v where the sum is representable (round u + v to bf16 first
    # and compare with the sum of runs on the same two addends split exactly).
    s = uf + vf
    sb = wl.f32_to_bf16_bits(s.astype(np.float32))
    r = s - oracle.bf16_to_f64(sb)              # remainder; the split sb + r is exact
    rb = wl.f32_to_bf16_bits(r.astype(np.float32))
    assert np.array_equal(oracle.bf16_to_f64(rb), r)
    Ss, ys = f(sb)
    Sr, yr = f(rb)
    np.testing.assert_allclose(Ss + Sr, Su + Sv, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(ys + yr, yu + yv, rtol=1e-12, atol=1e-12)
    # linearity in B with x fixed: B -> a B and B -> B1 + B2 (same exact-split trick)
    Bf = oracle.bf16_to_f64(pr.B)
    P_B, yB, _ = _run(pr, pool=pool0)
    aB = wl.f32_to_bf16_bits((a * Bf).astype(np.float32))
    assert np.array_equal(oracle.bf16_to_f64(aB), a * Bf)
    P_aB, yaB, _ = _run(pr, pool=pool0, B=aB)
    np.testing.assert_allclose(P_aB[pr.idx], a * P_B[pr.idx], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(yaB - D * x, a * (yB - D * x), rtol=1e-12, atol=1e-12)
    Bv = oracle.bf16_to_f64(wl.f32_to_bf16_bits(rng.standard_normal(pr.B.shape,
                                                                    dtype=np.float32)))
    t = Bf + Bv
    tb = wl.f32_to_bf16_bits(t.astype(np.float32))
    tr = t - oracle.bf16_to_f64(tb)
    trb = wl.f32_to_bf16_bits(tr.astype(np.float32))
    assert np.array_equal(oracle.bf16_to_f64(trb), tr)
    P_t, yt, _ = _run(pr, pool=pool0, B=tb)
    P_r, yr2, _ = _run(pr, pool=pool0, B=trb)
    P_v, yv2, _ = _run(pr, pool=pool0, B=wl.f32_to_bf16_bits(Bv.astype(np.float32)))
    np.testing.assert_allclose(P_t[pr.idx] + P_r[pr.idx], P_B[pr.idx] + P_v[pr.idx],
                               rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose((yt - D * x) + (yr2 - D * x), (yB - D * x) + (yv2 - D * x),
                               rtol=1e-12, atol=1e-12)


def test_T_steps_match_unrolled_recurrence():
    # Unrolling S_t = dA_t S_{t-1} + dt_t x_t (x) B_t over T steps gives
    #   S_T = (prod_t dA_t) S_0 + sum_t (prod_{u>t} dA_u) dt_t x_t (x) B_t,
    # and y_T = S_T C_T + D x_T.  A dropped dA or a wrong outer product fails.
    T, H, P, N = 5, 3, 4, 6
    rng = np.random.default_rng(7)
    pool = rng.standard_normal((2, H, P, N))
    slot = 1
    S0 = pool[slot].copy()
    dt_bias, A, D = wl.head_params(rng, H)
    steps = [wl.request_inputs(rng, 1, H, P, N, 1) for _ in range(T)]
    cur = pool.copy()
    for t in range(T):
        x, dt, B, C = steps[t]
        y, _ = oracle.ssu_step_inplace(cur, np.array([slot]), x, dt, dt_bias, A, B, C, D)
    dA = []
    terms = []
    for t in range(T):
        x, dt, B, C = steps[t]
        z = oracle.bf16_to_f64(dt)[0] + dt_bias.astype(np.float64)
        dtv = _softplus_lib(z)
        dA.append(np.exp(dtv * A.astype(np.float64)))                       # [H]
        xf = oracle.bf16_to_f64(x)[0]                                         # [H, P]
        Bf = oracle.bf16_to_f64(B)[0, 0]                                      # [N]
        terms.append(dtv[:, None, None] * xf[:, :, None] * Bf[None, None, :])
    closed = np.prod(dA, axis=0)[:, None, None] * S0
    for t in range(T):
        decay = np.prod(dA[t + 1:], axis=0) if t + 1 < T else np.ones(H)
        closed = closed + decay[:, None, None] * terms[t]
    np.testing.assert_allclose(cur[slot], closed, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(cur[0], pool[0])                           # other slot
    x, dt, B, C = steps[-1]
    yT = closed @ oracle.bf16_to_f64(C)[0, 0] + D.astype(np.float64)[:, None] * \
        oracle.bf16_to_f64(x)[0]
    np.testing.assert_allclose(y[0], yT, rtol=1e-12, atol=1e-12)


def test_heads_map_to_contiguous_groups():
    # H = 4, G = 2: heads 0,1 read group 0 and heads 2,3 read group 1 (g = h / (H/G)).
    # With group 1's B zeroed, heads 2 and 3 only decay; heads 0 and 1 do not.  An h % G
    # mapping would leave heads 1 and 3 decaying instead.
    pr = wl.make_problem(2, 4, 3, 8, 2, pool_size=4, seed=3)
    Bf = wl.bf16_bits_to_f32(pr.B).copy()
    Bf[:, 1, :] = 0.0
    new_pool, _, _ = _run(pr, B=_bits(Bf))
    z = oracle.bf16_to_f64(pr.dt) + pr.dt_bias.astype(np.float64)[None, :]
    dA = np.exp(_softplus_lib(z) * pr.A.astype(np.float64)[None, :])
    S0 = pr.pool.astype(np.float64)[pr.idx]
    decayed = S0 * dA[:, :, None, None]
    got = new_pool[pr.idx]
    np.testing.assert_allclose(got[:, 2:], decayed[:, 2:], rtol=1e-14)
    assert np.all(np.abs(got[:, :2] - decayed[:, :2]).max(axis=(2, 3)) > 1e-3)


def test_untouched_slots_and_out_of_range_requests():
    pr = wl.make_problem(4, 2, 3, 8, 1, pool_size=9, seed=21)
    idx = pr.idx.copy()
    idx[2] = 9        # one past the end: skipped and counted
    new_pool, y, skipped = _run(pr, idx=idx)
    assert skipped == 1
    assert np.isnan(y[2]).all() and not np.isnan(np.delete(y, 2, axis=0)).any()
    touched = set(int(s) for s in np.delete(idx, 2))
    for s in range(pr.pool_size):
        same = np.array_equal(new_pool[s], pr.pool[s].astype(np.float64))
        assert same == (s not in touched), s
    idx[1] = -1
    _, _, skipped = _run(pr, idx=idx)
    assert skipped == 2


def test_threaded_oracle_matches_single_thread_bitwise():
    pr = wl.make_problem(9, 3, 4, 8, 1, pool_size=12, seed=2)
    p1 = pr.pool.astype(np.float64)
    p4 = p1.copy()
    y1, _ = oracle.ssu_step_inplace(p1, pr.idx, pr.x, pr.dt, pr.dt_bias, pr.A, pr.B, pr.C,
                                    pr.D)
    y4, _ = oracle.ssu_step_inplace(p4, pr.idx, pr.x, pr.dt, pr.dt_bias, pr.A, pr.B, pr.C,
                                    pr.D, threads=4)
    assert np.array_equal(p1, p4) and np.array_equal(y1, y4)


# ---- bf16 conversions -------------------------------------------------------------------

@pytest.mark.parametrize("value,bits", [
    (1.0, 0x3F80), (-2.0, 0xC000), (0.0, 0x0000), (-0.0, 0x8000),
    (1.0 + 2.0 ** -8, 0x3F80),          # halfway between 1 and 1 + 2^-7: ties to even (down)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),      # halfway between 1+2^-7 and 1+2^-6: even is up
    (1.0 + 2.0 ** -8 + 2.0 ** -30, 0x3F81),  # just above halfway: up
    (3.3895313892515355e38, 0x7F7F),    # largest bf16
    (3.4e38, 0x7F80),                   # rounds past the largest: +inf
    (2.0 ** -133, 0x0001),              # smallest subnormal
    (2.0 ** -134, 0x0000),              # half the smallest subnormal: ties to even (zero)
    (3 * 2.0 ** -134, 0x0002),          # 1.5 subnormal steps: ties to even (two)
    (float("inf"), 0x7F80), (float("-inf"), 0xFF80),
])
def test_bf16_rne_special_values(value, bits):
    assert int(oracle.bf16_rne([value])[0]) == bits


def test_bf16_rne_matches_torch_on_fp32_values():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(4)
    v = np.concatenate([rng.standard_normal(20000), rng.standard_normal(2000) * 1e-39,
                        rng.standard_normal(2000) * 1e30]).astype(np.float32)
    ours = oracle.bf16_rne(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_widening():
    bits = np.array([0x3F80, 0xC000, 0x3F4F, 0x0001, 0x7F7F], dtype=np.uint16)
    np.testing.assert_array_equal(oracle.bf16_to_f64(bits),
                                  [1.0, -2.0, 207 / 256, 2.0 ** -133, 3.3895313892515355e38])


# ---- the input generators ----------------------------------------------------------------

def test_generator_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    v = np.random.default_rng(8).standard_normal(50000).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(wl.f32_to_bf16_bits(v), ref)


def test_generators_are_seeded_and_slots_distinct():
    a = wl.make_problem(8, 16, pool_size=32, seed=0)
    b = wl.make_problem(8, 16, pool_size=32, seed=0)
    for k in ("pool", "idx", "x", "dt", "dt_bias", "A", "B", "C", "D"):
        assert np.array_equal(getattr(a, k), getattr(b, k)), k
    assert len(set(a.idx.tolist())) == 8 and a.idx.min() >= 0 and a.idx.max() < 32
    dt = wl.bf16_bits_to_f32(a.dt)
    assert dt.min() >= -4.0 and dt.max() <= 0.0
    assert (a.A <= -1.0).all() and (a.A >= -16.0).all()
    assert (a.D >= 0).all() and (a.D <= 1).all()
    sets = wl.rotation_sets(128, 19)
    assert sets.shape == (19, 128)
    assert sorted(sets.ravel().tolist()) == list(range(19 * 128))


def test_cold_l2_set_count():
    # 128 requests x 16 heads x 32 KiB = 64 MiB per set; 3 x 126.5 MiB needs 6 sets, and the
    # batch-128 workload's 19 sets (1216 MiB) are well above that.
    l2 = int(126.5 * 2 ** 20)
    assert wl.sets_for_cold_l2(128, 16, l2) == 6
    assert wl.sets_for_cold_l2(8, 16, l2) == 95
    assert wl.sets_for_cold_l2(512, 16, l2, min_sets=3) == 3


# ---- the state-block copy ----------------------------------------------------------------

def test_copy_blocks_hand_case():
    # Two tensors of 4 blocks; requests copy 0 -> 2 and 3 -> 1; block ids written out by hand.
    a = np.arange(4 * 3, dtype=np.float32).reshape(4, 3)          # block k = [3k, 3k+1, 3k+2]
    b = np.array([[10, 11], [20, 21], [30, 31], [40, 41]], dtype=np.uint16)
    (na, nb), skipped = oracle.copy_blocks([a, b], [0, 3], [2, 1])
    assert skipped == 0
    np.testing.assert_array_equal(na, [[0, 1, 2], [9, 10, 11], [0, 1, 2], [9, 10, 11]])
    np.testing.assert_array_equal(nb, [[10, 11], [40, 41], [10, 11], [40, 41]])
    np.testing.assert_array_equal(a, np.arange(12).reshape(4, 3))  # inputs untouched


def test_copy_blocks_skips_requests_out_of_any_range():
    a = np.zeros((4, 2), dtype=np.float32)
    b = np.ones((3, 2), dtype=np.float32)
    a[1] = 5
    (na, nb), skipped = oracle.copy_blocks([a, b], [1, 3, -1], [0, 2, 0])
    # request 1 names block 3, valid in a but not in b: skipped for both tensors
    assert skipped == 2
    np.testing.assert_array_equal(na[0], [5, 5])
    np.testing.assert_array_equal(na[2], [0, 0])


def test_tokens_oracle_matches_the_unrolled_recurrence_at_every_token():
    # oracle.ssu_tokens: intermediate state after token t equals
    #   (prod_{u<=t} dA_u) S_0 + sum_{v<=t} (prod_{v<u<=t} dA_u) dt_v x_v (x) B_v,
    # and y_t = S_t C_t + D x_t; requests with an out-of-range slot are skipped.
    T, bs, H, P, N = 4, 3, 2, 3, 8
    rng = np.random.default_rng(31)
    pool = rng.standard_normal((5, H, P, N))
    idx = np.array([3, 0, 9])                       # request 2 names no slot
    dt_bias, A, D = wl.head_params(rng, H)
    steps = [wl.request_inputs(rng, bs, H, P, N, 1) for _ in range(T)]
    x, dt, B, C = (np.stack([s[k] for s in steps], 1) for k in range(4))
    new_pool, y, inter, skipped = oracle.ssu_tokens(pool, idx, x, dt, dt_bias, A, B, C, D)
    assert skipped == 1 and np.isnan(inter[2]).all()
    for b in (0, 1):
        S = pool[idx[b]].copy()
        dA_list, terms = [], []
        for t in range(T):
            z = oracle.bf16_to_f64(dt[b, t]) + dt_bias.astype(np.float64)
            dtv = _softplus_lib(z)
            dA_list.append(np.exp(dtv * A.astype(np.float64)))
            xf = oracle.bf16_to_f64(x[b, t])
            Bf = oracle.bf16_to_f64(B[b, t, 0])
            terms.append(dtv[:, None, None] * xf[:, :, None] * Bf[None, None, :])
            closed = np.prod(dA_list, axis=0)[:, None, None] * S
            for v in range(t + 1):
                decay = np.prod(dA_list[v + 1:t + 1], axis=0) if v < t else np.ones(H)
                closed = closed + decay[:, None, None] * terms[v]
            np.testing.assert_allclose(inter[b, t], closed, rtol=1e-12, atol=1e-12)
            yt = closed @ oracle.bf16_to_f64(C[b, t, 0]) + D.astype(np.float64)[:, None] * xf
            np.testing.assert_allclose(y[b, t], yt, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(new_pool[idx[b]], inter[b, T - 1], rtol=0, atol=0)
    np.testing.assert_array_equal(new_pool[[1, 2, 4]], pool[[1, 2, 4]])
