"""GPU parity: the CUDA path (through the C ABI) against the double-precision oracle.

Small problems are compared element by element in full.  The full-size workloads (batch 128
over a 19-set rotation pool, batch 512 on packed strided views, the head sweep at batch 256)
run in the launch configuration the bench times and are compared on sampled requests the
oracle computes one by one, plus bit-exact checks of every untouched slot.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import selective_state_update_02_gb300 as ssu
import workloads as wl
from parity_util import (bf16_tensor, bits_of, check_state, check_y, compare_every_request,
                         expected_terms, oracle_on_requests, to_device)

pytestmark = pytest.mark.gpu

DEV = "cuda"


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


def _compare_all(pr, t, before_pool):
    """Full comparison of every request, every slot."""
    rows = np.arange(pr.batch)
    ref_states, ref_y = oracle_on_requests(pr.pool, pr.idx, rows, pr.x, pr.dt, pr.dt_bias,
                                           pr.A, pr.B, pr.C, pr.D, pr.ngroups)
    got_pool = t["state_pool"].cpu().numpy()
    check_state(got_pool[pr.idx], ref_states)
    Ch, Dx = expected_terms(pr.x, pr.D, pr.C, pr.ngroups, pr.nheads)
    stats = check_y(bits_of(t["out"]), ref_y, ref_states, Ch, Dx, pr.pool.shape[-1])
    untouched = np.setdiff1d(np.arange(pr.pool_size), pr.idx)
    assert np.array_equal(got_pool[untouched], before_pool[untouched]), "untouched slot changed"
    return stats


@pytest.mark.parametrize("idx_dtype", [torch.int32, torch.int64])
def test_tiny_decode_step(op, idx_dtype):
    # batch 8, 16 heads, headdim 64, dstate 128, 32-slot pool, seed 0
    pr = wl.make_problem(8, 16, pool_size=32, seed=0)
    t = to_device(pr, DEV, idx_dtype)
    _run(op, t)
    assert op.get_error() == (0, -1)
    _compare_all(pr, t, pr.pool)


@pytest.mark.parametrize("P", [1, 3, 8, 40, 64, 100, 128])
def test_ragged_headdim(op, P):
    pr = wl.make_problem(5, 6, P=P, pool_size=13, seed=P)
    t = to_device(pr, DEV)
    _run(op, t)
    _compare_all(pr, t, pr.pool)


@pytest.mark.parametrize("H,G", [(8, 2), (8, 8), (12, 3)])
def test_groups(op, H, G):
    pr = wl.make_problem(6, H, G=G, pool_size=10, seed=H * G)
    t = to_device(pr, DEV)
    _run(op, t)
    _compare_all(pr, t, pr.pool)


VEC_SHAPES = [(ssu.SSU_MODE_VEC, r, w, 0) for r in (1, 2, 4, 8, 16) for w in (1, 2, 3, 4, 8, 16)]
SHAPES = VEC_SHAPES


@pytest.mark.parametrize("P", [64, 40])
def test_every_launch_shape_is_bitwise_identical(op, P):
    # Each row's readout is summed in one fixed order, so all shapes agree bit for bit
    # (state and output), as the launch configs of the pages' table do.
    pr = wl.make_problem(7, 16, P=P, pool_size=24, seed=3)
    ref = to_device(pr, DEV)
    op.set_launch(ssu.SSU_MODE_AUTO)
    _run(op, ref)
    _compare_all(pr, ref, pr.pool)
    try:
        for shape in SHAPES:
            t = to_device(pr, DEV)
            op.set_launch(*shape)
            _run(op, t)
            assert torch.equal(t["state_pool"], ref["state_pool"]), shape
            assert torch.equal(t["out"].view(torch.int16), ref["out"].view(torch.int16)), shape
        assert op.get_error() == (0, -1)
    finally:
        op.set_launch(ssu.SSU_MODE_AUTO)


@pytest.mark.parametrize("H,G", [(12, 3), (16, 4), (48, 16)])
def test_every_vec_shape_with_groups(op, H, G):
    # Several heads per group: each VEC shape (whichever way it forms a head's group index)
    # reads its B and C rows from group h / (H / G), checked against the oracle at every shape.
    pr = wl.make_problem(5, H, G=G, pool_size=11, seed=H + G)
    try:
        for shape in VEC_SHAPES:
            t = to_device(pr, DEV)
            op.set_launch(*shape)
            _run(op, t)
            _compare_all(pr, t, pr.pool)
        assert op.get_error() == (0, -1)
    finally:
        op.set_launch(ssu.SSU_MODE_AUTO)


@pytest.mark.parametrize("shape", [(ssu.SSU_MODE_VEC, 8, 4, 0), (ssu.SSU_MODE_VEC, 2, 1, 0),
                                   (ssu.SSU_MODE_VEC, 16, 4, 0)])
@pytest.mark.parametrize("idx_dtype", [torch.int32, torch.int64])
def test_many_requests_every_request_checked(op, shape, idx_dtype):
    # 96 requests (several waves of CTAs at every shape), every request against the oracle.
    bs, H = 96, 16
    pr = wl.make_problem(bs, H, pool_size=bs + 16, seed=17)
    t = to_device(pr, DEV, idx_dtype)
    op.set_launch(*shape)
    try:
        _run(op, t)
        assert op.get_error() == (0, -1)
    finally:
        op.set_launch(ssu.SSU_MODE_AUTO)
    _compare_all(pr, t, pr.pool)


def test_skipped_slots_among_many_requests(op):
    pr = wl.make_problem(40, 16, pool_size=48, seed=23)
    idx = pr.idx.copy()
    bad = [0, 5, 39]
    idx[bad] = [48, -1, 1 << 30]
    t = to_device(pr, DEV)
    t["state_batch_indices"] = torch.from_numpy(idx).to(DEV).to(torch.int32)
    t["out"].fill_(3.0)
    _run(op, t)
    assert op.get_error() == (3, 0)
    good = np.setdiff1d(np.arange(40), bad)
    assert (t["out"][bad].float() == 3.0).all()
    ref_states, ref_y = oracle_on_requests(pr.pool, idx, good, pr.x, pr.dt, pr.dt_bias, pr.A,
                                           pr.B, pr.C, pr.D)
    got_pool = t["state_pool"].cpu().numpy()
    check_state(got_pool[idx[good]], ref_states)
    untouched = np.setdiff1d(np.arange(48), idx[good])
    assert np.array_equal(got_pool[untouched], pr.pool[untouched])
    Ch, Dx = expected_terms(pr.x[good], pr.D, pr.C[good], 1, 16)
    check_y(bits_of(t["out"])[good], ref_y, ref_states, Ch, Dx, 128)


def test_padded_rows_leave_the_padding_alone(op):
    # rows padded to 132 floats (row stride 132): the update reads and writes the 128 columns
    # of each row only; the padding stays zero.
    pr = wl.make_problem(4, 16, pool_size=8, seed=29)
    padded = torch.zeros(8, 16, 64, 132, device=DEV)
    padded[..., :128] = torch.from_numpy(pr.pool).to(DEV)
    t = to_device(pr, DEV)
    t["state_pool"] = padded[..., :128]
    _run(op, t)
    _compare_all(pr, dict(t, state_pool=t["state_pool"]), pr.pool)
    assert (padded[..., 128:] == 0).all()


def test_packed_strided_views_and_broadcasts(op):
    # x, B and C are views into one packed bf16 tensor; dt, dt_bias, D and A are stride-0
    # head-expanded views (sglang PR #41223, Details / Kernel measurement).
    bs, H, P, N = 24, 16, 64, 128
    rng = np.random.default_rng(5)
    pool = wl.state_pool(rng, 40, H)
    idx = rng.permutation(40)[:bs].astype(np.int64)
    dt_bias, A, D = wl.head_params(rng, H)
    packed = wl.packed_xbc(rng, bs, H)
    dt = wl.f32_to_bf16_bits(rng.uniform(-4, 0, (bs, H)).astype(np.float32))
    xs = packed[:, :H * P].reshape(bs, H, P)
    Bs = packed[:, H * P:H * P + N].reshape(bs, 1, N)
    Cs = packed[:, H * P + N:].reshape(bs, 1, N)

    pk = bf16_tensor(packed, DEV)
    x_v = pk[:, :H * P].view(bs, H, P)
    B_v = pk[:, H * P:H * P + N].unsqueeze(1)
    C_v = pk[:, H * P + N:].unsqueeze(1)
    assert x_v.stride() == (H * P + 2 * N, P, 1) and B_v.stride()[0] == H * P + 2 * N
    dt_v = bf16_tensor(dt, DEV).unsqueeze(-1).expand(bs, H, P)
    bias_v = torch.from_numpy(dt_bias).to(DEV).unsqueeze(-1).expand(H, P)
    D_v = torch.from_numpy(D).to(DEV).unsqueeze(-1).expand(H, P)
    A_v = torch.from_numpy(A).to(DEV)[:, None, None].expand(H, P, N)
    pool_d = torch.from_numpy(pool).to(DEV)
    out = torch.zeros(bs, H, P, dtype=torch.bfloat16, device=DEV)
    op(pool_d, torch.from_numpy(idx).to(DEV), x_v, dt_v, bias_v, A_v, B_v, C_v, D_v, out)

    pr = wl.Problem(pool, idx, xs.copy(), dt, dt_bias, A, Bs.copy(), Cs.copy(), D, 1)
    t = dict(state_pool=pool_d, out=out)
    _compare_all(pr, t, pool)


def test_out_of_range_requests_are_skipped_and_counted(op):
    pr = wl.make_problem(10, 16, pool_size=16, seed=9)
    idx = pr.idx.copy()
    idx[3] = 16
    idx[7] = -5
    t = to_device(pr, DEV)
    t["state_batch_indices"] = torch.from_numpy(idx).to(DEV).to(torch.int32)
    sentinel = torch.full_like(t["out"], 7.0)
    t["out"].copy_(sentinel)
    _run(op, t)
    skipped, first = op.get_error()
    assert (skipped, first) == (2, 3)
    assert op.get_error() == (0, -1)             # reading clears the counters
    assert torch.equal(t["out"][[3, 7]], sentinel[[3, 7]])
    good = np.setdiff1d(np.arange(10), [3, 7])
    ref_states, ref_y = oracle_on_requests(pr.pool, idx, good, pr.x, pr.dt, pr.dt_bias, pr.A,
                                           pr.B, pr.C, pr.D)
    got_pool = t["state_pool"].cpu().numpy()
    check_state(got_pool[idx[good]], ref_states)
    untouched = np.setdiff1d(np.arange(16), idx[good])
    assert np.array_equal(got_pool[untouched], pr.pool[untouched])
    Ch, Dx = expected_terms(pr.x[good], pr.D, pr.C[good], 1, 16)
    check_y(bits_of(t["out"])[good], ref_y, ref_states, Ch, Dx, 128)


def test_empty_batch_enqueues_nothing(op):
    pr = wl.make_problem(0, 16, pool_size=4, seed=1)
    t = to_device(pr, DEV)
    _run(op, t)
    torch.cuda.synchronize()
    assert torch.equal(t["state_pool"].cpu(), torch.from_numpy(pr.pool))


def test_invalid_arguments_are_rejected_before_launch(op):
    pr = wl.make_problem(4, 16, pool_size=8, seed=2)
    t = to_device(pr, DEV)
    bad = dict(t)
    bad["state_pool"] = torch.zeros(8, 16, 64, 127, device=DEV)                 # dstate 127
    bad["B"] = torch.zeros(4, 1, 127, dtype=torch.bfloat16, device=DEV)
    bad["C"] = torch.zeros(4, 1, 127, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ssu.SsuError) as e:
        _run(op, bad)
    assert e.value.status == ssu.SSU_ERR_UNSUPPORTED
    bad = dict(t)
    bad["dt"] = torch.zeros(4, 16, 64, dtype=torch.bfloat16, device=DEV)        # P-stride 1
    with pytest.raises(ssu.SsuError) as e:
        _run(op, bad)
    assert e.value.status == ssu.SSU_ERR_UNSUPPORTED
    flat = torch.zeros(8 * 16 * 64 * 128 + 1, device=DEV)
    bad = dict(t)
    bad["state_pool"] = flat[1:].view(8, 16, 64, 128)                           # 4 B offset
    with pytest.raises(ssu.SsuError) as e:
        _run(op, bad)
    assert e.value.status == ssu.SSU_ERR_MISALIGNED


# ---- full-size workloads (every request against the oracle) ---------------------------

def test_serving_batch_128_rotation_pool(op):
    # batch 128, 16 heads: 2432-slot pool in 19 disjoint 128-slot sets (>= 3x L2); two
    # consecutive calls on different sets, as the timed sequence issues them.
    bs, H, n_sets = 128, 16, 19
    rng = np.random.default_rng(0)
    pool = wl.state_pool(rng, bs * n_sets, H)
    sets = wl.rotation_sets(bs, n_sets, seed=0)
    dt_bias, A, D = wl.head_params(rng, H)
    pool_d = torch.from_numpy(pool).to(DEV)
    for k in (0, 11):
        x, dt, B, C = wl.request_inputs(rng, bs, H)
        idx = sets[k]
        out = torch.zeros(bs, H, 64, dtype=torch.bfloat16, device=DEV)
        op(pool_d, torch.from_numpy(idx.astype(np.int32)).to(DEV), bf16_tensor(x, DEV),
           bf16_tensor(dt, DEV), torch.from_numpy(dt_bias).to(DEV), torch.from_numpy(A).to(DEV),
           bf16_tensor(B, DEV), bf16_tensor(C, DEV), torch.from_numpy(D).to(DEV), out)
        # every request against the oracle
        compare_every_request(pool, idx, x, dt, dt_bias, A, B, C, D, pool_d, bits_of(out))
        assert torch.isfinite(out.float()).all()
        # untouched slots stay bit-identical; the host copy tracks the expected pool
        mask = np.ones(pool.shape[0], bool)
        mask[idx] = False
        ref_untouched = torch.from_numpy(pool[mask]).to(DEV)
        assert torch.equal(pool_d[torch.from_numpy(np.nonzero(mask)[0]).to(DEV)], ref_untouched)
        pool[idx] = pool_d[torch.from_numpy(idx).to(DEV)].cpu().numpy()
        assert op.get_error() == (0, -1)


def test_large_batch_512_packed_views(op):
    # batch 512, 16 heads, x/B/C strided views of one packed tensor, stride-0 broadcasts,
    # 1536-slot pool in 3 disjoint sets.
    bs, H, P, N = 512, 16, 64, 128
    rng = np.random.default_rng(1)
    pool = wl.state_pool(rng, 3 * bs, H)
    sets = wl.rotation_sets(bs, 3, seed=1)
    dt_bias, A, D = wl.head_params(rng, H)
    packed = wl.packed_xbc(rng, bs, H)
    dt = wl.f32_to_bf16_bits(rng.uniform(-4, 0, (bs, H)).astype(np.float32))
    pk = bf16_tensor(packed, DEV)
    x_v = pk[:, :H * P].view(bs, H, P)
    B_v = pk[:, H * P:H * P + N].unsqueeze(1)
    C_v = pk[:, H * P + N:].unsqueeze(1)
    dt_v = bf16_tensor(dt, DEV).unsqueeze(-1).expand(bs, H, P)
    bias_v = torch.from_numpy(dt_bias).to(DEV).unsqueeze(-1).expand(H, P)
    D_v = torch.from_numpy(D).to(DEV).unsqueeze(-1).expand(H, P)
    A_v = torch.from_numpy(A).to(DEV)[:, None, None].expand(H, P, N)
    pool_d = torch.from_numpy(pool).to(DEV)
    idx = sets[2]
    out = torch.zeros(bs, H, P, dtype=torch.bfloat16, device=DEV)
    op(pool_d, torch.from_numpy(idx).to(DEV), x_v, dt_v, bias_v, A_v, B_v, C_v, D_v, out)
    xs = np.ascontiguousarray(packed[:, :H * P].reshape(bs, H, P))
    Bs = np.ascontiguousarray(packed[:, H * P:H * P + N].reshape(bs, 1, N))
    Cs = np.ascontiguousarray(packed[:, H * P + N:].reshape(bs, 1, N))
    # every request against the oracle
    compare_every_request(pool, idx, xs, dt, dt_bias, A, Bs, Cs, D, pool_d, bits_of(out))
    mask = np.ones(pool.shape[0], bool)
    mask[idx] = False
    keep = torch.from_numpy(np.nonzero(mask)[0]).to(DEV)
    assert torch.equal(pool_d[keep], torch.from_numpy(pool[mask]).to(DEV))


@pytest.mark.parametrize("H", [8, 32, 64, 128])
def test_head_sweep_batch_256(op, H):
    bs = 256
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    n_sets = wl.sets_for_cold_l2(bs, H, l2)
    rng = np.random.default_rng(H)
    pool = wl.state_pool(rng, bs * n_sets, H)
    idx = wl.rotation_sets(bs, n_sets, seed=H)[n_sets - 1]
    dt_bias, A, D = wl.head_params(rng, H)
    x, dt, B, C = wl.request_inputs(rng, bs, H)
    pool_d = torch.from_numpy(pool).to(DEV)
    out = torch.zeros(bs, H, 64, dtype=torch.bfloat16, device=DEV)
    op(pool_d, torch.from_numpy(idx).to(DEV), bf16_tensor(x, DEV), bf16_tensor(dt, DEV),
       torch.from_numpy(dt_bias).to(DEV), torch.from_numpy(A).to(DEV), bf16_tensor(B, DEV),
       bf16_tensor(C, DEV), torch.from_numpy(D).to(DEV), out)
    # every request against the oracle, 16 at a time (128 heads: 1 GiB of fp64 per chunk)
    compare_every_request(pool, idx, x, dt, dt_bias, A, B, C, D, pool_d, bits_of(out),
                          chunk=max(1, 2048 // H))
    mask = np.ones(pool.shape[0], bool)
    mask[idx] = False
    keep = torch.from_numpy(np.nonzero(mask)[0]).to(DEV)
    assert torch.equal(pool_d[keep], torch.from_numpy(pool[mask]).to(DEV))


def test_batch_beyond_one_grid_dimension(op):
    # 70,000 requests: more than one grid dimension holds, so the kernel loops over requests.
    bs = 70000
    pr = wl.make_problem(bs, 1, P=2, pool_size=bs + 10, seed=41)
    t = to_device(pr, DEV)
    _run(op, t)
    assert op.get_error() == (0, -1)
    _compare_all(pr, t, pr.pool)


def test_pool_beyond_2_31_elements(op):
    # 16400 slots x 16 heads x 64 x 128 fp32 (512 KiB per slot) = 8.6 GB: slots from 16384 on
    # start beyond 2^31 elements, so the address arithmetic must be 64-bit.  Only the touched
    # slots hold seeded values (written from the host); the rest is zero and must stay zero.
    slots, H, bs = 16400, 16, 6
    if torch.cuda.get_device_properties(0).total_memory < 32 * 2 ** 30:
        pytest.skip("needs a large device")
    rng = np.random.default_rng(77)
    per_slot = H * 64 * 128
    assert 16384 * per_slot == 2 ** 31
    idx = np.array([16399, 16384, 16383, 16390, 17, 9000], dtype=np.int64)
    sub = wl.state_pool(rng, bs, H)                              # the touched slots' states
    dt_bias, A, D = wl.head_params(rng, H)
    x, dt, B, C = wl.request_inputs(rng, bs, H)
    pool = torch.zeros(slots, H, 64, 128, device=DEV)
    pool[torch.from_numpy(idx).to(DEV)] = torch.from_numpy(sub).to(DEV)
    out = torch.zeros(bs, H, 64, dtype=torch.bfloat16, device=DEV)
    op(pool, torch.from_numpy(idx).to(DEV), bf16_tensor(x, DEV), bf16_tensor(dt, DEV),
       torch.from_numpy(dt_bias).to(DEV), torch.from_numpy(A).to(DEV), bf16_tensor(B, DEV),
       bf16_tensor(C, DEV), torch.from_numpy(D).to(DEV), out)
    torch.cuda.synchronize()
    ref_states, ref_y = oracle_on_requests(sub, np.arange(bs), np.arange(bs), x, dt, dt_bias, A,
                                           B, C, D)
    check_state(pool[torch.from_numpy(idx).to(DEV)].cpu().numpy(), ref_states)
    Ch, Dx = expected_terms(x, D, C, 1, H)
    check_y(bits_of(out), ref_y, ref_states, Ch, Dx, 128)
    mask = torch.ones(slots, dtype=torch.bool, device=DEV)
    mask[torch.from_numpy(idx).to(DEV)] = False
    assert not pool[mask].any()
    del pool
    torch.cuda.empty_cache()


@pytest.mark.parametrize("G", [3, 65535])
def test_most_heads_with_groups(op, G):
    # The largest head count the library accepts (65535), in 3 groups of 21845 heads or one
    # head per group, on the table's 8-rows-per-warp launch (headdim 8): the head's group is
    # h / (H / G) for every head, up to h = 65534.
    H, P, bs = 65535, 8, 2
    rng = np.random.default_rng(G)
    pool = wl.state_pool(rng, bs + 1, H, P=P)                   # slot 1 stays untouched
    idx = np.array([2, 0], dtype=np.int64)
    dt_bias, A, D = wl.head_params(rng, H)
    x, dt, B, C = wl.request_inputs(rng, bs, H, P=P, G=G)
    t = dict(state_pool=torch.from_numpy(pool).to(DEV),
             state_batch_indices=torch.from_numpy(idx).to(DEV).int(),
             x=bf16_tensor(x, DEV), dt=bf16_tensor(dt, DEV),
             dt_bias=torch.from_numpy(dt_bias).to(DEV), A=torch.from_numpy(A).to(DEV),
             B=bf16_tensor(B, DEV), C=bf16_tensor(C, DEV), D=torch.from_numpy(D).to(DEV),
             out=torch.zeros(bs, H, P, dtype=torch.bfloat16, device=DEV))
    _run(op, t)
    torch.cuda.synchronize()
    got = t["state_pool"].cpu().numpy()
    assert np.array_equal(got[1], pool[1])
    ref_states, ref_y = oracle_on_requests(pool, idx, np.arange(bs), x, dt, dt_bias, A, B, C, D,
                                           G)
    check_state(got[idx], ref_states)
    Ch, Dx = expected_terms(x, D, C, G, H)
    check_y(bits_of(t["out"]), ref_y, ref_states, Ch, Dx, 128)
    assert op.get_error() == (0, -1)


def test_degenerate_value_regimes(op):
    # Heads 0-3: dt + dt_bias above 20, where softplus is z itself; heads 4-7: far below zero,
    # so dt is ~1e-13 and dA rounds to 1 (the state carries over); heads 8-11: dt ~10 with
    # A = -16, so dA underflows to 0 in fp32 (the state is replaced by dt x B); heads 12-15 as
    # drawn.  Request 1 has x = 0 (pure decay, readout S'C), request 2 has C = 0 (readout D x).
    pr = wl.make_problem(6, 16, pool_size=9, seed=41)
    pr.dt_bias[0:4] = 25.0
    pr.dt_bias[4:8] = -30.0
    pr.dt_bias[8:12] = 10.0
    pr.A[8:12] = -16.0
    pr.x[1] = 0
    pr.C[2] = 0
    t = to_device(pr, DEV)
    _run(op, t)
    assert op.get_error() == (0, -1)
    _compare_all(pr, t, pr.pool)


def test_launch_override_from_text_and_environment(monkeypatch):
    # "rows,warps" (optionally "vec,rows,warps") forces a shape, "auto"/""/None restores the
    # table; malformed text and shapes the kernels lack are refused and change nothing.  The
    # same text in SSU_LAUNCH is a new handle's initial override; unparsable text there makes
    # ssu_create fail.
    pr = wl.make_problem(5, 16, pool_size=9, seed=13)
    base = ssu.SelectiveStateUpdate(0)
    try:
        t = to_device(pr, DEV)
        shp, _ = ssu.describe(t["state_pool"], t["state_batch_indices"], t["x"], t["dt"],
                              t["dt_bias"], t["A"], t["B"], t["C"], t["D"], t["out"])
        table = ssu.ssu_get_launch(base.handle, shp)
        for text, want in (("8,4", (1, 8, 4, 0)), (" vec, 2 ,16", (1, 2, 16, 0)),
                           ("VEC,1,1", (1, 1, 1, 0)), ("auto", table), ("", table),
                           (None, table)):
            ssu.ssu_set_launch_override(base.handle, text)
            assert ssu.ssu_get_launch(base.handle, shp) == want, text
        ssu.ssu_set_launch_override(base.handle, "4,2")
        for bad, status in (("8", ssu.SSU_ERR_INVALID_ARG), ("8,", ssu.SSU_ERR_INVALID_ARG),
                            ("x,8,4", ssu.SSU_ERR_INVALID_ARG), ("8,4,2", ssu.SSU_ERR_INVALID_ARG),
                            ("3,4", ssu.SSU_ERR_UNSUPPORTED), ("8,17", ssu.SSU_ERR_UNSUPPORTED),
                            ("-8,4", ssu.SSU_ERR_INVALID_ARG)):
            with pytest.raises(ssu.SsuError) as e:
                ssu.ssu_set_launch_override(base.handle, bad)
            assert e.value.status == status, bad
            assert ssu.ssu_get_launch(base.handle, shp) == (1, 4, 2, 0), bad
        _run(base, t)
        _compare_all(pr, t, pr.pool)
    finally:
        base.close()
    monkeypatch.setenv("SSU_LAUNCH", "2,8")
    h = ssu.ssu_create(0)
    try:
        assert ssu.ssu_get_launch(h, shp) == (1, 2, 8, 0)
    finally:
        ssu.ssu_destroy(h)
    monkeypatch.setenv("SSU_LAUNCH", "eight,four")
    with pytest.raises(ssu.SsuError) as e:
        ssu.ssu_create(0)
    assert e.value.status == ssu.SSU_ERR_INVALID_ARG
