"""GPU parity of the multi-token step (T consecutive tokens per request) against the oracle,
which applies its pinned single step T times in order."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import selective_state_update_02_gb300 as ssu
import workloads as wl
from parity_util import bf16_tensor, bits_of, check_state, check_y, expected_terms, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def op():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    o = ssu.SelectiveStateUpdate(0)
    yield o
    o.close()


def _tokens_problem(bs, T, H=16, P=64, N=128, G=1, pool_size=None, seed=0):
    pr = wl.make_problem(bs, H, P, N, G, pool_size=pool_size, seed=seed)
    rng = np.random.default_rng(seed + 7)
    steps = [wl.request_inputs(rng, bs, H, P, N, G) for _ in range(T)]
    x = np.stack([s[0] for s in steps], 1)       # [bs, T, H, P]
    dt = np.stack([s[1] for s in steps], 1)      # [bs, T, H]
    B = np.stack([s[2] for s in steps], 1)       # [bs, T, G, N]
    C = np.stack([s[3] for s in steps], 1)
    return pr, x, dt, B, C


def _run(op, pr, x, dt, B, C, idx=None, with_inter=True, idx_dtype=torch.int32):
    dev = to_device(pr, "cuda", idx_dtype)
    if idx is not None:
        dev["state_batch_indices"] = torch.from_numpy(idx).to("cuda").to(idx_dtype)
    bs, T, H, P = x.shape
    out = torch.zeros(bs, T, H, P, dtype=torch.bfloat16, device="cuda")
    inter = (torch.full((bs, T, H, P, pr.pool.shape[3]), 123.0, device="cuda")
             if with_inter else None)
    op.tokens(dev["state_pool"], dev["state_batch_indices"], bf16_tensor(x, "cuda"),
              bf16_tensor(dt, "cuda"), dev["dt_bias"], dev["A"], bf16_tensor(B, "cuda"),
              bf16_tensor(C, "cuda"), dev["D"], out, inter)
    torch.cuda.synchronize()
    return dev["state_pool"].cpu().numpy(), bits_of(out), (inter.cpu().numpy()
                                                           if with_inter else None)


def _check_all(pr, x, dt, B, C, got_pool, got_out, got_inter, idx=None):
    idx = pr.idx if idx is None else idx
    ref_pool, ref_y, ref_inter, skipped = oracle.ssu_tokens(pr.pool, idx, x, dt, pr.dt_bias,
                                                           pr.A, B, C, pr.D, pr.ngroups)
    ok = (idx >= 0) & (idx < pr.pool_size)
    check_state(got_pool[idx[ok]], ref_pool[idx[ok]])
    untouched = np.setdiff1d(np.arange(pr.pool_size), idx[ok])
    assert np.array_equal(got_pool[untouched], pr.pool[untouched])
    T = x.shape[1]
    for t in range(T):
        Ch, Dx = expected_terms(x[ok, t], pr.D, C[ok, t], pr.ngroups, pr.nheads)
        check_y(got_out[ok, t], ref_y[ok, t], ref_inter[ok, t], Ch, Dx, pr.pool.shape[3],
                f"y token {t}")
        if got_inter is not None:
            check_state(got_inter[ok, t], ref_inter[ok, t], f"intermediate token {t}")
    return skipped


def test_one_token_equals_ssu_update_bitwise(op):
    pr, x, dt, B, C = _tokens_problem(12, 1, seed=1)
    got_pool, got_out, _ = _run(op, pr, x, dt, B, C, with_inter=False)
    ref = to_device(pr, "cuda")
    ref["x"], ref["dt"] = bf16_tensor(x[:, 0], "cuda"), bf16_tensor(dt[:, 0], "cuda")
    ref["B"], ref["C"] = bf16_tensor(B[:, 0], "cuda"), bf16_tensor(C[:, 0], "cuda")
    op(ref["state_pool"], ref["state_batch_indices"], ref["x"], ref["dt"], ref["dt_bias"],
       ref["A"], ref["B"], ref["C"], ref["D"], ref["out"])
    torch.cuda.synchronize()
    assert np.array_equal(got_pool, ref["state_pool"].cpu().numpy())
    assert np.array_equal(got_out[:, 0], bits_of(ref["out"]))


# Calls with intermediate states run the general kernel, calls without the rescaling one.
WITH_INTER = pytest.mark.parametrize("with_inter", [True, False], ids=["inter", "no_inter"])


@pytest.mark.parametrize("T", [2, 3, 4, 8])
@pytest.mark.parametrize("idx_dtype", [torch.int32, torch.int64])
@WITH_INTER
def test_tokens_match_oracle(op, T, idx_dtype, with_inter):
    pr, x, dt, B, C = _tokens_problem(10, T, seed=T)
    got = _run(op, pr, x, dt, B, C, idx_dtype=idx_dtype, with_inter=with_inter)
    assert _check_all(pr, x, dt, B, C, *got) == 0
    assert op.get_error() == (0, -1)


@pytest.mark.parametrize("P,G", [(40, 1), (3, 2), (100, 4)])
@WITH_INTER
def test_tokens_ragged_headdim_and_groups(op, P, G, with_inter):
    pr, x, dt, B, C = _tokens_problem(6, 3, H=8, P=P, G=G, seed=P)
    got = _run(op, pr, x, dt, B, C, with_inter=with_inter)
    _check_all(pr, x, dt, B, C, *got)


def test_tokens_without_intermediate(op):
    pr, x, dt, B, C = _tokens_problem(9, 3, seed=11)
    got_pool, got_out, _ = _run(op, pr, x, dt, B, C, with_inter=False)
    _check_all(pr, x, dt, B, C, got_pool, got_out, None)


def test_tokens_skip_out_of_range_requests(op):
    pr, x, dt, B, C = _tokens_problem(8, 3, pool_size=12, seed=5)
    idx = pr.idx.copy()
    idx[[2, 6]] = [12, -3]
    got_pool, got_out, got_inter = _run(op, pr, x, dt, B, C, idx=idx)
    assert _check_all(pr, x, dt, B, C, got_pool, got_out, got_inter, idx) == 2
    assert op.get_error() == (2, 2)
    assert (got_inter[[2, 6]] == 123.0).all() and (got_out[[2, 6]] == 0).all()


def test_tokens_strided_views(op):
    # x, B, C of every token as views into one packed [bs, T, H*P + 2N] bf16 tensor; dt as a
    # head-expanded stride-0 view; per-head operands expanded as in ssu_update's tests.
    bs, T, H, P, N = 7, 3, 16, 64, 128
    pr, _, _, _, _ = _tokens_problem(bs, 1, seed=21)
    rng = np.random.default_rng(22)
    packed = wl.f32_to_bf16_bits(rng.standard_normal((bs, T, H * P + 2 * N), dtype=np.float32))
    dt = wl.f32_to_bf16_bits(rng.uniform(-4, 0, (bs, T, H)).astype(np.float32))
    pk = bf16_tensor(packed, "cuda")
    xv = pk[:, :, :H * P].view(bs, T, H, P)
    Bv = pk[:, :, H * P:H * P + N].unsqueeze(2)
    Cv = pk[:, :, H * P + N:].unsqueeze(2)
    dtv = bf16_tensor(dt, "cuda").unsqueeze(-1).expand(bs, T, H, P)
    dev = to_device(pr, "cuda")
    out = torch.zeros(bs, T, H, P, dtype=torch.bfloat16, device="cuda")
    op.tokens(dev["state_pool"], dev["state_batch_indices"], xv, dtv,
              dev["dt_bias"].unsqueeze(-1).expand(H, P), dev["A"][:, None, None].expand(H, P, N),
              Bv, Cv, dev["D"].unsqueeze(-1).expand(H, P), out)
    torch.cuda.synchronize()
    x = packed[:, :, :H * P].reshape(bs, T, H, P)
    B = packed[:, :, H * P:H * P + N].reshape(bs, T, 1, N)
    C = packed[:, :, H * P + N:].reshape(bs, T, 1, N)
    _check_all(pr, x, dt, B, C, dev["state_pool"].cpu().numpy(), bits_of(out), None)


@pytest.mark.parametrize("T,with_inter", [(3, True), (3, False), (8, False)],
                         ids=["3-inter", "3-no_inter", "8-no_inter"])
def test_tokens_serving_batch_128_every_request(op, T, with_inter):
    # batch 128, 16 heads, 3 tokens per request (one verified token plus two drafts) and 8
    # (the bench's longest), a 2432-slot pool, the built-in launch table: every request's
    # state, readouts and intermediate states (where asked for) against the oracle (in chunks
    # of 32 requests), untouched slots bit-identical.
    bs, H = 128, 16
    rng = np.random.default_rng(3)
    pool = wl.state_pool(rng, 2432, H)
    idx = wl.rotation_sets(bs, 19, seed=3)[4]
    dt_bias, A, D = wl.head_params(rng, H)
    steps = [wl.request_inputs(rng, bs, H) for _ in range(T)]
    x, dt, B, C = (np.stack([s[k] for s in steps], 1) for k in range(4))
    pool_d = torch.from_numpy(pool).cuda()
    out = torch.zeros(bs, T, H, 64, dtype=torch.bfloat16, device="cuda")
    inter = torch.empty(bs, T, H, 64, 128, device="cuda") if with_inter else None
    op.tokens(pool_d, torch.from_numpy(idx).cuda(), bf16_tensor(x, "cuda"), bf16_tensor(dt, "cuda"),
              torch.from_numpy(dt_bias).cuda(), torch.from_numpy(A).cuda(), bf16_tensor(B, "cuda"),
              bf16_tensor(C, "cuda"), torch.from_numpy(D).cuda(), out, inter)
    torch.cuda.synchronize()
    out_bits = bits_of(out)
    for lo in range(0, bs, 32):
        rows = np.arange(lo, lo + 32)
        sub = pool[idx[rows]]
        ref_pool, ref_y, ref_inter, _ = oracle.ssu_tokens(sub, np.arange(len(rows)), x[rows],
                                                         dt[rows], dt_bias, A, B[rows], C[rows],
                                                         D)
        got_pool = pool_d[torch.from_numpy(idx[rows]).cuda()].cpu().numpy()
        check_state(got_pool, ref_pool)
        got_inter = inter[torch.from_numpy(rows).cuda()].cpu().numpy() if with_inter else None
        for t in range(T):
            if with_inter:
                check_state(got_inter[:, t], ref_inter[:, t])
            Ch, Dx = expected_terms(x[rows, t], D, C[rows, t], 1, H)
            check_y(out_bits[rows, t], ref_y[:, t], ref_inter[:, t], Ch, Dx, 128)
    mask = np.ones(2432, bool)
    mask[idx] = False
    keep = torch.from_numpy(np.nonzero(mask)[0]).cuda()
    assert torch.equal(pool_d[keep], torch.from_numpy(pool[mask]).cuda())


@pytest.mark.parametrize("idx_dtype", [torch.int32, torch.int64])
@WITH_INTER
def test_tokens_many_requests_with_skips(op, idx_dtype, with_inter):
    """More requests than the grid's third dimension holds at once in flight, with skipped
    requests scattered among them: every request against the oracle, the skipped ones counted
    and left alone."""
    bs, T, H = 300, 2, 16
    pr, x, dt, B, C = _tokens_problem(bs, T, H=H, pool_size=bs + 40, seed=41)
    idx = pr.idx.copy()
    bad = [0, 7, 150, 151, 299]
    idx[bad] = [bs + 40, -1, -5, 1 << 30, bs + 41]
    got_pool, got_out, got_inter = _run(op, pr, x, dt, B, C, idx=idx, idx_dtype=idx_dtype,
                                        with_inter=with_inter)
    skipped = _check_all(pr, x, dt, B, C, got_pool, got_out, got_inter, idx=idx)
    assert skipped == len(bad)
    assert op.get_error() == (len(bad), 0)
    assert (got_out[bad] == 0).all()
    if with_inter:
        assert (got_inter[bad] == 123.0).all()


@pytest.mark.parametrize("T,N", [(2, 128), (5, 128), (3, 64), (4, 256)])
@WITH_INTER
def test_unaligned_B_C_take_the_scalar_loads_with_the_same_bits(op, T, N, with_inter):
    """B and C one element past an 8-byte boundary (only 2-byte aligned) cannot be read as
    column vectors; the kernel then loads them element by element.  With intermediate states
    both forms run the general kernel and must give the same bits, at several token counts
    (the input ring refills on odd and even tokens).  Without them the aligned call runs the
    chunked kernel (dstate 64 and 128) and the unaligned one the general kernel: both against
    the oracle."""
    bs, H = 10, 8
    pr, x, dt, B, C = _tokens_problem(bs, T, H=H, N=N, seed=T + N)
    aligned_pool, aligned_out, aligned_inter = _run(op, pr, x, dt, B, C, with_inter=with_inter)
    dev = to_device(pr, "cuda")
    out = torch.zeros(bs, T, H, 64, dtype=torch.bfloat16, device="cuda")
    inter = torch.full((bs, T, H, 64, N), 123.0, device="cuda") if with_inter else None
    # [bs, T, 1, N] views at element offset 1 of a wider buffer: 2-byte alignment only
    width = 2 * N + 3
    buf = torch.zeros(bs, T, width, dtype=torch.bfloat16, device="cuda")
    buf[:, :, 1:1 + N] = bf16_tensor(B, "cuda")[:, :, 0]
    buf[:, :, 2 + N:2 + 2 * N] = bf16_tensor(C, "cuda")[:, :, 0]
    Bv = buf[:, :, 1:1 + N].unsqueeze(2)
    Cv = buf[:, :, 2 + N:2 + 2 * N].unsqueeze(2)
    assert Bv.data_ptr() % 8 != 0
    op.tokens(dev["state_pool"], dev["state_batch_indices"], bf16_tensor(x, "cuda"),
              bf16_tensor(dt, "cuda"), dev["dt_bias"], dev["A"], Bv, Cv, dev["D"], out, inter)
    torch.cuda.synchronize()
    if with_inter or N == 256:
        assert np.array_equal(dev["state_pool"].cpu().numpy(), aligned_pool)
        assert np.array_equal(bits_of(out), aligned_out)
        if with_inter:
            assert np.array_equal(inter.cpu().numpy(), aligned_inter)
    else:
        _check_all(pr, x, dt, B, C, aligned_pool, aligned_out, None)
        _check_all(pr, x, dt, B, C, dev["state_pool"].cpu().numpy(), bits_of(out), None)


@WITH_INTER
def test_long_token_runs_cross_the_per_warp_scalar_batches(op, with_inter):
    """dt and dA are computed 32 tokens at a time (one per lane), and a rescaled batch ends
    there; 40 tokens cross a batch."""
    pr, x, dt, B, C = _tokens_problem(3, 40, H=4, seed=21)
    got_pool, got_out, got_inter = _run(op, pr, x, dt, B, C, with_inter=with_inter)
    _check_all(pr, x, dt, B, C, got_pool, got_out, got_inter)


def test_one_token_with_intermediate_runs_the_token_kernel_bitwise(op):
    """T = 1 with an intermediate buffer stays on the multi-token kernel (without one the call
    runs as ssu_update): same bits as ssu_update, and the intermediate is the new state."""
    pr, x, dt, B, C = _tokens_problem(12, 1, seed=2)
    got_pool, got_out, got_inter = _run(op, pr, x, dt, B, C, with_inter=True)
    ref = to_device(pr, "cuda")
    ref["x"], ref["dt"] = bf16_tensor(x[:, 0], "cuda"), bf16_tensor(dt[:, 0], "cuda")
    ref["B"], ref["C"] = bf16_tensor(B[:, 0], "cuda"), bf16_tensor(C[:, 0], "cuda")
    op(ref["state_pool"], ref["state_batch_indices"], ref["x"], ref["dt"], ref["dt_bias"],
       ref["A"], ref["B"], ref["C"], ref["D"], ref["out"])
    torch.cuda.synchronize()
    assert np.array_equal(got_pool, ref["state_pool"].cpu().numpy())
    assert np.array_equal(got_out[:, 0], bits_of(ref["out"]))
    assert np.array_equal(got_inter[:, 0], got_pool[pr.idx])


@pytest.mark.parametrize("N", [128, 256])
@WITH_INTER
def test_most_tokens_per_call(op, N, with_inter):
    """The largest token count one call takes (SSU_MAX_TOKENS = 64): every token's readout and
    intermediate state against the oracle; one more token is refused before any launch."""
    pr = wl.make_problem(3, 4, 64, N, 1, pool_size=5, seed=31)
    rng = np.random.default_rng(38)
    steps = [wl.request_inputs(rng, 3, 4, 64, N, 1) for _ in range(64)]
    x, dt, B, C = (np.stack([s[i] for s in steps], 1) for i in range(4))
    got_pool, got_out, got_inter = _run(op, pr, x, dt, B, C, with_inter=with_inter)
    _check_all(pr, x, dt, B, C, got_pool, got_out, got_inter)
    assert op.get_error() == (0, -1)
    steps.append(wl.request_inputs(rng, 3, 4, 64, N, 1))
    x, dt, B, C = (np.stack([s[i] for s in steps], 1) for i in range(4))
    with pytest.raises(ssu.SsuError) as e:
        _run(op, pr, x, dt, B, C, with_inter=False)
    assert e.value.status == ssu.SSU_ERR_INVALID_ARG


def _extreme_heads(pr, dt, kind):
    """Per-head parameters whose decay products leave the rescaling range [2^-60, 2^60]:
    "underflow": dt near 200, so dA = exp(dt A) is 0 in fp32 from the first token on;
    "growth": A = +1 and every dt = softplus(2.5) = 2.58, so dA = 13.2 and the product of 17
    tokens' dA passes 2^60 (e^43.9 > e^41.6) while the state stays finite (e^46 at most)."""
    if kind == "underflow":
        pr.dt_bias[:] = 200.0
        return dt
    pr.A[:] = 1.0
    pr.dt_bias[:] = 2.5
    return np.zeros_like(dt)


@pytest.mark.parametrize("kind,T", [("underflow", 6), ("growth", 18)])
@WITH_INTER
def test_decay_products_outside_the_chunk_range(op, kind, T, with_inter):
    """Decay products outside [2^-60, 2^60]: without intermediate states (and 5 tokens or more,
    fp32 state) the chunked kernel then runs token by token (a plain update where dA itself is
    out of range, shorter chunks where the running product leaves the range); both kernels
    within the oracle's tolerance."""
    pr, x, dt, B, C = _tokens_problem(6, T, H=8, seed=51 + T)
    dt = _extreme_heads(pr, dt, kind)
    fast_pool, fast_out, _ = _run(op, pr, x, dt, B, C, with_inter=with_inter)
    if kind == "underflow":
        _check_all(pr, x, dt, B, C, fast_pool, fast_out, None)
        return
    # Growth: the state's terms reach e^44, and an entry where they cancel keeps an fp32 error
    # of the terms' size, so the check is relative to each slot's (and readout row's) largest
    # value: fp32 state within 1e-5 of it, bf16 readouts within 2^-7 of it.
    ref_pool, ref_y, _, _ = oracle.ssu_tokens(pr.pool, pr.idx, x, dt, pr.dt_bias, pr.A, B, C,
                                              pr.D, pr.ngroups)
    got = fast_pool[pr.idx].astype(np.float64)
    ref = ref_pool[pr.idx]
    scale = np.abs(ref).max(axis=(2, 3), keepdims=True)
    assert (np.abs(got - ref) <= 1e-5 * (1 + scale)).all()
    y = oracle.bf16_to_f64(fast_out)
    yscale = np.abs(ref_y).max(axis=-1, keepdims=True)
    assert (np.abs(y - ref_y) <= 2.0 ** -7 * yscale).all()


def test_heads_in_and_out_of_the_chunk_range_in_one_call(op):
    """Half the heads decay so fast (dA = 0) that every token of theirs takes the plain
    update alone, the others run in chunks: every readout and state against the oracle."""
    pr, x, dt, B, C = _tokens_problem(6, 6, H=8, seed=61)
    pr.dt_bias[::2] = 200.0
    got_pool, got_out, _ = _run(op, pr, x, dt, B, C, with_inter=False)
    _check_all(pr, x, dt, B, C, got_pool, got_out, None)


@pytest.mark.parametrize("P,G,T", [(40, 4, 6), (96, 2, 9), (128, 1, 5), (8, 2, 7)])
def test_chunked_kernel_headdim_groups_and_chunks(op, P, G, T):
    """The chunked kernel (no intermediate states, fp32 state, 5 tokens or more) on head groups,
    a headdim that ends inside a warp's 16 rows (40, 8), two 64-row slabs per head (96, 128)
    and a second chunk (9 tokens): every readout and state against the oracle."""
    pr, x, dt, B, C = _tokens_problem(5, T, H=8, P=P, G=G, seed=70 + P + T)
    got = _run(op, pr, x, dt, B, C, with_inter=False)
    assert _check_all(pr, x, dt, B, C, *got) == 0


def test_chunked_kernel_on_packed_strided_views(op):
    """x, B and C of 6 tokens as views into one packed [bs, T, H*P + 2N] bf16 tensor (16-byte
    aligned, strides multiples of 8 elements), dt and the per-head operands as stride-0
    expansions: the chunked kernel reads them in place."""
    bs, T, H, P, N = 7, 6, 16, 64, 128
    pr, _, _, _, _ = _tokens_problem(bs, 1, seed=23)
    rng = np.random.default_rng(24)
    packed = wl.f32_to_bf16_bits(rng.standard_normal((bs, T, H * P + 2 * N), dtype=np.float32))
    dt = wl.f32_to_bf16_bits(rng.uniform(-4, 0, (bs, T, H)).astype(np.float32))
    pk = bf16_tensor(packed, "cuda")
    xv = pk[:, :, :H * P].view(bs, T, H, P)
    Bv = pk[:, :, H * P:H * P + N].unsqueeze(2)
    Cv = pk[:, :, H * P + N:].unsqueeze(2)
    assert Bv.data_ptr() % 16 == 0 and Cv.data_ptr() % 16 == 0
    dtv = bf16_tensor(dt, "cuda").unsqueeze(-1).expand(bs, T, H, P)
    dev = to_device(pr, "cuda")
    out = torch.zeros(bs, T, H, P, dtype=torch.bfloat16, device="cuda")
    op.tokens(dev["state_pool"], dev["state_batch_indices"], xv, dtv,
              dev["dt_bias"].unsqueeze(-1).expand(H, P), dev["A"][:, None, None].expand(H, P, N),
              Bv, Cv, dev["D"].unsqueeze(-1).expand(H, P), out)
    torch.cuda.synchronize()
    x = packed[:, :, :H * P].reshape(bs, T, H, P)
    B = packed[:, :, H * P:H * P + N].reshape(bs, T, 1, N)
    C = packed[:, :, H * P + N:].reshape(bs, T, 1, N)
    _check_all(pr, x, dt, B, C, dev["state_pool"].cpu().numpy(), bits_of(out), None)


def _fuzz_cases(n=40, seed=2026):
    """Seeded random shapes that the chunked kernel takes (no intermediate states, headdim a
    multiple of 8): fp32 state at dstate 64 / 128 from 5 tokens, bf16 at dstate 128 from 16."""
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        bf16 = i % 8 == 7
        N = 128 if bf16 else int(rng.choice([64, 128]))
        T = int(rng.integers(16, 25)) if bf16 else int(rng.integers(5, 25))
        H = int(rng.choice([1, 2, 3, 4, 6, 8]))
        G = int(rng.choice([g for g in (1, 2, 3) if H % g == 0]))
        P = int(rng.choice([8, 16, 24, 40, 64, 72, 96, 128]))
        bs = int(rng.integers(1, 24))
        cases.append((i, bs, T, H, G, P, N, "bf16" if bf16 else "f32", bool(rng.integers(0, 2))))
    return cases


@pytest.mark.parametrize("case", _fuzz_cases(), ids=lambda c: f"case{c[0]}")
def test_chunked_kernel_random_shapes(op, case):
    """Every request of a random call against the oracle (shape, groups, token count across
    chunk boundaries, index width and state type drawn from one seeded generator)."""
    i, bs, T, H, G, P, N, sdt, i64 = case
    pr = wl.make_problem(bs, H, P, N, G, pool_size=bs + 5, seed=1000 + i, state_dtype=sdt)
    rng = np.random.default_rng(2000 + i)
    steps = [wl.request_inputs(rng, bs, H, P, N, G) for _ in range(T)]
    x, dt, B, C = (np.stack([s[k] for s in steps], 1) for k in range(4))
    dev = to_device(pr, "cuda", torch.int64 if i64 else torch.int32)
    out = torch.zeros(bs, T, H, P, dtype=torch.bfloat16, device="cuda")
    op.tokens(dev["state_pool"], dev["state_batch_indices"], bf16_tensor(x, "cuda"),
              bf16_tensor(dt, "cuda"), dev["dt_bias"], dev["A"], bf16_tensor(B, "cuda"),
              bf16_tensor(C, "cuda"), dev["D"], out)
    torch.cuda.synchronize()
    untouched = np.setdiff1d(np.arange(pr.pool.shape[0]), pr.idx)
    if sdt == "bf16":
        from parity_util import ulp_bf16
        bits = dev["state_pool"].cpu().view(torch.int16).numpy().view(np.uint16)
        ref_pool, ref_y, ref_inter, _ = oracle.ssu_tokens(oracle.bf16_to_f64(pr.pool), pr.idx,
                                                         x, dt, pr.dt_bias, pr.A, B, C, pr.D, G)
        got, ref = oracle.bf16_to_f64(bits[pr.idx]), ref_pool[pr.idx]
        # the stored state is the fp32 one rounded to bf16: half a bf16 step on top of the fp32
        # state's 1e-5 (1 + |ref|)
        excess = np.maximum(np.abs(got - ref) - 0.5 * ulp_bf16(ref), 0.0)
        assert (excess / (1.0 + np.abs(ref))).max() <= 1e-5
        assert np.array_equal(bits[untouched], pr.pool[untouched])
    else:
        ref_pool, ref_y, ref_inter, _ = oracle.ssu_tokens(pr.pool, pr.idx, x, dt, pr.dt_bias,
                                                         pr.A, B, C, pr.D, G)
        got = dev["state_pool"].cpu().numpy()
        check_state(got[pr.idx], ref_pool[pr.idx])
        assert np.array_equal(got[untouched], pr.pool[untouched])
    out_bits = bits_of(out)
    for t in range(T):
        Ch, Dx = expected_terms(x[:, t], pr.D, C[:, t], G, H)
        check_y(out_bits[:, t], ref_y[:, t], ref_inter[:, t], Ch, Dx, N, f"y token {t}")
    assert op.get_error() == (0, -1)
