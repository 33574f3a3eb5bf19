"""ssu_update_from_host: the per-step operands (indices, x, dt, B, C) and the readout in
page-locked host memory.  The step runs the same decode-step kernel on staged copies, so every
case is compared bit for bit with ssu_update on device copies of the same values (itself
checked against the oracle in test_parity_gpu.py), and one case directly with the oracle."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import selective_state_update_02_gb300 as ssu
import workloads as wl
from parity_util import (bits_of, check_state, check_y, expected_terms, oracle_on_requests,
                         pool_host, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def handle():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    h = ssu.ssu_create(0)
    yield h
    ssu.ssu_destroy(h)


def host_operands(pr, packed: bool, i64: bool, out_pad: int = 0):
    """Pinned host tensors for the per-step operands of ``pr`` (and a pinned ``out``).

    ``packed``: x, B and C are strided views of one pinned [bs, H*P + 2*G*N] bf16 buffer and
    dt a head-expanded view (stride 0 over headdim); ``out_pad`` > 0 makes ``out`` a strided
    view with a row pitch of P + out_pad elements."""
    bs, H, P = pr.x.shape
    G, N = pr.B.shape[1], pr.B.shape[2]
    idx = torch.from_numpy(pr.idx).to(torch.int64 if i64 else torch.int32).pin_memory()
    dt = torch.from_numpy(pr.dt.view(np.int16)).view(torch.bfloat16).pin_memory()
    if packed:
        width = H * P + 2 * G * N
        buf = torch.empty(bs, width, dtype=torch.bfloat16).pin_memory()
        bits = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
        buf[:, :H * P] = bits(pr.x).reshape(bs, H * P)
        buf[:, H * P:H * P + G * N] = bits(pr.B).reshape(bs, G * N)
        buf[:, H * P + G * N:] = bits(pr.C).reshape(bs, G * N)
        x = buf[:, :H * P].view(bs, H, P)
        B = buf[:, H * P:H * P + G * N].view(bs, G, N)
        C = buf[:, H * P + G * N:].view(bs, G, N)
        dt = dt.unsqueeze(-1).expand(bs, H, P)
    else:
        x = torch.from_numpy(pr.x.view(np.int16)).view(torch.bfloat16).pin_memory()
        B = torch.from_numpy(pr.B.view(np.int16)).view(torch.bfloat16).pin_memory()
        C = torch.from_numpy(pr.C.view(np.int16)).view(torch.bfloat16).pin_memory()
    out_full = torch.full((bs, H, P + out_pad), -1.0, dtype=torch.bfloat16).pin_memory()
    out = out_full[..., :P]
    return dict(state_batch_indices=idx, x=x, dt=dt, B=B, C=C, out=out)


def workspace_for(dev_ops, host_ops):
    shape, _ = ssu.describe(dev_ops["state_pool"], host_ops["state_batch_indices"],
                            host_ops["x"], host_ops["dt"], dev_ops["dt_bias"], dev_ops["A"],
                            host_ops["B"], host_ops["C"], dev_ops["D"], host_ops["out"])
    n = ssu.ssu_host_workspace_bytes(shape)
    return torch.empty(max(n, 256), dtype=torch.uint8, device="cuda")


def run_both(handle, pr, packed, i64, out_pad=0, ws=None):
    """ssu_update on device copies and ssu_update_from_host on pinned host copies of ``pr``;
    returns (reference device operands, host-path device operands, host operands)."""
    ref = to_device(pr, "cuda", torch.int64 if i64 else torch.int32)
    dev = to_device(pr, "cuda", torch.int64 if i64 else torch.int32)
    hop = host_operands(pr, packed, i64, out_pad)
    ws = workspace_for(dev, hop) if ws is None else ws
    ssu.ssu_update(handle, **ref)
    ssu.ssu_update_from_host(handle, dev["state_pool"], hop["state_batch_indices"], hop["x"],
                             hop["dt"], dev["dt_bias"], dev["A"], hop["B"], hop["C"], dev["D"],
                             hop["out"], ws)
    torch.cuda.synchronize()
    return ref, dev, hop


def assert_same(ref, dev, hop):
    assert torch.equal(ref["state_pool"].view(torch.uint8),
                       dev["state_pool"].view(torch.uint8)), "state differs"
    got = bits_of(hop["out"])
    want = bits_of(ref["out"])
    assert np.array_equal(got, want), "readout differs"


CASES = [
    # bs, H, P, N, G, state, i64, packed, out_pad
    (8, 16, 64, 128, 1, "f32", False, False, 0),
    (128, 16, 64, 128, 1, "f32", False, True, 0),
    (5, 6, 40, 64, 2, "bf16", True, True, 8),
    (3, 4, 24, 256, 1, "f32", True, False, 3),
    (70, 8, 64, 128, 1, "bf16", False, True, 0),
    (1, 2, 3, 128, 2, "f32", False, True, 1),
    # past the 65,535 CTAs of the grid's third dimension (the staging kernel loops)
    (70_000, 1, 16, 64, 1, "f32", False, True, 0),
]


@pytest.mark.parametrize("bs,H,P,N,G,state,i64,packed,out_pad", CASES)
def test_matches_ssu_update_bit_for_bit(handle, bs, H, P, N, G, state, i64, packed, out_pad):
    pr = wl.make_problem(bs, H, P, N, G, pool_size=bs + 9, seed=bs * 7 + P, state_dtype=state)
    ref, dev, hop = run_both(handle, pr, packed, i64, out_pad)
    assert_same(ref, dev, hop)
    if out_pad:
        pad = hop["out"].as_strided((bs, H, out_pad), (H * (P + out_pad), P + out_pad, 1),
                                    hop["out"].storage_offset() + P)
        assert bool((pad == -1.0).all()), "bytes between out rows were written"


def test_against_the_oracle(handle):
    pr = wl.make_problem(8, 16, pool_size=32, seed=0)
    pool0 = pr.pool.copy()
    _, dev, hop = run_both(handle, pr, packed=True, i64=False)
    rows = np.arange(8)
    new_ref, y_ref = oracle_on_requests(pool0, pr.idx, rows, pr.x, pr.dt, pr.dt_bias, pr.A,
                                        pr.B, pr.C, pr.D)
    got_pool = pool_host(dev["state_pool"])
    check_state(got_pool[pr.idx], new_ref)
    Ch, Dx = expected_terms(pr.x, pr.D, pr.C, 1, 16)
    check_y(bits_of(hop["out"]), y_ref, new_ref, Ch, Dx, 128)
    untouched = np.setdiff1d(np.arange(32), pr.idx)
    assert np.array_equal(got_pool[untouched], pool0[untouched])


@pytest.mark.parametrize("pdl", [False, True])
def test_consecutive_steps_reuse_one_workspace(handle, pdl):
    """Three steps on one pool, new host inputs each step, one workspace: each step's staging
    must wait for the previous step's kernel to finish reading the workspace."""
    bs, H = 32, 16
    pr = wl.make_problem(bs, H, pool_size=48, seed=5)
    ref = to_device(pr, "cuda")
    dev = to_device(pr, "cuda")
    rng = np.random.default_rng(17)
    steps = []
    for _ in range(3):
        x, dt, B, C = wl.request_inputs(rng, bs, H)
        step = wl.Problem(pr.pool, pr.idx, x, dt, pr.dt_bias, pr.A, B, C, pr.D, 1)
        steps.append(host_operands(step, packed=True, i64=False))
    ws = workspace_for(dev, steps[0])
    ssu.ssu_set_pdl(handle, pdl)
    try:
        for hop in steps:            # enqueued back to back, no synchronisation between
            ssu.ssu_update_from_host(handle, dev["state_pool"], hop["state_batch_indices"],
                                     hop["x"], hop["dt"], dev["dt_bias"], dev["A"], hop["B"],
                                     hop["C"], dev["D"], hop["out"], ws)
        torch.cuda.synchronize()
    finally:
        ssu.ssu_set_pdl(handle, True)  # the default
    for hop in steps:
        r = dict(ref)
        r.update({k: hop[k].cuda() for k in ("state_batch_indices", "x", "B", "C")})
        r["dt"] = hop["dt"][..., 0].cuda()                 # [bs, H]: the stride-0 form
        r["out"] = torch.empty_like(ref["out"])
        ssu.ssu_update(handle, **r)
        torch.cuda.synchronize()
        assert np.array_equal(bits_of(hop["out"]), bits_of(r["out"]))
    assert torch.equal(ref["state_pool"], dev["state_pool"])


def test_skipped_requests_are_counted(handle):
    bs = 12
    pr = wl.make_problem(bs, 16, pool_size=20, seed=3)
    pr.idx[[2, 9]] = [20, -1]
    ssu.ssu_get_error(handle)                  # start from cleared counters
    pool0 = pr.pool.copy()
    ref, dev, hop = run_both(handle, pr, packed=False, i64=True)
    # both calls counted their two skipped requests (the counters accumulate until read)
    assert ssu.ssu_get_error(handle) == (4, 2)
    assert torch.equal(ref["state_pool"], dev["state_pool"])
    live = np.setdiff1d(np.arange(bs), [2, 9])
    assert np.array_equal(bits_of(hop["out"])[live], bits_of(ref["out"])[live])
    # skipped requests leave their out rows untouched (the pinned buffer started at -1.0)
    assert bool((hop["out"][[2, 9]] == -1.0).all())
    untouched = np.setdiff1d(np.arange(20), pr.idx[live])
    assert np.array_equal(pool_host(dev["state_pool"])[untouched], pool0[untouched])


def test_device_operands_are_accepted(handle):
    pr = wl.make_problem(16, 16, pool_size=24, seed=8)
    ref = to_device(pr, "cuda")
    dev = to_device(pr, "cuda")
    ws = workspace_for(dev, dev)
    ssu.ssu_update(handle, **ref)
    ssu.ssu_update_from_host(handle, dev["state_pool"], dev["state_batch_indices"], dev["x"],
                             dev["dt"], dev["dt_bias"], dev["A"], dev["B"], dev["C"], dev["D"],
                             dev["out"], ws)
    torch.cuda.synchronize()
    assert torch.equal(ref["state_pool"], dev["state_pool"])
    assert torch.equal(ref["out"].view(torch.int16), dev["out"].view(torch.int16))


def test_graph_capture_replays_the_same_steps(handle):
    bs, H, n = 24, 16, 3
    pr = wl.make_problem(bs, H, pool_size=bs * n, seed=11)
    dev = to_device(pr, "cuda")
    eager = to_device(pr, "cuda")
    sets = np.random.default_rng(2).permutation(bs * n).reshape(n, bs)
    rng = np.random.default_rng(4)
    hops = []
    for k in range(n):
        x, dt, B, C = wl.request_inputs(rng, bs, H)
        hops.append(host_operands(wl.Problem(pr.pool, sets[k], x, dt, pr.dt_bias, pr.A, B, C,
                                             pr.D, 1), packed=True, i64=False))
    ws = workspace_for(dev, hops[0])
    outs_eager = []
    for hop in hops:
        ssu.ssu_update_from_host(handle, eager["state_pool"], hop["state_batch_indices"],
                                 hop["x"], hop["dt"], eager["dt_bias"], eager["A"], hop["B"],
                                 hop["C"], eager["D"], hop["out"], ws)
        torch.cuda.synchronize()
        outs_eager.append(bits_of(hop["out"]).copy())
        hop["out"].fill_(0)
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for hop in hops:
            ssu.ssu_update_from_host(handle, dev["state_pool"], hop["state_batch_indices"],
                                     hop["x"], hop["dt"], dev["dt_bias"], dev["A"], hop["B"],
                                     hop["C"], dev["D"], hop["out"], ws,
                                     stream=torch.cuda.current_stream())
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager["state_pool"], dev["state_pool"])
    for hop, want in zip(hops, outs_eager):
        assert np.array_equal(bits_of(hop["out"]), want)


def test_rejections_before_any_launch(handle):
    pr = wl.make_problem(4, 16, pool_size=8, seed=1)
    dev = to_device(pr, "cuda")
    hop = host_operands(pr, packed=False, i64=False)
    ws = workspace_for(dev, hop)
    args = lambda **kw: {**dict(state_pool=dev["state_pool"], **{k: hop[k] for k in hop},
                                dt_bias=dev["dt_bias"], A=dev["A"], D=dev["D"], workspace=ws),
                         **kw}

    def call(**kw):
        a = args(**kw)
        ssu.ssu_update_from_host(handle, a["state_pool"], a["state_batch_indices"], a["x"],
                                 a["dt"], a["dt_bias"], a["A"], a["B"], a["C"], a["D"],
                                 a["out"], a["workspace"])

    pool0 = dev["state_pool"].clone()
    pageable = torch.from_numpy(pr.x.view(np.int16)).view(torch.bfloat16).clone()
    assert not pageable.is_pinned()
    with pytest.raises(ssu.SsuError) as e:
        call(x=pageable)
    assert e.value.status == ssu.SSU_ERR_INVALID_ARG and "pageable" in ssu.last_error()
    with pytest.raises(ssu.SsuError) as e:
        call(workspace=ws[:64])
    assert e.value.status == ssu.SSU_ERR_INVALID_ARG and "workspace" in ssu.last_error()
    with pytest.raises(ssu.SsuError) as e:
        call(workspace=ws[16:])
    assert e.value.status == ssu.SSU_ERR_MISALIGNED
    torch.cuda.synchronize()
    assert torch.equal(pool0, dev["state_pool"])          # nothing was launched


@pytest.mark.parametrize("i64", [False, True])
def test_strided_index_and_dt_views(handle, i64):
    """Indices every other element of a wider pinned array, dt a [bs, H] view with head
    stride 2: the staging jobs gather them; the step matches ssu_update on dense copies."""
    bs, H = 12, 8
    pr = wl.make_problem(bs, H, pool_size=20, seed=61)
    ref = to_device(pr, "cuda", torch.int64 if i64 else torch.int32)
    dev = to_device(pr, "cuda", torch.int64 if i64 else torch.int32)
    hop = host_operands(pr, packed=True, i64=i64)
    wide_idx = torch.zeros(2 * bs, dtype=hop["state_batch_indices"].dtype).pin_memory()
    wide_idx[::2] = hop["state_batch_indices"]
    wide_idx[1::2] = -7                       # never read
    hop["state_batch_indices"] = wide_idx[::2]
    wide_dt = torch.zeros(bs, 2 * H, dtype=torch.bfloat16).pin_memory()
    wide_dt[:, ::2] = torch.from_numpy(pr.dt.view(np.int16)).view(torch.bfloat16)
    hop["dt"] = wide_dt[:, ::2]
    assert hop["state_batch_indices"].stride(0) == 2 and hop["dt"].stride(1) == 2
    ws = workspace_for(dev, hop)
    ssu.ssu_update(handle, **ref)
    ssu.ssu_update_from_host(handle, dev["state_pool"], hop["state_batch_indices"], hop["x"],
                             hop["dt"], dev["dt_bias"], dev["A"], hop["B"], hop["C"], dev["D"],
                             hop["out"], ws)
    torch.cuda.synchronize()
    assert_same(ref, dev, hop)
    assert ssu.ssu_get_error(handle) == (0, -1)
