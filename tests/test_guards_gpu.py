"""Canary regions around every buffer the kernels write (state pool, readout, intermediate
states, block-copy tensors, host readout, staging workspace): 4 KiB of a fixed byte pattern on
each side must be intact after calls whose requests name the first and last slots and slots
outside the pool.  With compute-sanitizer unavailable, this stands in for its out-of-bounds
write check; the results themselves are compared with unguarded calls bit for bit."""

from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import selective_state_update_02_gb300 as ssu
import workloads as wl
from parity_util import bf16_tensor, bits_of, to_device

pytestmark = pytest.mark.gpu

GUARD = 4096
CANARY = 0xA5


@pytest.fixture(scope="module")
def op():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    o = ssu.SelectiveStateUpdate(0)
    yield o
    o.close()


class Guarded:
    """A tensor of `shape` placed between two canary regions of one allocation."""

    def __init__(self, like: torch.Tensor, pinned: bool = False):
        self.nbytes = like.numel() * like.element_size()
        if pinned:
            self.raw = torch.full((2 * GUARD + self.nbytes,), CANARY, dtype=torch.uint8).pin_memory()
        else:
            self.raw = torch.full((2 * GUARD + self.nbytes,), CANARY, dtype=torch.uint8,
                                  device=like.device)
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(like.dtype).view(like.shape)
        self.t.copy_(like)

    def intact(self) -> bool:
        torch.cuda.synchronize()
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.nbytes:]
        return bool((head == CANARY).all()) and bool((tail == CANARY).all())


def _problem(bs, H, P, N, G, pool_size, dtype, seed):
    pr = wl.make_problem(bs, H, P, N, G, pool_size=pool_size, seed=seed, state_dtype=dtype)
    idx = pr.idx.copy()
    idx[0], idx[1] = 0, pool_size - 1          # the first and the last slot
    idx[2], idx[3] = pool_size, -1             # outside the pool: skipped
    # keep the remaining slots distinct from 0 and pool_size - 1
    rest = np.setdiff1d(np.arange(1, pool_size - 1), idx[:4])
    idx[4:] = rest[:bs - 4]
    pr.idx = idx
    return pr


def _same(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


@pytest.mark.parametrize("N,dtype", [(128, "f32"), (64, "bf16"), (256, "f32"), (256, "bf16")])
def test_decode_step_writes_nothing_outside_its_buffers(op, N, dtype):
    pr = _problem(10, 8, 40, N, 2, 16, dtype, seed=N)
    ref = to_device(pr)
    op(**ref)
    dev = to_device(pr)
    pool, out = Guarded(dev["state_pool"]), Guarded(dev["out"])
    op(pool.t, dev["state_batch_indices"], dev["x"], dev["dt"], dev["dt_bias"], dev["A"],
       dev["B"], dev["C"], dev["D"], out.t)
    assert op.get_error() == (4, 2)            # 2 skipped per call, smallest request 2
    assert pool.intact() and out.intact()
    assert _same(pool.t, ref["state_pool"]) and _same(out.t, ref["out"])


@pytest.mark.parametrize("N,dtype,T", [(128, "f32", 3), (64, "bf16", 2), (256, "f32", 5),
                                       (128, "f32", 11), (64, "f32", 9), (128, "bf16", 17)])
@pytest.mark.parametrize("with_inter", [True, False], ids=["inter", "no_inter"])
def test_multi_token_step_writes_nothing_outside_its_buffers(op, N, dtype, T, with_inter):
    # without intermediate states the longer calls at dstate 64 and 128 run the chunked kernel
    # (headdim 40 is a multiple of 8), whose warps stage their inputs in chunks of 8 tokens
    bs, H, P, G = 10, 8, 40, 2
    pr = _problem(bs, H, P, N, G, 16, dtype, seed=T + N)
    rng = np.random.default_rng(T)
    steps = [wl.request_inputs(rng, bs, H, P, N, G) for _ in range(T)]
    x = bf16_tensor(np.stack([s[0] for s in steps], 1), "cuda")
    dt = bf16_tensor(np.stack([s[1] for s in steps], 1), "cuda")
    B = bf16_tensor(np.stack([s[2] for s in steps], 1), "cuda")
    C = bf16_tensor(np.stack([s[3] for s in steps], 1), "cuda")
    sdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    results = []
    for guarded in (False, True):
        dev = to_device(pr)
        out = torch.zeros(bs, T, H, P, dtype=torch.bfloat16, device="cuda")
        inter = torch.zeros(bs, T, H, P, N, dtype=sdt, device="cuda")
        if guarded:
            gp, go, gi = Guarded(dev["state_pool"]), Guarded(out), Guarded(inter)
            pool, out, inter = gp.t, go.t, gi.t
        else:
            pool = dev["state_pool"]
        op.tokens(pool, dev["state_batch_indices"], x, dt, dev["dt_bias"], dev["A"], B, C,
                  dev["D"], out, inter if with_inter else None)
        assert op.get_error() == (2, 2)
        results.append((pool, out, inter))
    assert gp.intact() and go.intact() and gi.intact()
    for a, b in zip(*results):
        assert _same(a, b)


def test_block_copy_writes_nothing_outside_its_tensors(op):
    rng = np.random.default_rng(3)
    blocks = 9
    tensors = [torch.from_numpy(rng.standard_normal((blocks, 4, 33)).astype(np.float32)).cuda(),
               torch.from_numpy(rng.integers(0, 2**15, (blocks, 40), dtype=np.int16)).cuda()
               .view(torch.bfloat16),
               torch.from_numpy(rng.standard_normal((blocks, 8)).astype(np.float32)).cuda()]
    src = torch.tensor([8, 0, 3, 9], dtype=torch.int32, device="cuda")   # 9: outside
    dst = torch.tensor([0, 8, 5, 1], dtype=torch.int32, device="cuda")
    ref = [t.clone() for t in tensors]
    op.copy_blocks(ref, src, dst)
    guarded = [Guarded(t) for t in tensors]
    op.copy_blocks([g.t for g in guarded], src, dst)
    assert op.get_error()[0] == 2
    for g, r in zip(guarded, ref):
        assert g.intact()
        assert _same(g.t, r)


def test_host_operand_step_writes_nothing_outside_its_buffers(op):
    bs, H, P, N = 10, 8, 40, 128
    pr = _problem(bs, H, P, N, 1, 16, "f32", seed=77)
    ref = to_device(pr)
    op(**ref)
    assert op.get_error() == (2, 2)
    dev = to_device(pr)
    host = {k: dev[k].cpu().pin_memory() for k in ("state_batch_indices", "x", "B", "C")}
    host["dt"] = dev["dt"].cpu().pin_memory()
    out = Guarded(torch.zeros(bs, H, P, dtype=torch.bfloat16), pinned=True)
    pool = Guarded(dev["state_pool"])
    shape, _ = ssu.describe(pool.t, host["state_batch_indices"], host["x"], host["dt"],
                            dev["dt_bias"], dev["A"], host["B"], host["C"], dev["D"], out.t)
    n = ssu.ssu_host_workspace_bytes(shape)
    ws = Guarded(torch.zeros(n, dtype=torch.uint8, device="cuda"))
    ssu.ssu_update_from_host(op.handle, pool.t, host["state_batch_indices"], host["x"],
                             host["dt"], dev["dt_bias"], dev["A"], host["B"], host["C"], dev["D"],
                             out.t, ws.t)
    assert op.get_error() == (2, 2)
    assert pool.intact() and out.intact() and ws.intact()
    assert _same(pool.t, ref["state_pool"])
    live = np.setdiff1d(np.arange(bs), [2, 3])
    assert np.array_equal(bits_of(out.t)[live], bits_of(ref["out"])[live])
    assert math.isclose(float(out.t[[2, 3]].abs().sum()), 0.0)   # skipped rows untouched
