"""Programmatic dependent launch (ssu_set_pdl) changes timing only: chains of calls that each
read what the previous kernel wrote give bit-identical results with and without it, eagerly
and inside a CUDA graph, including when another kernel rewrites an input between calls."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import selective_state_update_02_gb300 as ssu
import workloads as wl
from parity_util import bf16_tensor, to_device

pytestmark = pytest.mark.gpu


def _chain(pdl: bool, graph: bool, tokens: bool = False, steps: int = 24):
    pr = wl.make_problem(32, 16, pool_size=40, seed=13)
    t = to_device(pr)
    op = ssu.SelectiveStateUpdate(0)
    ssu.ssu_set_pdl(op.handle, pdl)
    outs = torch.zeros(steps, *t["out"].shape, dtype=torch.bfloat16, device="cuda")
    if tokens:
        rng = np.random.default_rng(3)
        xs = bf16_tensor(wl.f32_to_bf16_bits(rng.standard_normal((32, 2, 16, 64),
                                                                  dtype=np.float32)), "cuda")
        dts = bf16_tensor(wl.f32_to_bf16_bits(rng.uniform(-4, 0, (32, 2, 16))
                                              .astype(np.float32)), "cuda")
        Bs = bf16_tensor(wl.f32_to_bf16_bits(rng.standard_normal((32, 2, 1, 128),
                                                                  dtype=np.float32)), "cuda")
        outs = torch.zeros(steps, 32, 2, 16, 64, dtype=torch.bfloat16, device="cuda")

    def body():
        for i in range(steps):
            # another kernel rewrites an input the next call reads
            t["x"].mul_(0.96875)
            if tokens:
                xs.mul_(0.96875)
                op.tokens(t["state_pool"], t["state_batch_indices"], xs, dts, t["dt_bias"],
                          t["A"], Bs, Bs, t["D"], outs[i])
            else:
                op(t["state_pool"], t["state_batch_indices"], t["x"], t["dt"], t["dt_bias"],
                   t["A"], t["B"], t["C"], t["D"], outs[i])

    s = torch.cuda.Stream()
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            body()
        g.replay()
    else:
        with torch.cuda.stream(s):
            body()
    torch.cuda.synchronize()
    assert op.get_error() == (0, -1)
    op.close()
    return t["state_pool"].cpu(), outs.view(torch.int16).cpu()


@pytest.mark.parametrize("graph", [False, True])
@pytest.mark.parametrize("tokens", [False, True])
def test_pdl_chain_is_bit_identical(graph, tokens):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ref_pool, ref_out = _chain(False, graph, tokens)
    pool, out = _chain(True, graph, tokens)
    assert torch.equal(pool, ref_pool)
    assert torch.equal(out, ref_out)
