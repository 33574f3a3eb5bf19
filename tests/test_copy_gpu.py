"""GPU parity of the state-block copy (vLLM PR #48110, Purpose) against the oracle's plain
copy: bit-exact for every byte, every launch shape, skipped requests and ragged blocks."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import selective_state_update_02_gb300 as ssu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def op():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    o = ssu.SelectiveStateUpdate(0)
    yield o
    o.close()


def _tensors(rng, specs):
    """Host arrays [num_blocks, ...] of random bits for each (num_blocks, shape, dtype)."""
    out = []
    for nb, shape, dtype in specs:
        n = nb * int(np.prod(shape)) * np.dtype(dtype).itemsize
        raw = rng.integers(0, 256, n, dtype=np.uint8)
        out.append(raw.view(dtype).reshape((nb,) + tuple(shape)))
    return out


TORCH = {np.float32: torch.float32, np.uint16: torch.int16, np.uint8: torch.uint8}


def _to_dev(a):
    t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
    return t.to("cuda")


def _bits(t):
    return t.cpu().numpy()


# a small stand-in of the pages' layout: fp32 temporal blocks and bf16 conv blocks, plus a
# ragged block (not a multiple of the chunk) and a 16-byte block
SPECS = [(12, (8, 128), np.float32), (12, (3, 1280), np.uint16), (12, (4104,), np.float32),
         (12, (4,), np.float32), (12, (2, 16, 128), np.float32)]


def _run_and_compare(op, specs, src, dst, idx_dtype=torch.int32, seed=0):
    rng = np.random.default_rng(seed)
    host = _tensors(rng, specs)
    dev = [_to_dev(a) for a in host]
    op.copy_blocks(dev, torch.tensor(src, dtype=idx_dtype, device="cuda"),
                   torch.tensor(dst, dtype=idx_dtype, device="cuda"))
    torch.cuda.synchronize()
    ref, skipped = oracle.copy_blocks(host, src, dst)
    for a, r in zip(dev, ref):
        got = _bits(a)
        assert np.array_equal(got.view(np.uint8), r.view(np.uint8))
    return skipped


@pytest.mark.parametrize("idx_dtype", [torch.int32, torch.int64])
def test_copy_matches_oracle(op, idx_dtype):
    skipped = _run_and_compare(op, SPECS, [0, 5, 7, 2], [9, 1, 3, 11], idx_dtype)
    assert skipped == 0 and op.get_error() == (0, -1)


COPY_SHAPES = [(ssu.SSU_COPY_VEC, c, v, t) for c in (4, 8, 16, 32, 64) for v in (1, 2, 4, 8, 16)
               for t in (64, 256)]


def test_unknown_copy_mode_is_refused(op):
    with pytest.raises(ssu.SsuError) as e:
        ssu.ssu_copy_set_launch(op.handle, 2, 64, 6, 0)
    assert e.value.status == ssu.SSU_ERR_UNSUPPORTED


def test_every_copy_shape(op):
    try:
        for shape in COPY_SHAPES:
            op_shape = list(shape)
            ssu.ssu_copy_set_launch(op.handle, *op_shape)
            _run_and_compare(op, SPECS, [3, 0, 10, 6, 8], [1, 2, 4, 5, 7], seed=hash(shape) % 97)
        assert op.get_error() == (0, -1)
    finally:
        ssu.ssu_copy_set_launch(op.handle, ssu.SSU_COPY_AUTO)


@pytest.mark.parametrize("vectors", [1, 8])
def test_copy_skips_out_of_range_requests(op, vectors):
    ssu.ssu_copy_set_launch(op.handle, ssu.SSU_COPY_VEC, 8, vectors, 256)
    try:
        # request 1: dst out of range; request 3: negative src
        skipped = _run_and_compare(op, SPECS, [0, 1, 2, -1, 4], [5, 12, 6, 7, 8])
    finally:
        ssu.ssu_copy_set_launch(op.handle, ssu.SSU_COPY_AUTO)
    assert skipped == 2
    assert op.get_error() == (2, 1)


def test_copy_with_no_requests_enqueues_nothing(op):
    assert _run_and_compare(op, SPECS, [], []) == 0


def test_copy_rejects_misaligned_blocks(op):
    t = torch.zeros(8, 6, dtype=torch.int16, device="cuda")        # 12-byte blocks
    with pytest.raises(ssu.SsuError) as e:
        op.copy_blocks([t], torch.tensor([0], device="cuda", dtype=torch.int32),
                       torch.tensor([1], device="cuda", dtype=torch.int32))
    assert e.value.status == ssu.SSU_ERR_MISALIGNED


def test_copy_many_requests_many_tensors(op):
    # 48 tensors as on the pages' hybrid model (24 fp32 temporal + 24 bf16 conv states, scaled
    # down), 40 requests with distinct source and destination blocks.
    specs = [(96, (4, 64, 64), np.float32)] * 24 + [(96, (3, 2560), np.uint16)] * 24
    perm = np.random.default_rng(4).permutation(96)
    skipped = _run_and_compare(op, specs, perm[:40].tolist(), perm[40:80].tolist(), seed=4)
    assert skipped == 0


def test_copy_pages_layout_at_bench_size(op):
    """The bench's workload on the table's launch shape for calls above 1 GiB: 48 tensors (24
    fp32 blocks of 2 MiB, 24 bf16 blocks of 80 KiB per request, as on the vLLM page), 32
    requests (3.3 GB per call), disjoint source and destination sets.  Checked on the device:
    every destination block equals its source block byte for byte, every other block is
    unchanged (compared against a copy taken before the call)."""
    reqs = 32
    blocks = 2 * reqs + 4
    gen = torch.Generator(device="cuda").manual_seed(11)
    tensors = []
    for shape, dtype in [((32, 128, 128), torch.float32)] * 24 + [((10240, 4), torch.bfloat16)] * 24:
        t = torch.empty((blocks,) + shape, dtype=dtype, device="cuda")
        t.uniform_(-1, 1, generator=gen)
        tensors.append(t)
    perm = torch.from_numpy(np.random.default_rng(11).permutation(blocks).astype(np.int32))
    src, dst = perm[:reqs].cuda(), perm[reqs:2 * reqs].cuda()
    rest = perm[2 * reqs:].cuda()
    before_src = [t[src].clone() for t in tensors[:1]]   # spot copy of one tensor's sources
    before_rest = [t[rest].clone() for t in tensors]
    op.copy_blocks(tensors, src, dst)
    torch.cuda.synchronize()
    assert op.get_error() == (0, -1)
    for t, r in zip(tensors, before_rest):
        assert torch.equal(t[dst].view(torch.uint8), t[src].view(torch.uint8))
        assert torch.equal(t[rest].view(torch.uint8), r.view(torch.uint8))
    assert torch.equal(tensors[0][src].view(torch.uint8), before_src[0].view(torch.uint8))
