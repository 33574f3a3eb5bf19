"""The C ABI without a GPU: the library loads, exports what include/ssu.h declares, and its
host-side validation returns the documented codes (pointers are never dereferenced)."""

from __future__ import annotations

import ctypes
import re
import subprocess
from pathlib import Path

import pytest
import torch

ROOT = Path(__file__).resolve().parent.parent
HEADER = ROOT / "include" / "ssu.h"


@pytest.fixture(scope="module")
def ssu():
    from selective_state_update_02_gb300 import _build
    _build.build()
    import selective_state_update_02_gb300 as m
    m.lib()
    return m


def declared_functions() -> list[str]:
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(ssu_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("ssu_create", "ssu_update", "ssu_destroy", "ssu_get_error", "ssu_validate",
                 "ssu_set_launch", "ssu_set_launch_override", "ssu_get_launch"):
        assert must in names


def test_library_exports_every_declared_symbol(ssu):
    from selective_state_update_02_gb300 import LIB_PATH
    dyn = subprocess.run(["nm", "-D", "--defined-only", str(LIB_PATH)], capture_output=True,
                         text=True, check=True).stdout
    exported = set(line.split()[-1] for line in dyn.splitlines() if line.strip())
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(ssu.lib(), name)


def test_binding_covers_every_declared_function(ssu):
    for name in declared_functions():
        assert name in ssu._EXPORTS, name


def test_version_and_status_strings(ssu):
    assert ssu.ssu_abi_version() == 2 == ssu.SSU_ABI_VERSION
    assert ssu.status_string(ssu.SSU_ERR_MISALIGNED) == "SSU_ERR_MISALIGNED"
    assert ssu.status_string(99) == "SSU_ERR_UNKNOWN"


def test_struct_layout_matches_header(ssu):
    assert ctypes.sizeof(ssu.ssu_shape_t) == 6 * 8 + 2 * 4
    assert ctypes.sizeof(ssu.ssu_strides_t) == (4 + 3 + 3 + 3 + 3 + 3 + 2 + 2 + 3 + 1) * 8
    assert ctypes.sizeof(ssu.ssu_launch_t) == 16


# ---- host validation -------------------------------------------------------------------

BASE = 1 << 32  # fake, 256-byte aligned device addresses: never dereferenced


def canonical(bs=8, H=16, P=64, N=128, G=1, pool=32, i64=False):
    s = __import__("selective_state_update_02_gb300")
    shape = s.ssu_shape_t(bs, H, P, N, G, pool, 1 if i64 else 0, 0)
    st = s.ssu_strides_t()
    st.state[:] = [H * P * N, P * N, N, 1]
    st.x[:] = [H * P, P, 1]
    st.out[:] = [H * P, P, 1]
    st.dt[:] = [H, 1, 0]
    st.B[:] = [G * N, N, 1]
    st.C[:] = [G * N, N, 1]
    st.dt_bias[:] = [1, 0]
    st.D[:] = [1, 0]
    st.A[:] = [1, 0, 0]
    st.idx = 1
    ptrs = [BASE + k * (1 << 28) for k in range(10)]
    return ptrs, shape, st


def validate(ssu, ptrs, shape, st):
    return ssu.ssu_validate(*ptrs, shape=shape, strides=st)


def test_valid_call_passes(ssu):
    assert validate(ssu, *canonical()) == ssu.SSU_OK
    assert validate(ssu, *canonical(i64=True)) == ssu.SSU_OK
    assert validate(ssu, *canonical(P=3)) == ssu.SSU_OK          # ragged headdim is fine


def test_empty_batch_needs_no_pointers(ssu):
    ptrs, shape, st = canonical(bs=0)
    assert validate(ssu, [None] * 10, shape, st) == ssu.SSU_OK


@pytest.mark.parametrize("mutate,code", [
    (lambda p, s, t: p.__setitem__(2, None), "INVALID_ARG"),
    (lambda p, s, t: setattr(s, "batch", -1), "INVALID_ARG"),
    (lambda p, s, t: setattr(s, "ngroups", 3), "INVALID_ARG"),           # 16 % 3 != 0
    (lambda p, s, t: setattr(s, "index_dtype", 7), "INVALID_ARG"),
    (lambda p, s, t: setattr(s, "dstate", 96), "UNSUPPORTED"),
    (lambda p, s, t: setattr(s, "state_dtype", 5), "INVALID_ARG"),
    (lambda p, s, t: t.state.__setitem__(3, 2), "UNSUPPORTED"),
    (lambda p, s, t: t.state.__setitem__(2, 130), "MISALIGNED"),
    (lambda p, s, t: p.__setitem__(0, BASE + 4), "MISALIGNED"),
    (lambda p, s, t: p.__setitem__(2, BASE + 1), "MISALIGNED"),          # odd bf16 address
    (lambda p, s, t: t.dt.__setitem__(2, 1), "UNSUPPORTED"),
    (lambda p, s, t: t.A.__setitem__(2, 1), "UNSUPPORTED"),
    (lambda p, s, t: t.dt_bias.__setitem__(1, 1), "UNSUPPORTED"),
    (lambda p, s, t: t.x.__setitem__(2, 2), "UNSUPPORTED"),
    (lambda p, s, t: t.B.__setitem__(0, -1), "INVALID_ARG"),
    (lambda p, s, t: setattr(t, "idx", -1), "INVALID_ARG"),
])
def test_invalid_calls_return_their_code(ssu, mutate, code):
    ptrs, shape, st = canonical()
    mutate(ptrs, shape, st)
    assert validate(ssu, ptrs, shape, st) == getattr(ssu, "SSU_ERR_" + code)
    assert ssu.last_error() != ""


def test_other_dstate_buckets_and_bf16_state(ssu):
    for N in (64, 256):
        assert validate(ssu, *canonical(N=N)) == ssu.SSU_OK
    ptrs, shape, st = canonical()
    shape.state_dtype = ssu.SSU_STATE_BF16
    assert validate(ssu, ptrs, shape, st) == ssu.SSU_OK
    st.state[2] = 132            # 264 bytes: not a multiple of 16 for bf16 rows
    assert validate(ssu, ptrs, shape, st) == ssu.SSU_ERR_MISALIGNED
    shape.state_dtype = ssu.SSU_STATE_F32
    assert validate(ssu, ptrs, shape, st) == ssu.SSU_OK   # 528 bytes for fp32


def test_i64_indices_must_be_8_byte_aligned(ssu):
    ptrs, shape, st = canonical(i64=True)
    ptrs[1] = BASE + 4
    assert validate(ssu, ptrs, shape, st) == ssu.SSU_ERR_MISALIGNED


def test_null_handle_is_rejected_before_any_cuda_call(ssu):
    ptrs, shape, st = canonical()
    assert ssu.ssu_update_raw(None, ptrs, shape, st, None) == ssu.SSU_ERR_INVALID_ARG
    assert ssu.lib().ssu_set_launch(None, None) == ssu.SSU_ERR_INVALID_ARG
    assert ssu.lib().ssu_set_launch_override(None, b"8,4") == ssu.SSU_ERR_INVALID_ARG
    assert ssu.lib().ssu_destroy(None) == ssu.SSU_OK


def test_static_counters_out_is_checked_before_the_call(ssu):
    # counters_out receives a 12-byte device copy: a CPU tensor, a 2-byte dtype, a float
    # dtype or fewer than 3 elements are refused in Python, before the library is called.
    bs, H, P, N = 2, 2, 8, 128
    pool = torch.zeros(4, H, P, N)
    x = torch.zeros(bs, H, P, dtype=torch.bfloat16)
    bc = torch.zeros(bs, 1, N, dtype=torch.bfloat16)
    args = (pool, torch.arange(bs, dtype=torch.int32), x, torch.zeros(bs, H, dtype=torch.bfloat16),
            torch.zeros(H), torch.zeros(H), bc, bc, torch.zeros(H), torch.zeros_like(x))
    for bad in (torch.zeros(3, dtype=torch.int32), torch.zeros(3, dtype=torch.int16),
                torch.zeros(3, dtype=torch.float32), torch.zeros(2, dtype=torch.int32)):
        with pytest.raises(ValueError):
            ssu.ssu_update_static(*args, counters_out=bad)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_create_without_a_device_fails_cleanly(ssu):
    with pytest.raises(ssu.SsuError) as e:
        ssu.ssu_create(0)
    assert e.value.status == ssu.SSU_ERR_CUDA


# ---- marshalling of tensors into the ABI structs -----------------------------------------

def test_describe_packed_views_and_broadcasts(ssu):
    bs, H, P, N = 6, 16, 64, 128
    pool = torch.zeros(10, H, P, N)
    packed = torch.zeros(bs, H * P + 2 * N, dtype=torch.bfloat16)
    x = packed[:, :H * P].view(bs, H, P)
    B = packed[:, H * P:H * P + N].unsqueeze(1)
    C = packed[:, H * P + N:].unsqueeze(1)
    dt = torch.zeros(bs, H, dtype=torch.bfloat16).unsqueeze(-1).expand(bs, H, P)
    bias = torch.zeros(H).unsqueeze(-1).expand(H, P)
    A = torch.zeros(H)[:, None, None].expand(H, P, N)
    D = torch.zeros(H)
    out = torch.zeros(bs, H, P, dtype=torch.bfloat16)
    idx = torch.arange(bs, dtype=torch.int64)
    shape, st = ssu.describe(pool, idx, x, dt, bias, A, B, C, D, out)
    assert (shape.batch, shape.nheads, shape.headdim, shape.dstate, shape.ngroups,
            shape.pool_size, shape.index_dtype) == (bs, H, P, N, 1, 10, 1)
    assert list(st.x) == [H * P + 2 * N, P, 1]
    assert list(st.B)[0] == H * P + 2 * N and list(st.B)[2] == 1
    assert list(st.dt) == [H, 1, 0] and list(st.dt_bias) == [1, 0]
    assert list(st.A) == [1, 0, 0] and list(st.D) == [1, 0]
    # the CPU tensors' addresses are only checked for alignment here
    assert ssu.ssu_validate(pool, idx, x, dt, bias, A, B, C, D, out) == ssu.SSU_OK


def test_describe_rejects_wrong_dtypes(ssu):
    pool = torch.zeros(4, 2, 8, 128)
    x = torch.zeros(2, 2, 8, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        ssu.describe(pool, torch.zeros(2, dtype=torch.float32), x, x[:, :, 0], torch.zeros(2),
                     torch.zeros(2), torch.zeros(2, 1, 128, dtype=torch.bfloat16),
                     torch.zeros(2, 1, 128, dtype=torch.bfloat16), torch.zeros(2), x)
    with pytest.raises(TypeError):
        ssu.describe(pool.double(), torch.zeros(2, dtype=torch.int32), x, x[:, :, 0],
                     torch.zeros(2), torch.zeros(2),
                     torch.zeros(2, 1, 128, dtype=torch.bfloat16),
                     torch.zeros(2, 1, 128, dtype=torch.bfloat16), torch.zeros(2), x)


def test_check_indices_finds_repeats_and_out_of_range(ssu):
    import numpy as np
    ok = torch.from_numpy(np.random.default_rng(0).permutation(1000)[:300].astype(np.int32))
    assert ssu.ssu_check_indices(ok, 1000) == -1
    assert ssu.ssu_check_indices(ok.to(torch.int64), 1000) == -1
    rep = ok.clone()
    rep[200] = rep[17]
    assert ssu.ssu_check_indices(rep, 1000) == 200
    oob = ok.clone()
    oob[5] = 1000
    assert ssu.ssu_check_indices(oob, 1000) == 5
    neg = ok.to(torch.int64)
    neg[9] = -1
    assert ssu.ssu_check_indices(neg, 1000) == 9
    assert ssu.ssu_check_indices(torch.zeros(0, dtype=torch.int32), 0) == -1
    assert ssu.ssu_check_indices(rep, 1000) == 200 and "repeats slot" in ssu.last_error()


# ---- host-operand entry point: workspace size and the checks made before any CUDA call ----

def test_host_workspace_bytes_closed_form(ssu):
    """Dense idx, x, dt, B, C sections, each rounded up to 256 bytes."""
    r = lambda v: (v + 255) // 256 * 256
    for bs, H, P, N, G, i64 in ((128, 16, 64, 128, 1, False), (3, 5, 7, 64, 1, True),
                                (1, 4, 3, 256, 2, False), (0, 16, 64, 128, 1, False)):
        shape = ssu.ssu_shape_t(bs, H, P, N, G, bs + 1, 1 if i64 else 0, 0)
        want = (r(bs * (8 if i64 else 4)) + r(bs * H * P * 2) + r(bs * H * 2)
                + 2 * r(bs * G * N * 2))
        assert ssu.ssu_host_workspace_bytes(shape) == want
    # batch 128, 16 heads: exactly the step's 332,288 input bytes (every section a multiple
    # of 256 already)
    assert ssu.ssu_host_workspace_bytes(ssu.ssu_shape_t(128, 16, 64, 128, 1, 129, 0, 0)) == \
        128 * 4 + 128 * (16 * 64 + 256) * 2 + 128 * 16 * 2


def test_host_workspace_bytes_rejects_bad_shapes(ssu):
    n = ctypes.c_int64()
    assert ssu.lib().ssu_host_workspace_bytes(None, ctypes.byref(n)) == ssu.SSU_ERR_INVALID_ARG
    for bad in (dict(batch=-1), dict(nheads=0), dict(dstate=0)):
        shape = ssu.ssu_shape_t(8, 16, 64, 128, 1, 9, 0, 0)
        for k, v in bad.items():
            setattr(shape, k, v)
        assert ssu.lib().ssu_host_workspace_bytes(ctypes.byref(shape), ctypes.byref(n)) == \
            ssu.SSU_ERR_INVALID_ARG


def test_host_entry_rejects_null_handle_and_invalid_operands(ssu):
    ptrs, shape, st = canonical()
    f = ssu.ssu_update_from_host_raw
    assert f(None, ptrs, shape, st, BASE, 1 << 20, None) == ssu.SSU_ERR_INVALID_ARG
    assert "handle" in ssu.last_error()
