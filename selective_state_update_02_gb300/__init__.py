"""GB300 (sm_103a) Mamba2 decode-step selective state update.

Python binding of ``libssu.so`` (C ABI declared in ``include/ssu.h``).  The functions carry
the C names and only marshal arguments: tensor pointers, sizes and element strides go into
the ABI structs, and every step of the update runs in the library's CUDA kernels.  There is
no CPU or PyTorch fallback: if the library is missing, every entry point raises.

Operand layout (sglang PR #41223, Details / Kernel measurement): ``state_pool`` fp32 or bf16
``[pool, H, P, N]`` (N = 64, 128 or 256); ``state_batch_indices`` int32/int64 ``[bs]``; ``x`` and ``out`` bf16
``[bs, H, P]``; ``B`` and ``C`` bf16 ``[bs, G, N]``; ``dt`` bf16 ``[bs, H]`` (or the
head-expanded ``[bs, H, P]`` view with stride 0 over P); ``dt_bias`` and ``D`` fp32 ``[H]``
(or ``[H, P]`` with stride 0); ``A`` fp32 ``[H]`` (or ``[H, P, N]`` with strides 0).
Strided views are accepted as they are; nothing is copied.
"""

from __future__ import annotations

import ctypes
from pathlib import Path

import torch

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libssu.so"

SSU_OK = 0
SSU_ERR_INVALID_ARG = 1
SSU_ERR_UNSUPPORTED = 2
SSU_ERR_MISALIGNED = 3
SSU_ERR_CUDA = 4
SSU_ERR_INDEX_OOB = 5

SSU_INDEX_I32 = 0
SSU_INDEX_I64 = 1

SSU_STATE_F32 = 0
SSU_STATE_BF16 = 1

SSU_MODE_AUTO = 0
SSU_MODE_VEC = 1

_i64 = ctypes.c_int64


class ssu_shape_t(ctypes.Structure):
    _fields_ = [("batch", _i64), ("nheads", _i64), ("headdim", _i64), ("dstate", _i64),
                ("ngroups", _i64), ("pool_size", _i64), ("index_dtype", ctypes.c_int32),
                ("state_dtype", ctypes.c_int32)]


class ssu_strides_t(ctypes.Structure):
    _fields_ = [("state", _i64 * 4), ("x", _i64 * 3), ("out", _i64 * 3), ("dt", _i64 * 3),
                ("B", _i64 * 3), ("C", _i64 * 3), ("dt_bias", _i64 * 2), ("D", _i64 * 2),
                ("A", _i64 * 3), ("idx", _i64)]


class ssu_launch_t(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("rows_per_warp", ctypes.c_int32),
                ("warps_per_cta", ctypes.c_int32), ("stages", ctypes.c_int32)]


class ssu_token_strides_t(ctypes.Structure):
    _fields_ = [("x", _i64), ("out", _i64), ("dt", _i64), ("B", _i64), ("C", _i64),
                ("intermediate", _i64 * 5)]


SSU_MAX_TOKENS = 64


class ssu_block_tensor_t(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("block_bytes", _i64),
                ("block_stride_bytes", _i64), ("num_blocks", _i64)]


class ssu_copy_launch_t(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("chunk_kib", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("threads", ctypes.c_int32)]


SSU_COPY_AUTO = 0
SSU_COPY_VEC = 1
SSU_COPY_MAX_TENSORS = 64


class SsuError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}: {message}")


_lib = None
_vp = ctypes.c_void_p
_EXPORTS = {
    "ssu_abi_version": (ctypes.c_int32, []),
    "ssu_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "ssu_last_error": (ctypes.c_char_p, []),
    "ssu_create": (ctypes.c_int, [ctypes.POINTER(_vp), ctypes.c_int32]),
    "ssu_destroy": (ctypes.c_int, [_vp]),
    "ssu_validate": (ctypes.c_int, [_vp] * 10 + [ctypes.POINTER(ssu_shape_t),
                                                 ctypes.POINTER(ssu_strides_t)]),
    "ssu_update": (ctypes.c_int, [_vp] * 11 + [ctypes.POINTER(ssu_shape_t),
                                               ctypes.POINTER(ssu_strides_t), _vp]),
    "ssu_get_error": (ctypes.c_int, [_vp, _vp, ctypes.POINTER(ctypes.c_uint32),
                                     ctypes.POINTER(ctypes.c_int64)]),
    "ssu_set_launch": (ctypes.c_int, [_vp, ctypes.POINTER(ssu_launch_t)]),
    "ssu_set_launch_override": (ctypes.c_int, [_vp, ctypes.c_char_p]),
    "ssu_get_launch": (ctypes.c_int, [_vp, ctypes.POINTER(ssu_shape_t),
                                      ctypes.POINTER(ssu_launch_t)]),
    "ssu_set_pdl": (ctypes.c_int, [_vp, ctypes.c_int32]),
    "ssu_check_indices": (ctypes.c_int, [_vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int64,
                                         ctypes.POINTER(ctypes.c_int64)]),
    "ssu_update_tokens": (ctypes.c_int, [_vp] * 12 + [ctypes.POINTER(ssu_shape_t),
                                                      ctypes.POINTER(ssu_strides_t),
                                                      ctypes.c_int64,
                                                      ctypes.POINTER(ssu_token_strides_t), _vp]),
    "ssu_copy_blocks": (ctypes.c_int, [_vp, ctypes.POINTER(ssu_block_tensor_t), ctypes.c_int32,
                                       _vp, _vp, ctypes.c_int64, ctypes.c_int32, _vp]),
    "ssu_copy_set_launch": (ctypes.c_int, [_vp, ctypes.POINTER(ssu_copy_launch_t)]),
    "ssu_update_static": (ctypes.c_int, [_vp] * 10 + [ctypes.POINTER(ssu_shape_t),
                                                      ctypes.POINTER(ssu_strides_t), _vp, _vp]),
    "ssu_host_workspace_bytes": (ctypes.c_int, [ctypes.POINTER(ssu_shape_t),
                                                ctypes.POINTER(ctypes.c_int64)]),
    "ssu_update_from_host": (ctypes.c_int, [_vp] * 11 + [ctypes.POINTER(ssu_shape_t),
                                                         ctypes.POINTER(ssu_strides_t), _vp,
                                                         ctypes.c_int64, _vp]),
}

SSU_STATIC_SCRATCH_BYTES = 256
SSU_ABI_VERSION = 2
SSU_STATIC_MAX_BATCH = 2147483647


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        handle = ctypes.CDLL(str(LIB_PATH))
        for name, (res, args) in _EXPORTS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        if handle.ssu_abi_version() != SSU_ABI_VERSION:
            raise RuntimeError("libssu.so ABI version mismatch")
        _lib = handle
    return _lib


def status_string(status: int) -> str:
    return lib().ssu_status_string(status).decode()


def last_error() -> str:
    return lib().ssu_last_error().decode()


def _check(status: int, where: str) -> None:
    if status != SSU_OK:
        raise SsuError(status, where, last_error())


# ---- marshalling -------------------------------------------------------------------------

def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _expect(t: torch.Tensor, name: str, dtype: torch.dtype, ndims: tuple[int, ...]):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() not in ndims:
        raise ValueError(f"{name} must have {' or '.join(map(str, ndims))} dims, got {t.dim()}")


def _broadcast_strides(t: torch.Tensor, name: str, dims: tuple[int, ...], full: int):
    """Strides of a per-head operand in its expanded form of `full` dims (missing dims: 0)."""
    if t.shape[:1] != dims[:1]:
        raise ValueError(f"{name} must start with dimension {dims[0]}, got {tuple(t.shape)}")
    st = list(t.stride()) + [0] * (full - t.dim())
    for i in range(1, t.dim()):
        if t.shape[i] != dims[i]:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected prefix of {dims}")
    return st


def describe(state_pool, state_batch_indices, x, dt, dt_bias, A, B, C, D, out):
    """Build ``(ssu_shape_t, ssu_strides_t)`` for a set of tensors (no data is touched)."""
    if not isinstance(state_pool, torch.Tensor) or state_pool.dim() != 4 or \
            state_pool.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("state_pool must be a 4-D float32 or bfloat16 tensor")
    if state_batch_indices.dtype not in (torch.int32, torch.int64) or \
            state_batch_indices.dim() != 1:
        raise TypeError("state_batch_indices must be a 1-D int32 or int64 tensor")
    _expect(x, "x", torch.bfloat16, (3,))
    _expect(out, "out", torch.bfloat16, (3,))
    _expect(dt, "dt", torch.bfloat16, (2, 3))
    _expect(dt_bias, "dt_bias", torch.float32, (1, 2))
    _expect(D, "D", torch.float32, (1, 2))
    _expect(A, "A", torch.float32, (1, 3))
    _expect(B, "B", torch.bfloat16, (3,))
    _expect(C, "C", torch.bfloat16, (3,))
    pool, H, P, N = state_pool.shape
    bs = x.shape[0]
    G = B.shape[1]
    if tuple(x.shape) != (bs, H, P) or tuple(out.shape) != (bs, H, P):
        raise ValueError(f"x and out must be [bs, H, P] = {(bs, H, P)}")
    if tuple(B.shape) != (bs, G, N) or tuple(C.shape) != (bs, G, N):
        raise ValueError(f"B and C must be [bs, G, N] = {(bs, G, N)}")
    if state_batch_indices.shape[0] != bs:
        raise ValueError("state_batch_indices must have one entry per request")
    if tuple(dt.shape[:2]) != (bs, H) or (dt.dim() == 3 and dt.shape[2] != P):
        raise ValueError("dt must be [bs, H] or [bs, H, P]")
    shape = ssu_shape_t(bs, H, P, N, G, pool,
                        SSU_INDEX_I64 if state_batch_indices.dtype == torch.int64
                        else SSU_INDEX_I32,
                        SSU_STATE_BF16 if state_pool.dtype == torch.bfloat16 else SSU_STATE_F32)
    st = ssu_strides_t()
    st.state[:] = list(state_pool.stride())
    st.x[:] = list(x.stride())
    st.out[:] = list(out.stride())
    st.dt[:] = list(dt.stride()) + [0] * (3 - dt.dim())
    st.B[:] = list(B.stride())
    st.C[:] = list(C.stride())
    st.dt_bias[:] = _broadcast_strides(dt_bias, "dt_bias", (H, P), 2)
    st.D[:] = _broadcast_strides(D, "D", (H, P), 2)
    st.A[:] = _broadcast_strides(A, "A", (H, P, N), 3)
    st.idx = state_batch_indices.stride(0)
    return shape, st


def _stream_ptr(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---- the C entry points --------------------------------------------------------------------

def ssu_abi_version() -> int:
    return int(lib().ssu_abi_version())


def ssu_create(device: int = 0) -> int:
    """Create a handle on ``device``; returns it as an integer."""
    h = _vp()
    _check(lib().ssu_create(ctypes.byref(h), int(device)), "ssu_create")
    return h.value


def ssu_destroy(handle: int) -> None:
    _check(lib().ssu_destroy(handle), "ssu_destroy")


def ssu_validate(state_pool, state_batch_indices, x, dt, dt_bias, A, B, C, D, out,
                 shape: ssu_shape_t | None = None, strides: ssu_strides_t | None = None) -> int:
    """Host-side validation only; returns the status code (0 = valid).

    With tensors, the shape and strides are derived from them.  With integer pointers (no
    memory is touched), ``shape`` and ``strides`` must be given.
    """
    if shape is None or strides is None:
        shape, strides = describe(state_pool, state_batch_indices, x, dt, dt_bias, A, B, C, D,
                                  out)
    ptrs = [_ptr(t) for t in (state_pool, state_batch_indices, x, dt, dt_bias, A, B, C, D, out)]
    return int(lib().ssu_validate(*ptrs, ctypes.byref(shape), ctypes.byref(strides)))


def ssu_update(handle: int, state_pool, state_batch_indices, x, dt, dt_bias, A, B, C, D, out,
               stream=None) -> None:
    """Enqueue one decode step on ``stream`` (default: torch's current stream)."""
    shape, strides = describe(state_pool, state_batch_indices, x, dt, dt_bias, A, B, C, D, out)
    ptrs = [_ptr(t) for t in (state_pool, state_batch_indices, x, dt, dt_bias, A, B, C, D, out)]
    _check(lib().ssu_update(handle, *ptrs, ctypes.byref(shape), ctypes.byref(strides),
                            _stream_ptr(stream)), "ssu_update")


def ssu_update_static(state_pool, state_batch_indices, x, dt, dt_bias, A, B, C, D, out,
                      counters_out=None, stream=None) -> None:
    """Allocation-free ssu_update on the current device (no handle).

    For callers that cannot allocate device memory: the kernel's counters live in a fixed
    256-byte array inside the library.  ``counters_out`` is an optional caller-owned int32/uint32
    device tensor of >= 3 elements that receives [skipped, smallest skipped index or
    0xFFFFFFFF, 0].  Calls that overlap on the GPU race on the shared counters.
    """
    shape, strides = describe(state_pool, state_batch_indices, x, dt, dt_bias, A, B, C, D, out)
    if counters_out is not None:
        _check_counters(counters_out, state_pool)
    ptrs = [_ptr(t) for t in (state_pool, state_batch_indices, x, dt, dt_bias, A, B, C, D, out)]
    _check(lib().ssu_update_static(*ptrs, ctypes.byref(shape), ctypes.byref(strides),
                                   _ptr(counters_out), _stream_ptr(stream)),
           "ssu_update_static")


def _check_counters(counters_out, state_pool) -> None:
    """``counters_out`` receives a 12-byte device-to-device copy: it must be a contiguous CUDA
    tensor of 4-byte elements with at least 3 of them, on the state pool's device."""
    t = counters_out
    if not isinstance(t, torch.Tensor):
        raise ValueError("counters_out must be a torch.Tensor (or None)")
    if t.device.type != "cuda" or t.device != state_pool.device:
        raise ValueError(f"counters_out must be on {state_pool.device}, got {t.device}")
    if t.element_size() != 4 or t.dtype.is_floating_point:
        raise ValueError(f"counters_out must hold 4-byte integers, got {t.dtype}")
    if t.numel() < 3 or not t.is_contiguous():
        raise ValueError("counters_out must be contiguous with at least 3 elements")


def ssu_host_workspace_bytes(shape: ssu_shape_t) -> int:
    """Device workspace bytes ``ssu_update_from_host`` needs for ``shape``."""
    n = ctypes.c_int64()
    _check(lib().ssu_host_workspace_bytes(ctypes.byref(shape), ctypes.byref(n)),
           "ssu_host_workspace_bytes")
    return int(n.value)


def ssu_update_from_host(handle: int, state_pool, state_batch_indices, x, dt, dt_bias, A, B, C,
                         D, out, workspace, stream=None) -> None:
    """One decode step with the per-step operands (``state_batch_indices``, ``x``, ``dt``,
    ``B``, ``C``) and ``out`` in page-locked host memory (``pin_memory()`` tensors); the state
    pool, ``dt_bias``, ``A`` and ``D`` on the device.  ``workspace`` is a device uint8 tensor of
    at least ``ssu_host_workspace_bytes(shape)`` bytes.  ``out`` is complete once ``stream``
    has passed the call."""
    shape, strides = describe(state_pool, state_batch_indices, x, dt, dt_bias, A, B, C, D, out)
    ptrs = [_ptr(t) for t in (state_pool, state_batch_indices, x, dt, dt_bias, A, B, C, D, out)]
    nbytes = workspace.numel() * workspace.element_size() if isinstance(workspace, torch.Tensor) \
        else 0
    _check(lib().ssu_update_from_host(handle, *ptrs, ctypes.byref(shape), ctypes.byref(strides),
                                      _ptr(workspace), nbytes, _stream_ptr(stream)),
           "ssu_update_from_host")


def ssu_update_from_host_raw(handle: int, ptrs, shape: ssu_shape_t, strides: ssu_strides_t,
                             workspace: int, workspace_bytes: int, stream: int | None) -> int:
    """ssu_update_from_host with precomputed pointers/structs; returns the status."""
    return int(lib().ssu_update_from_host(handle, *ptrs, ctypes.byref(shape),
                                          ctypes.byref(strides), workspace, workspace_bytes,
                                          stream))


def ssu_update_raw(handle: int, ptrs, shape: ssu_shape_t, strides: ssu_strides_t,
                   stream: int | None) -> int:
    """ssu_update with precomputed pointers/structs (for tight timing loops); returns status."""
    return int(lib().ssu_update(handle, *ptrs, ctypes.byref(shape), ctypes.byref(strides),
                                stream))


def ssu_get_error(handle: int, stream=None) -> tuple[int, int]:
    """Synchronise, then read and clear the skipped-request counters: (skipped, first_bad)."""
    skipped = ctypes.c_uint32()
    first = ctypes.c_int64()
    st = lib().ssu_get_error(handle, _stream_ptr(stream), ctypes.byref(skipped),
                             ctypes.byref(first))
    if st not in (SSU_OK, SSU_ERR_INDEX_OOB):
        _check(st, "ssu_get_error")
    return int(skipped.value), int(first.value)


def ssu_set_launch(handle: int, mode: int = SSU_MODE_AUTO, rows_per_warp: int = 0,
                   warps_per_cta: int = 0, stages: int = 0) -> None:
    """Force a launch shape (mode AUTO restores the built-in table)."""
    cfg = ssu_launch_t(mode, rows_per_warp, warps_per_cta, stages)
    _check(lib().ssu_set_launch(handle, ctypes.byref(cfg)), "ssu_set_launch")


def ssu_set_launch_override(handle: int, spec: str | None) -> None:
    """Force a launch shape from text: "rows_per_warp,warps_per_cta" (optionally "vec,..."),
    or None / "" / "auto" for the built-in table."""
    _check(lib().ssu_set_launch_override(handle, None if spec is None else spec.encode()),
           "ssu_set_launch_override")


def ssu_check_indices(state_batch_indices, pool_size: int) -> int:
    """Debug check of a host (CPU) index tensor: in range and no repeated slot.  Returns -1
    when the indices are valid, else the position of the first bad entry."""
    t = state_batch_indices
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu" or t.dim() != 1:
        raise TypeError("state_batch_indices must be a 1-D CPU tensor")
    if t.dtype not in (torch.int32, torch.int64):
        raise TypeError("state_batch_indices must be int32 or int64")
    t = t.contiguous()
    first = ctypes.c_int64(-1)
    st = lib().ssu_check_indices(t.data_ptr(), t.shape[0],
                                 SSU_INDEX_I64 if t.dtype == torch.int64 else SSU_INDEX_I32,
                                 int(pool_size), ctypes.byref(first))
    if st not in (SSU_OK, SSU_ERR_INVALID_ARG):
        _check(st, "ssu_check_indices")
    return int(first.value) if st != SSU_OK else -1


def ssu_set_pdl(handle: int, enable: bool = True) -> None:
    """Turn programmatic dependent launch on or off for this handle (on by default)."""
    _check(lib().ssu_set_pdl(handle, 1 if enable else 0), "ssu_set_pdl")


def ssu_get_launch(handle: int, shape: ssu_shape_t) -> tuple[int, int, int, int]:
    cfg = ssu_launch_t()
    _check(lib().ssu_get_launch(handle, ctypes.byref(shape), ctypes.byref(cfg)),
           "ssu_get_launch")
    return cfg.mode, cfg.rows_per_warp, cfg.warps_per_cta, cfg.stages


def ssu_update_tokens(handle: int, state_pool, state_batch_indices, x, dt, dt_bias, A, B, C, D,
                      out, intermediate=None, stream=None) -> None:
    """T consecutive decode steps per request.  ``x`` and ``out`` are ``[bs, T, H, P]``;
    ``dt`` is ``[bs, T, H]`` (or ``[bs, T, H, P]`` with stride 0 over P); ``B`` and ``C`` are
    ``[bs, T, G, N]``; ``intermediate`` (optional, ``[bs, T, H, P, N]`` of the state's dtype)
    receives the state after every token.  Per-head operands as for ``ssu_update``."""
    for name, t, nd in (("x", x, 4), ("out", out, 4), ("B", B, 4), ("C", C, 4)):
        if not isinstance(t, torch.Tensor) or t.dim() != nd:
            raise ValueError(f"{name} must be a {nd}-D tensor with a token dimension")
    if dt.dim() not in (3, 4):
        raise ValueError("dt must be [bs, T, H] or [bs, T, H, P]")
    T = x.shape[1]
    for name, t in (("out", out), ("dt", dt), ("B", B), ("C", C)):
        if t.shape[1] != T:
            raise ValueError(f"{name} must have {T} tokens")
    shape, strides = describe(state_pool, state_batch_indices, x[:, 0], dt[:, 0], dt_bias, A,
                              B[:, 0], C[:, 0], D, out[:, 0])
    ts = ssu_token_strides_t()
    ts.x, ts.out, ts.dt, ts.B, ts.C = (x.stride(1), out.stride(1), dt.stride(1), B.stride(1),
                                       C.stride(1))
    if intermediate is not None:
        _expect(intermediate, "intermediate", state_pool.dtype, (5,))
        if tuple(intermediate.shape) != (x.shape[0], T, x.shape[2], x.shape[3],
                                         state_pool.shape[3]):
            raise ValueError("intermediate must be [bs, T, H, P, N]")
        ts.intermediate[:] = list(intermediate.stride())
    ptrs = [_ptr(t) for t in (state_pool, state_batch_indices, x, dt, dt_bias, A, B, C, D, out,
                               intermediate)]
    _check(lib().ssu_update_tokens(handle, *ptrs, ctypes.byref(shape), ctypes.byref(strides), T,
                                   ctypes.byref(ts), _stream_ptr(stream)), "ssu_update_tokens")


def describe_blocks(tensors) -> tuple[ctypes.Array, int]:
    """ABI descriptors for state tensors laid out as ``[num_blocks, ...]``: block k is the
    slice ``t[k]``, which must be contiguous (its bytes are copied verbatim)."""
    arr = (ssu_block_tensor_t * len(tensors))()
    for i, t in enumerate(tensors):
        if not isinstance(t, torch.Tensor) or t.dim() < 1:
            raise TypeError("each state tensor must be a torch.Tensor of >= 1 dims")
        if t.dim() > 1 and not t[0].is_contiguous():
            raise ValueError("each block (t[k]) must be contiguous")
        item = t.element_size()
        block = item * (t[0].numel() if t.dim() > 1 else 1)
        arr[i] = ssu_block_tensor_t(t.data_ptr(), block, t.stride(0) * item, t.shape[0])
    return arr, len(tensors)


def ssu_copy_blocks(handle: int, tensors, src_idx, dst_idx, stream=None) -> None:
    """Copy block src_idx[i] -> dst_idx[i] of every tensor in ``tensors`` (each
    ``[num_blocks, ...]``), for every request i.  Enqueued on ``stream``."""
    if src_idx.dtype != dst_idx.dtype or src_idx.dtype not in (torch.int32, torch.int64):
        raise TypeError("src_idx and dst_idx must both be int32 or both int64")
    if src_idx.dim() != 1 or src_idx.shape != dst_idx.shape:
        raise ValueError("src_idx and dst_idx must be 1-D of the same length")
    if not (src_idx.is_contiguous() and dst_idx.is_contiguous()):
        raise ValueError("src_idx and dst_idx must be contiguous")
    arr, count = describe_blocks(tensors)
    dtype = SSU_INDEX_I64 if src_idx.dtype == torch.int64 else SSU_INDEX_I32
    _check(lib().ssu_copy_blocks(handle, arr, count, src_idx.data_ptr(), dst_idx.data_ptr(),
                                 src_idx.shape[0], dtype, _stream_ptr(stream)),
           "ssu_copy_blocks")


def ssu_copy_set_launch(handle: int, mode: int = SSU_COPY_AUTO, chunk_kib: int = 32,
                        stages: int = 8, threads: int = 256) -> None:
    cfg = ssu_copy_launch_t(mode, chunk_kib, stages, threads)
    _check(lib().ssu_copy_set_launch(handle, ctypes.byref(cfg)), "ssu_copy_set_launch")


class SelectiveStateUpdate:
    """Owns one handle; ``__call__`` is ``ssu_update`` on it."""

    def __init__(self, device: int | None = None):
        if device is None:
            device = torch.cuda.current_device()
        self.device = int(device)
        self.handle = ssu_create(self.device)

    def __call__(self, state_pool, state_batch_indices, x, dt, dt_bias, A, B, C, D, out,
                 stream=None):
        ssu_update(self.handle, state_pool, state_batch_indices, x, dt, dt_bias, A, B, C, D,
                   out, stream)
        return out

    def tokens(self, state_pool, state_batch_indices, x, dt, dt_bias, A, B, C, D, out,
               intermediate=None, stream=None):
        ssu_update_tokens(self.handle, state_pool, state_batch_indices, x, dt, dt_bias, A, B, C,
                          D, out, intermediate, stream)
        return out

    def copy_blocks(self, tensors, src_idx, dst_idx, stream=None):
        ssu_copy_blocks(self.handle, tensors, src_idx, dst_idx, stream)

    def get_error(self, stream=None):
        return ssu_get_error(self.handle, stream)

    def set_launch(self, *args, **kw):
        ssu_set_launch(self.handle, *args, **kw)

    def close(self):
        if self.handle:
            ssu_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
