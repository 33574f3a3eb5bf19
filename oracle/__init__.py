"""Double-precision CPU oracle for the Mamba2 decode-step selective state update.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package; the product path (the CUDA library and its binding)
never does, and this package imports nothing from it.

The arithmetic lives in ``ssu_oracle.c`` (plain C loops in IEEE double, compiled with FMA
contraction off so x86 and Arm give the same bits).  This module only

* builds that file with gcc into ``liboracle_ssu.so`` next to it,
* widens the operands exactly to double (bf16 patterns and fp32 values), and
* calls it.

The operands and their shapes follow sglang PR #41223, Details / Kernel measurement: an fp32
state pool ``[pool, H, headdim, dstate]`` gathered by ``state_batch_indices``; ``x`` of shape
``[bs, H, headdim]``; ``B`` and ``C`` of shape ``[bs, ngroups, dstate]``; per-head ``dt``,
``A``, ``D`` and ``dt_bias``.  The step itself is written out in the C file's header.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "ssu_oracle.c"
_LIB = _HERE / "liboracle_ssu.so"
_lib = None


def build(force: bool = False) -> Path:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    if force or not _LIB.exists() or _LIB.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB.with_suffix(f".so.tmp{os.getpid()}")
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", str(_SRC), "-o", str(tmp), "-lm"],
            check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(str(build()))
        d = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        lib.oracle_ssu_step.restype = i64
        lib.oracle_ssu_step.argtypes = [
            d, i64, ctypes.POINTER(i64), d, d, d, d, d, d, d, i64, i64, i64, i64, i64, d]
        lib.oracle_bf16_rne.restype = None
        lib.oracle_bf16_rne.argtypes = [d, ctypes.POINTER(ctypes.c_uint16), i64]
        _lib = lib
    return _lib


_executors: dict = {}


def _executor(threads: int):
    """One thread pool per thread count, kept for the life of the process (ctypes releases
    the interpreter lock while the C step runs, so the chunks run in parallel)."""
    ex = _executors.get(threads)
    if ex is None:
        from concurrent.futures import ThreadPoolExecutor
        ex = _executors[threads] = ThreadPoolExecutor(threads)
    return ex


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float64 exactly: a bf16 is the top half of an fp32."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_rne(values) -> np.ndarray:
    """Round float64 values to bf16 (round to nearest, ties to even) in one step; uint16 out."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_bf16_rne(_ptr(v, ctypes.c_double), _ptr(out, ctypes.c_uint16), v.size)
    return out


def ssu_step_inplace(pool64: np.ndarray, idx, x, dt, dt_bias, A, B, C, D,
                     ngroups: int = 1, threads: int = 1) -> tuple[np.ndarray, int]:
    """One decode step on a float64 pool, updated in place.

    ``pool64`` is a C-contiguous float64 array ``[pool, H, P, N]``.  ``x``, ``dt``, ``B`` and
    ``C`` are bf16 bit patterns (uint16) of shapes ``[bs,H,P]``, ``[bs,H]``, ``[bs,G,N]``,
    ``[bs,G,N]``; ``dt_bias``, ``A`` and ``D`` are per-head real arrays ``[H]``; ``idx`` holds
    integer slot ids ``[bs]``.  Returns ``(y, skipped)`` with ``y`` float64 ``[bs, H, P]``
    (NaN rows for skipped requests).  ``threads > 1`` splits the batch into contiguous chunks
    that run the same C function concurrently (requests are independent and their slots
    distinct); the arithmetic per request is unchanged.
    """
    if pool64.dtype != np.float64 or not pool64.flags.c_contiguous:
        raise ValueError("pool64 must be a C-contiguous float64 array")
    npool, H, P, N = pool64.shape
    xd = np.ascontiguousarray(bf16_to_f64(x))
    bs = xd.shape[0]
    G = int(ngroups)
    dtd = np.ascontiguousarray(bf16_to_f64(dt)).reshape(bs, H)
    Bd = np.ascontiguousarray(bf16_to_f64(B)).reshape(bs, G, N)
    Cd = np.ascontiguousarray(bf16_to_f64(C)).reshape(bs, G, N)
    xd = xd.reshape(bs, H, P)
    bias = np.ascontiguousarray(dt_bias, dtype=np.float64).reshape(H)
    Ad = np.ascontiguousarray(A, dtype=np.float64).reshape(H)
    Dd = np.ascontiguousarray(D, dtype=np.float64).reshape(H)
    ix = np.ascontiguousarray(idx, dtype=np.int64).reshape(bs)
    y = np.empty((bs, H, P), dtype=np.float64)
    lib = _load()
    dp = ctypes.c_double

    def run(b0: int, b1: int) -> int:
        n = b1 - b0
        return lib.oracle_ssu_step(
            _ptr(pool64, dp), npool, _ptr(ix[b0:b1], ctypes.c_int64), _ptr(xd[b0:b1], dp),
            _ptr(dtd[b0:b1], dp), _ptr(bias, dp), _ptr(Ad, dp), _ptr(Bd[b0:b1], dp),
            _ptr(Cd[b0:b1], dp), _ptr(Dd, dp), n, H, P, N, G, _ptr(y[b0:b1], dp))

    if threads <= 1 or bs < 2:
        skipped = run(0, bs)
    else:
        cuts = np.linspace(0, bs, min(threads, bs) + 1).astype(int)
        parts = list(_executor(threads).map(lambda i: run(int(cuts[i]), int(cuts[i + 1])),
                                            range(len(cuts) - 1)))
        skipped = -1 if min(parts) < 0 else sum(parts)
    if skipped < 0:
        raise ValueError("oracle rejected the shape")
    return y, int(skipped)


def ssu_step(pool, idx, x, dt, dt_bias, A, B, C, D, ngroups: int = 1):
    """One decode step on a copy of ``pool`` (fp32 or float64).

    Returns ``(new_pool64, y64, skipped)``: the whole pool after the step in float64, the
    float64 readout ``[bs, H, P]`` and the number of skipped (out-of-range) requests.
    """
    pool64 = np.array(pool, dtype=np.float64, order="C", copy=True)
    y, skipped = ssu_step_inplace(pool64, idx, x, dt, dt_bias, A, B, C, D, ngroups)
    return pool64, y, skipped


def copy_blocks(tensors, src, dst):
    """State-block copy, written out plainly (vLLM PR #48110, Purpose): for every request i
    and every tensor (an array whose first axis indexes blocks), block dst[i] receives the
    bytes of block src[i].  Returns new arrays; a request whose ids fall outside any tensor's
    range is skipped for every tensor.  Returns (new_tensors, skipped)."""
    out = [np.array(t, copy=True) for t in tensors]
    skipped = 0
    for s_, d_ in zip(np.asarray(src).tolist(), np.asarray(dst).tolist()):
        if not all(0 <= s_ < len(t) and 0 <= d_ < len(t) for t in tensors):
            skipped += 1
            continue
        for t, o in zip(tensors, out):
            o[d_] = t[s_]
    return out, skipped


def ssu_tokens(pool, idx, x, dt, dt_bias, A, B, C, D, ngroups: int = 1):
    """T consecutive decode steps: the single step above applied to tokens t = 0 .. T-1 in
    order, each starting from the state the previous token left (the multi-token verification
    of speculative decoding, vLLM PR #48110, Test Plan).  ``x`` is ``[bs, T, H, P]``, ``dt``
    ``[bs, T, H]``, ``B``/``C`` ``[bs, T, G, N]`` (bf16 patterns).  Returns
    ``(new_pool64, y64 [bs, T, H, P], intermediate64 [bs, T, H, P, N], skipped)``;
    intermediate[b, t] is request b's state after token t (NaN for skipped requests)."""
    pool64 = np.array(pool, dtype=np.float64, order="C", copy=True)
    x = np.asarray(x)
    bs, T, H, P = x.shape
    N = pool64.shape[3]
    idx = np.asarray(idx, dtype=np.int64)
    ok = (idx >= 0) & (idx < pool64.shape[0])
    y = np.empty((bs, T, H, P))
    inter = np.full((bs, T, H, P, N), np.nan)
    skipped = 0
    for t in range(T):
        y[:, t], skipped = ssu_step_inplace(pool64, idx, x[:, t], np.asarray(dt)[:, t], dt_bias,
                                            A, np.asarray(B)[:, t], np.asarray(C)[:, t], D,
                                            ngroups)
        inter[ok, t] = pool64[idx[ok]]
    return pool64, y, inter, skipped
