"""Seeded synthetic inputs for the decode-step selective state update.

This module is shared by the tests, ``bench.py`` and the smoke check, and it feeds both the
CUDA path and the CPU oracle.  It holds none of the method's arithmetic: it draws numbers,
rounds them to the storage types, and lays them out.

Shapes and value distributions follow the kernel measurement of sglang PR #41223
(Details / Kernel measurement): headdim 64, dstate 128, one group, an fp32 state pool
``[pool, H, 64, 128]`` with random ``state_batch_indices``, bf16 ``x``/``B``/``C``, per-head
``dt``/``A``/``D``/``dt_bias``.  The value ranges are

* state ~ N(0, 1) fp32; x, B, C ~ N(0, 1) rounded to bf16;
* dt ~ U(-4, 0) rounded to bf16; dt_bias ~ U(-1, 1); A = -exp(U(0, ln 16)); D ~ U(0, 1) (fp32),

and the generator is numpy's PCG64 (``numpy.random.default_rng(seed)``), drawn in a fixed
order so one seed always gives the same problem.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

HEADDIM = 64
DSTATE = 128


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round fp32 values to bf16 bit patterns (nearest, ties to even).  Inputs are finite."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns to fp32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class Problem:
    """One decode-step problem in host memory (bf16 operands held as uint16 patterns)."""

    pool: np.ndarray      # float32 [pool_size, H, P, N], or uint16 bf16 patterns
    idx: np.ndarray       # int64 [bs] (or [n_sets, bs] for rotation sets)
    x: np.ndarray         # uint16 [bs, H, P]
    dt: np.ndarray        # uint16 [bs, H]
    dt_bias: np.ndarray   # float32 [H]
    A: np.ndarray         # float32 [H]
    B: np.ndarray         # uint16 [bs, G, N]
    C: np.ndarray         # uint16 [bs, G, N]
    D: np.ndarray         # float32 [H]
    ngroups: int = 1
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.x.shape[0])

    @property
    def nheads(self) -> int:
        return int(self.x.shape[1])

    @property
    def pool_size(self) -> int:
        return int(self.pool.shape[0])


def head_params(rng: np.random.Generator, H: int):
    """Per-head dt_bias ~ U(-1,1), A = -exp(U(0, ln 16)), D ~ U(0,1), all fp32."""
    dt_bias = rng.uniform(-1.0, 1.0, H).astype(np.float32)
    A = (-np.exp(rng.uniform(0.0, math.log(16.0), H))).astype(np.float32)
    D = rng.uniform(0.0, 1.0, H).astype(np.float32)
    return dt_bias, A, D


def request_inputs(rng: np.random.Generator, bs: int, H: int, P: int = HEADDIM,
                   N: int = DSTATE, G: int = 1):
    """Per-request x, dt, B, C as bf16 patterns."""
    x = f32_to_bf16_bits(rng.standard_normal((bs, H, P), dtype=np.float32))
    dt = f32_to_bf16_bits(rng.uniform(-4.0, 0.0, (bs, H)).astype(np.float32))
    B = f32_to_bf16_bits(rng.standard_normal((bs, G, N), dtype=np.float32))
    C = f32_to_bf16_bits(rng.standard_normal((bs, G, N), dtype=np.float32))
    return x, dt, B, C


def state_pool(rng: np.random.Generator, pool_size: int, H: int, P: int = HEADDIM,
               N: int = DSTATE, dtype: str = "f32") -> np.ndarray:
    """State pool ~ N(0, 1): fp32 values, or (dtype "bf16") the same draws rounded to bf16
    patterns (uint16)."""
    pool = rng.standard_normal((pool_size, H, P, N), dtype=np.float32)
    return f32_to_bf16_bits(pool) if dtype == "bf16" else pool


def make_problem(bs: int, H: int = 16, P: int = HEADDIM, N: int = DSTATE, G: int = 1,
                 pool_size: int | None = None, seed: int = 0, state_dtype: str = "f32") -> Problem:
    """A problem whose ``idx`` is ``bs`` distinct slots drawn at random from the pool.

    The tiny parity workload is ``make_problem(8, 16, pool_size=32, seed=0)``: batch 8,
    16 heads, a 32-slot pool and a random permutation giving 8 distinct slots.
    """
    if pool_size is None:
        pool_size = bs + 16
    if pool_size < bs:
        raise ValueError("pool must hold at least one slot per request")
    rng = np.random.default_rng(seed)
    pool = state_pool(rng, pool_size, H, P, N, state_dtype)
    idx = rng.permutation(pool_size)[:bs].astype(np.int64)
    dt_bias, A, D = head_params(rng, H)
    x, dt, B, C = request_inputs(rng, bs, H, P, N, G)
    return Problem(pool, idx, x, dt, dt_bias, A, B, C, D, G)


def rotation_sets(bs: int, n_sets: int, seed: int = 0) -> np.ndarray:
    """``n_sets`` disjoint sets of ``bs`` slots covering a pool of ``bs * n_sets`` slots.

    Slots are a random permutation of the pool cut into consecutive sets, so each set is
    scattered over the pool (random, non-contiguous ``state_batch_indices``) and no two sets
    share a slot.  Returns int64 ``[n_sets, bs]``.
    """
    rng = np.random.default_rng(seed + 1_000_003)
    return rng.permutation(bs * n_sets).astype(np.int64).reshape(n_sets, bs)


def sets_for_cold_l2(bs: int, H: int, l2_bytes: int, factor: float = 3.0,
                     P: int = HEADDIM, N: int = DSTATE, min_sets: int = 3,
                     elem_bytes: int = 4) -> int:
    """Number of disjoint slot sets whose states together hold ``factor`` x the L2 size.

    Mirrors the cold-L2 rotation of sglang PR #41223 (Details / Kernel measurement): call i of
    a timed sequence touches set (i mod K), and the K sets hold at least 3x the L2.
    """
    set_bytes = bs * H * P * N * elem_bytes
    return max(min_sets, math.ceil(factor * l2_bytes / set_bytes))


def packed_xbc(rng: np.random.Generator, bs: int, H: int, P: int = HEADDIM, N: int = DSTATE,
               G: int = 1) -> np.ndarray:
    """One packed bf16 tensor ``[bs, H*P + 2*G*N]`` holding x, then B, then C per request.

    The strided-view workload (batch 512) takes x, B and C as views into this one tensor,
    as the kernel measurement of sglang PR #41223 does (Details / Kernel measurement).
    """
    return f32_to_bf16_bits(rng.standard_normal((bs, H * P + 2 * G * N), dtype=np.float32))
