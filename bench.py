#!/usr/bin/env python
"""Benchmark of the decode-step selective state update on one GB300 (or N replicas).

A step is one ``ssu_update`` call: one decode step of every request in the batch, all heads
(index gather, dt/dA, state load, update and in-place store, readout).  The default
workload is the serving decode batch: 128 requests, 16 heads, headdim 64, dstate 128, fp32
state, bf16 x/B/C, over a 2432-slot pool split into 19 disjoint 128-slot sets.

Timing follows the kernel measurement of sglang PR #41223 (Details / Kernel measurement):
the calls are captured in CUDA graphs, call i touches slot set (i mod K), and the K sets
together hold at least 3x the L2, so every call reads its state from HBM.  The K timed
steps are bracketed by CUDA events on the launching stream; the reported value is the
time per call (lower is better).  Batches 8 and 512 are measured the same way and reported
under ``by_batch``.

``--impl reference`` times the double-precision CPU oracle instead (the reference arm):
the same metric and workload, on the host cores.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

import numpy as np  # noqa: E402

METRIC = "µs/call and achieved HBM TB/s (% of peak), H=16 at batch 8/128/512, cold L2"
UNIT = "us/call"
NHEADS, HEADDIM, DSTATE, NGROUPS = 16, 64, 128, 1
DEFAULT_BATCH = 128
SERVING_SETS = 19            # 2432 slots at batch 128
NOMINAL_HBM_GBS = 8000.0     # the pages' round GB200/B200 HBM3e figure
FALLBACK_HBM_GBS = 6800.0
PAGE_US = {8: 4.02, 128: 24.1, 512: 85.7}   # sglang PR #41223 Speedup Result, B200 (context)
CSRC = ROOT / "selective_state_update_02_gb300" / "csrc"
KERNEL_SOURCES = [CSRC / "ssu_vec.cuh", CSRC / "ssu_device.cuh"]     # VEC kernel
TOKENS_SOURCES = [CSRC / "ssu_tokens.cuh", CSRC / "ssu_device.cuh"]  # multi-token kernel
MMA_SOURCES = [CSRC / "ssu_tokens_mma.cuh", CSRC / "ssu_tokens.cuh",  # chunked multi-token
               CSRC / "ssu_device.cuh"]
COPY_SOURCES = [CSRC / "ssu_copy.cu", CSRC / "ssu_device.cuh"]       # block-copy kernels


# ---- arithmetic of the measurement (host logic, tested on CPU) ---------------------------


def tokens_kernel(T: int, with_inter: bool, N: int, state_dtype: str, forced: bool) -> str:
    """The kernel the library's ssu_update_tokens picks for the bench's aligned operands (the
    rule of mma_min_tokens in ssu_tokens.cu): the chunked one without intermediate states and
    without a forced launch shape, for an fp32 state (dstate 64 or 128) from 5 tokens and a
    bf16 state of dstate 128 from 16; else the general one.  Names the roofline's kernel."""
    if with_inter or forced or N not in (64, 128):
        return "ssu_tokens_kernel"
    if state_dtype == "f32":
        return "ssu_tokens_mma_kernel" if T >= 5 else "ssu_tokens_kernel"
    return "ssu_tokens_mma_kernel" if (N == 128 and T >= 16) else "ssu_tokens_kernel"


def bytes_per_call(bs: int, H: int = NHEADS, P: int = HEADDIM, N: int = DSTATE,
                   G: int = NGROUPS, idx_bytes: int = 4, state_bytes: int = 4) -> int:
    """Algorithmic HBM bytes of one call: the state read and written once, every input read
    once, the output written once; per-head parameters counted once (stride-0 broadcasts)."""
    state = 2 * bs * H * P * N * state_bytes
    x = bs * H * P * 2
    y = bs * H * P * 2
    bc = 2 * bs * G * N * 2
    dt = bs * H * 2
    idx = bs * idx_bytes
    params = 3 * H * 4
    return state + x + y + bc + dt + idx + params


def flops_per_call(bs: int, H: int = NHEADS, P: int = HEADDIM, N: int = DSTATE) -> int:
    """Update (multiply + fma) and readout (fma) per state element."""
    return 5 * bs * H * P * N


def sets_for(bs: int, H: int, l2_bytes: int, N: int = DSTATE, elem_bytes: int = 4) -> int:
    import workloads as wl
    n = wl.sets_for_cold_l2(bs, H, l2_bytes, N=N, elem_bytes=elem_bytes)
    if bs == DEFAULT_BATCH and H == NHEADS and N == DSTATE and elem_bytes == 4:
        return max(SERVING_SETS, n)
    return n


def load_peaks() -> dict:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback"}


def source_digest(files=None) -> str:
    """Digest of the sources that define the timed kernel (its own header and the device
    helpers it includes): counters taken on other sources are not reported."""
    h = hashlib.sha256()
    for f in files or KERNEL_SOURCES:
        h.update(f.read_bytes())
    return h.hexdigest()[:16]


def recorded_traffic(workload_tag: str, sources=None) -> int | None:
    """DRAM bytes per launch from a committed ncu summary, if it was taken on this source.

    The summaries under profiles/ carry a line
    ``traffic_per_launch_bytes: <int> source: <digest> workload: <tag>``.  The digest covers
    ``sources`` (default: the VEC kernel's).
    """
    digest = source_digest(sources or KERNEL_SOURCES)
    for f in sorted((ROOT / "profiles").glob("*.md")):
        for m in re.finditer(r"traffic_per_launch_bytes:\s*(\d+)\s+source:\s*([0-9a-f]+)\s+"
                             r"workload:\s*(\S+)", f.read_text()):
            if m.group(2) == digest and m.group(3) == workload_tag:
                return int(m.group(1))
    return None


def aggregate_value(elapsed_us_per_rank: list[float], steps: int) -> float:
    """Whole-job time per call: the slowest rank's time over every rank's calls."""
    return max(elapsed_us_per_rank) / (steps * len(elapsed_us_per_rank))


def gather_elapsed(elapsed_us: float, world: int, device) -> list[float]:
    """Every rank's timed-region length (µs), gathered on every rank (no data-path
    collective: this is the only exchange, after the timed region)."""
    if world <= 1:
        return [elapsed_us]
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed_us], dtype=torch.float64, device=device)
    parts = [torch.zeros_like(t) for _ in range(world)]
    dist.all_gather(parts, t)
    return [float(v.item()) for v in parts]


def parse_clocks(csv_text: str) -> dict | None:
    rows = []
    for line in csv_text.splitlines():
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9 or not parts[0].isdigit():
            continue
        try:
            sm = float(parts[1].split()[0])
            smax = float(parts[2].split()[0])
            power = float(parts[3].split()[0])
        except ValueError:
            continue
        rows.append((sm, smax, power, parts[5:9]))
    if not rows:
        return None
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v == "Active"})
    loaded = [r[0] for r in rows if r[2] > 200.0] or [r[0] for r in rows]
    return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[1] for r in rows),
            "reasons": reasons, "samples": len(rows)}


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.text = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.text, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.text, _ = self.proc.communicate()
        return False

    def result(self):
        return parse_clocks(getattr(self, "text", ""))


# ---- the GPU arm --------------------------------------------------------------------------

class Workload:
    """Device-resident rotation workload for one batch size."""

    def __init__(self, bs: int, H: int, dev, seed: int, l2_bytes: int, packed: bool = False,
                 N: int = DSTATE, state_dtype: str = "f32"):
        import torch

        import selective_state_update_02_gb300 as ssu
        import workloads as wl
        self.bs, self.H, self.N = bs, H, N
        self.elem_bytes = 2 if state_dtype == "bf16" else 4
        self.n_sets = sets_for(bs, H, l2_bytes, N, self.elem_bytes)
        rng = np.random.default_rng(seed)
        pool = wl.state_pool(rng, bs * self.n_sets, H, N=N, dtype=state_dtype)
        if state_dtype == "bf16":
            self.pool = torch.from_numpy(pool.view(np.int16)).view(torch.bfloat16).to(dev)
        else:
            self.pool = torch.from_numpy(pool).to(dev)
        del pool
        self.sets = torch.from_numpy(wl.rotation_sets(bs, self.n_sets, seed).astype(np.int32)) \
            .to(dev)
        dt_bias, A, D = wl.head_params(rng, H)
        self.dt_bias = torch.from_numpy(dt_bias).to(dev).unsqueeze(-1).expand(H, HEADDIM)
        self.A = torch.from_numpy(A).to(dev)[:, None, None].expand(H, HEADDIM, N)
        self.D = torch.from_numpy(D).to(dev).unsqueeze(-1).expand(H, HEADDIM)
        # per set: x, B, C as strided views of one packed bf16 tensor, dt head-expanded
        width = H * HEADDIM + 2 * NGROUPS * N
        self.packed = torch.from_numpy(
            wl.packed_xbc(rng, bs * self.n_sets, H, N=N).view(np.int16)).view(torch.bfloat16) \
            .to(dev).view(self.n_sets, bs, width)
        self.dt = torch.from_numpy(wl.f32_to_bf16_bits(
            rng.uniform(-4, 0, (self.n_sets, bs, H)).astype(np.float32)).view(np.int16)) \
            .view(torch.bfloat16).to(dev)
        self.out = torch.zeros(self.n_sets, bs, H, HEADDIM, dtype=torch.bfloat16, device=dev)
        self.args = []
        for k in range(self.n_sets):
            pk = self.packed[k]
            x = pk[:, :H * HEADDIM].view(bs, H, HEADDIM)
            B = pk[:, H * HEADDIM:H * HEADDIM + N].unsqueeze(1)
            C = pk[:, H * HEADDIM + N:].unsqueeze(1)
            dt = self.dt[k].unsqueeze(-1).expand(bs, H, HEADDIM)
            tensors = (self.pool, self.sets[k], x, dt, self.dt_bias, self.A, B, C, self.D,
                       self.out[k])
            shape, strides = ssu.describe(*tensors)
            self.args.append(([t.data_ptr() for t in tensors], shape, strides))
        self.packed_layout = packed

    def call(self, handle, i: int, stream_ptr: int) -> None:
        import selective_state_update_02_gb300 as ssu
        ptrs, shape, strides = self.args[i % self.n_sets]
        st = ssu.ssu_update_raw(handle, ptrs, shape, strides, stream_ptr)
        if st != 0:
            raise ssu.SsuError(st, "ssu_update", ssu.last_error())


def time_calls(wl_, handle, steps: int, warmup: int, clocks_gpu: int | None = None,
               repeats: int = 1, barrier=None):
    """Warm up, then time exactly `steps` calls replayed from CUDA graphs, `repeats` times
    (each repeat bracketed by `barrier` (if any), a device synchronisation and CUDA events on
    the launching stream).

    Returns (elapsed_ms per repeat, untimed_calls, clocks).
    """
    import torch
    stream = torch.cuda.Stream()
    per_graph = wl_.n_sets * max(1, math.ceil(200 / wl_.n_sets))
    per_graph = min(per_graph, max(steps, 1))
    full, rem = divmod(steps, per_graph)
    with torch.cuda.stream(stream):
        for i in range(warmup):
            wl_.call(handle, i, stream.cuda_stream)
    stream.synchronize()
    graphs = []
    for n in ([per_graph] if full else []) + ([rem] if rem else []):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            cur = torch.cuda.current_stream().cuda_stream
            for i in range(n):
                wl_.call(handle, i, cur)
        graphs.append((g, n))
    # one untimed replay of each graph (uploads it and warms the launch path)
    untimed = warmup
    with torch.cuda.stream(stream):
        for g, n in graphs:
            g.replay()
            untimed += n
    stream.synchronize()
    sampler = ClockSampler(clocks_gpu) if clocks_gpu is not None else None
    if sampler:
        sampler.__enter__()
    times = []
    for _ in range(repeats):
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if barrier is not None:
            barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            ev0.record(stream)
            if full:
                g, _ = graphs[0]
                for _ in range(full):
                    g.replay()
            if rem:
                graphs[-1][0].replay()
            ev1.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
        if barrier is not None:
            barrier()
        times.append(ev0.elapsed_time(ev1))
    clocks = None
    if sampler:
        sampler.__exit__(None, None, None)
        clocks = sampler.result()
    return times, untimed, clocks


def time_e2e(wl_, handle, steps: int, dev) -> dict:
    """Public-API path with host buffers, per step: the step's inputs (indices, x/B/C, dt)
    cross from pinned host memory to the device and the readout comes back to pinned host
    memory.  ``value`` is ssu_update_from_host (one C-ABI call per step); the copy-engine
    path (explicit copies around ssu_update) and the zero-copy path are reported beside it."""
    import torch

    import selective_state_update_02_gb300 as ssu
    bs, H, N = wl_.bs, wl_.H, wl_.N
    width = H * HEADDIM + 2 * N
    # one pinned staging buffer per step input set: [idx int32 | packed x/B/C | dt] as bytes
    n_idx, n_xbc, n_dt = bs * 4, bs * width * 2, bs * H * 2
    step_bytes = n_idx + n_xbc + n_dt
    host_in = torch.empty(wl_.n_sets, step_bytes, dtype=torch.uint8, pin_memory=True)
    for k in range(wl_.n_sets):
        host_in[k, :n_idx].copy_(wl_.sets[k].cpu().view(torch.uint8))
        host_in[k, n_idx:n_idx + n_xbc].copy_(wl_.packed[k].cpu().reshape(-1).view(torch.uint8))
        host_in[k, n_idx + n_xbc:].copy_(wl_.dt[k].cpu().reshape(-1).view(torch.uint8))
    dev_in = torch.empty(step_bytes, dtype=torch.uint8, device=dev)
    idx = dev_in[:n_idx].view(torch.int32)
    pk = dev_in[n_idx:n_idx + n_xbc].view(torch.bfloat16).view(bs, width)
    dt = dev_in[n_idx + n_xbc:].view(torch.bfloat16).view(bs, H).unsqueeze(-1) \
        .expand(bs, H, HEADDIM)
    x = pk[:, :H * HEADDIM].view(bs, H, HEADDIM)
    B = pk[:, H * HEADDIM:H * HEADDIM + N].unsqueeze(1)
    C = pk[:, H * HEADDIM + N:].unsqueeze(1)
    out = torch.empty(bs, H, HEADDIM, dtype=torch.bfloat16, device=dev)
    host_out = torch.empty(wl_.n_sets, bs, H, HEADDIM, dtype=torch.bfloat16, pin_memory=True)
    stream = torch.cuda.Stream()

    def step(k):
        dev_in.copy_(host_in[k], non_blocking=True)
        ssu.ssu_update(handle, wl_.pool, idx, x, dt, wl_.dt_bias, wl_.A, B, C, wl_.D, out,
                       stream)
        host_out[k].copy_(out, non_blocking=True)

    with torch.cuda.stream(stream):
        for i in range(5):
            step(i % wl_.n_sets)
    stream.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(steps):
            step(i % wl_.n_sets)
        ev1.record(stream)
    stream.synchronize()
    ms = ev0.elapsed_time(ev1)
    # The same calls captured once in a CUDA graph (copies from and to the same pinned host
    # buffers are graph nodes), as a serving loop that replays its decode step would run them.
    g = torch.cuda.CUDAGraph()
    per_graph = wl_.n_sets * max(1, math.ceil(100 / wl_.n_sets))
    with torch.cuda.graph(g, stream=stream):
        for i in range(per_graph):
            step(i % wl_.n_sets)
    g.replay()
    stream.synchronize()
    reps = max(10, steps // per_graph)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(reps):
            g.replay()
        ev1.record(stream)
    stream.synchronize()
    graph_us = ev0.elapsed_time(ev1) * 1000.0 / (reps * per_graph)

    # Zero-copy: the kernel reads the step's inputs straight from the pinned host buffer and
    # writes the readout straight into pinned host memory (coherent over the CPU-GPU link);
    # no copy call, the same bytes cross the link.
    host_views = []
    for k in range(wl_.n_sets):
        hk = host_in[k]
        hpk = hk[n_idx:n_idx + n_xbc].view(torch.bfloat16).view(bs, width)
        host_views.append((hk[:n_idx].view(torch.int32), hpk[:, :H * HEADDIM].view(bs, H, HEADDIM),
                           hk[n_idx + n_xbc:].view(torch.bfloat16).view(bs, H).unsqueeze(-1)
                           .expand(bs, H, HEADDIM),
                           hpk[:, H * HEADDIM:H * HEADDIM + N].unsqueeze(1),
                           hpk[:, H * HEADDIM + N:].unsqueeze(1)))

    def zstep(k):
        hidx, hx, hdt, hB, hC = host_views[k]
        ssu.ssu_update(handle, wl_.pool, hidx, hx, hdt, wl_.dt_bias, wl_.A, hB, hC, wl_.D,
                       host_out[k], stream)

    with torch.cuda.stream(stream):
        for i in range(5):
            zstep(i % wl_.n_sets)
    stream.synchronize()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(steps):
            zstep(i % wl_.n_sets)
        ev1.record(stream)
    stream.synchronize()
    zero_us = ev0.elapsed_time(ev1) * 1000.0 / steps

    # The host-operand entry point, called through the C ABI with the step's pinned host
    # buffers: a staging kernel reads the indices/x/B/C/dt across the link in one pass into a
    # device workspace, the decode-step kernel follows as a programmatic dependent and writes
    # the readout straight into pinned host memory.
    host_calls = []
    ws = None
    for k in range(wl_.n_sets):
        hidx, hx, hdt, hB, hC = host_views[k]
        tensors = (wl_.pool, hidx, hx, hdt, wl_.dt_bias, wl_.A, hB, hC, wl_.D, host_out[k])
        shape, strides = ssu.describe(*tensors)
        if ws is None:
            ws = torch.empty(ssu.ssu_host_workspace_bytes(shape), dtype=torch.uint8,
                             device=dev)
        host_calls.append(([t.data_ptr() for t in tensors], shape, strides))
    ws_ptr, ws_bytes = ws.data_ptr(), ws.numel()

    def hstep(k, s_ptr):
        ptrs, shape, strides = host_calls[k]
        st = ssu.ssu_update_from_host_raw(handle, ptrs, shape, strides, ws_ptr, ws_bytes, s_ptr)
        if st != 0:
            raise ssu.SsuError(st, "ssu_update_from_host", ssu.last_error())

    with torch.cuda.stream(stream):
        for i in range(5):
            hstep(i % wl_.n_sets, stream.cuda_stream)
    stream.synchronize()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(steps):
            hstep(i % wl_.n_sets, stream.cuda_stream)
        ev1.record(stream)
    stream.synchronize()
    host_us = ev0.elapsed_time(ev1) * 1000.0 / steps
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=stream):
        cur = torch.cuda.current_stream().cuda_stream
        for i in range(per_graph):
            hstep(i % wl_.n_sets, cur)
    g2.replay()
    stream.synchronize()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(reps):
            g2.replay()
        ev1.record(stream)
    stream.synchronize()
    host_graph_us = ev0.elapsed_time(ev1) * 1000.0 / (reps * per_graph)
    return {"value": round(host_us, 3), "unit": UNIT, "steps": steps,
            "h2d_bytes_per_step": step_bytes, "d2h_bytes_per_step": bs * H * HEADDIM * 2,
            "path": "C ABI ssu_update_from_host per step on pinned host buffers (staging "
                    "kernel for the inputs, readout written to host memory), eager",
            "graph_value": round(host_graph_us, 3),
            "graph_path": "the same calls captured in a CUDA graph",
            "copy_engine_value": round(ms * 1000.0 / steps, 3),
            "copy_engine_path": "one cudaMemcpyAsync of the inputs (pinned host to device), "
                                "ssu_update, one cudaMemcpyAsync of the readout back, eager",
            "copy_engine_graph_value": round(graph_us, 3),
            "zero_copy_value": round(zero_us, 3),
            "zero_copy_path": "ssu_update reading inputs from and writing out to pinned host "
                              "memory directly (no copy calls), eager"}


# ---- the oracle on the host cores -----------------------------------------------------------

class OracleCall:
    """One decode step of the batch run by the double-precision oracle on the host cores."""

    def __init__(self, bs: int, H: int, seed: int, N: int = DSTATE):
        import oracle
        import workloads as wl
        oracle.build()
        self.oracle = oracle
        rng = np.random.default_rng(seed)
        # the call's own slots: a pool of bs slots addressed by a random permutation
        self.pool0 = wl.state_pool(rng, bs, H, N=N).astype(np.float64)
        self.idx = rng.permutation(bs).astype(np.int64)
        self.dt_bias, self.A, self.D = wl.head_params(rng, H)
        self.x, self.dt, self.B, self.C = wl.request_inputs(rng, bs, H, N=N)
        self.bs = bs
        self.threads = os.cpu_count() or 1
        self.pool = self.pool0.copy()

    def run(self, requests: int | None = None) -> float:
        """Seconds of one oracle call over the first `requests` requests (all by default),
        timed around the call alone; the pool is refreshed from its initial copy outside the
        timed region (the state values only drift, so each call does the same work)."""
        n = self.bs if requests is None else max(1, min(self.bs, requests))
        np.copyto(self.pool, self.pool0)
        t0 = time.perf_counter()
        self.oracle.ssu_step_inplace(self.pool, self.idx[:n], self.x[:n], self.dt[:n],
                                     self.dt_bias, self.A, self.B[:n], self.C[:n], self.D,
                                     threads=self.threads)
        return time.perf_counter() - t0


def oracle_call_us(oc: OracleCall, calls: int, requests: int, warmup: int = 1) -> tuple:
    """The oracle's µs per full-batch call: `warmup` untimed calls, then `calls` timed calls
    over `requests` requests each, scaled by bs / requests; (median, per-call list).  The
    reference arm and the cpu_baseline leg both time the oracle with this one routine."""
    for _ in range(warmup):
        oc.run(requests)
    per = [oc.run(requests) * (oc.bs / requests) * 1e6 for _ in range(calls)]
    return statistics.median(per), per


def cpu_baseline(bs: int, H: int, budget_s: float = 12.0, N: int = DSTATE) -> dict:
    oc = OracleCall(bs, H, seed=7, N=N)
    t_full = oc.run()
    calls = int(max(3, min(50, budget_s / max(t_full, 1e-6))))
    med, per = oracle_call_us(oc, calls, bs)
    # the same oracle on one thread, over a quarter of the batch (scaled to the full call)
    threads, oc.threads = oc.threads, 1
    quarter = max(1, bs // 4)
    single, _ = oracle_call_us(oc, 3, quarter)
    oc.threads = threads
    return {"value": round(med, 1), "unit": UNIT, "cores": oc.threads, "kind": "oracle",
            "sample": f"{calls} full calls (batch {bs}, {H} heads, headdim 64, dstate {N}) "
                      f"of the fp64 C oracle split over {oc.threads} host threads (one "
                      f"persistent pool), each timed around the call alone; median",
            "single_thread_value": round(single, 1),
            "single_thread_sample": f"3 calls over {quarter} of the {bs} requests on one "
                                    f"thread, scaled to the full batch; median"}


def cpu_baseline_tokens(bs: int, H: int, T: int, budget_s: float = 6.0) -> dict:
    """The oracle's multi-token step (the single step applied T times, intermediate states
    kept) on a bounded sample of the batch, scaled to the full call."""
    import oracle
    import workloads as wl
    oracle.build()
    rng = np.random.default_rng(11)
    pool = wl.state_pool(rng, bs, H)
    idx = rng.permutation(bs).astype(np.int64)
    dt_bias, A, D = wl.head_params(rng, H)
    per_tok = [wl.request_inputs(rng, bs, H) for _ in range(T)]
    x, dt, B, C = (np.stack([pt[i] for pt in per_tok], axis=1) for i in range(4))
    req = max(1, bs // 16)
    oracle.ssu_tokens(pool[:0], idx[:0], x[:0], dt[:0], dt_bias, A, B[:0], C[:0], D)
    times = []
    t_start = time.perf_counter()
    while time.perf_counter() - t_start < budget_s and len(times) < 20:
        sub = np.ascontiguousarray(pool[:req])
        t0 = time.perf_counter()
        oracle.ssu_tokens(sub, np.arange(req), x[:req], dt[:req], dt_bias, A, B[:req], C[:req],
                          D)
        times.append((time.perf_counter() - t0) * (bs / req))
    return {"value": round(statistics.median(times) * 1e6, 1), "unit": UNIT, "cores": 1,
            "kind": "oracle",
            "sample": f"{len(times)} runs of the oracle's {T}-token step (fp64 C single step "
                      f"applied {T} times, intermediate states kept) over {req} of the {bs} "
                      f"requests ({H} heads, headdim 64, dstate 128) on one thread, scaled "
                      f"to the full batch; median"}


def cpu_baseline_copy(reqs: int, budget_s: float = 6.0) -> dict:
    """The oracle's block copy (plain numpy assignment) of the page's per-request blocks, on a
    bounded sample of the requests, scaled to the full call."""
    import oracle
    rng = np.random.default_rng(13)
    blocks = 4
    tensors = ([rng.standard_normal((blocks,) + COPY_TEMPORAL, dtype=np.float32)
                for _ in range(COPY_LAYERS)] +
               [rng.integers(0, 2 ** 16, (blocks,) + COPY_CONV, dtype=np.uint16)
                for _ in range(COPY_LAYERS)])
    src, dst = np.array([0, 1]), np.array([2, 3])
    times = []
    t_start = time.perf_counter()
    while time.perf_counter() - t_start < budget_s and len(times) < 20:
        t0 = time.perf_counter()
        oracle.copy_blocks(tensors, src, dst)
        times.append((time.perf_counter() - t0) * reqs / len(src))
    return {"value": round(statistics.median(times) * 1e6, 1), "unit": UNIT, "cores": 1,
            "kind": "oracle",
            "sample": f"{len(times)} runs of the oracle's copy (numpy; it copies each whole "
                      f"tensor before assigning blocks) over {len(src)} requests of the page's "
                      f"{2 * COPY_LAYERS} tensors with {blocks} blocks each, on one thread, "
                      f"scaled to {reqs} requests; median"}


# ---- main ---------------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def run_reference(args) -> None:
    """The reference arm: the fp64 oracle on the host cores, timed by the routine the
    cpu_baseline leg uses (oracle_call_us); each step is one oracle call over a sample of the
    requests sized so the whole run stays within about two minutes, scaled to the full
    batch; the median step is reported."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    bs, H = args.batch, NHEADS
    oc = OracleCall(bs, H, seed=7)
    t_full = min(oc.run() for _ in range(2))
    budget = 120.0
    total = args.steps + args.warmup
    req = max(1, min(bs, int(bs * budget / max(total * t_full, 1e-9))))
    value, per = oracle_call_us(oc, args.steps, req, warmup=args.warmup)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(value / 1000.0, 4), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_for(bs, sets_for(bs, H, 126 * 2 ** 20)),
        "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": oc.threads,
                         "kind": "oracle",
                         "sample": f"each step: the fp64 C oracle on {req} of {bs} requests "
                                   f"({H} heads) over {oc.threads} host threads (one "
                                   f"persistent pool), timed around the call alone and scaled "
                                   f"to the full batch; median of {args.steps} steps"},
        "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_for(bs: int, n_sets: int, N: int = DSTATE, state_dtype: str = "f32",
               H: int = NHEADS) -> dict:
    eb = 2 if state_dtype == "bf16" else 4
    return {"workload": f"decode step, batch {bs}, {H} heads, headdim {HEADDIM}, dstate "
                        f"{N}, {state_dtype} state pool of {bs * n_sets} slots in {n_sets} "
                        f"disjoint {bs}-slot rotation sets; x/B/C strided views of one packed "
                        f"bf16 tensor, dt/A/D/dt_bias stride-0 broadcasts",
            "batch": bs, "nheads": H, "headdim": HEADDIM, "dstate": N,
            "state_dtype": state_dtype, "ngroups": NGROUPS, "pool_slots": bs * n_sets,
            "l2": f"inputs larger than L2: call i touches set i mod {n_sets}; the sets hold "
                  f"{bs * n_sets * H * HEADDIM * N * eb / 2 ** 20:.0f} MiB of state"}


REPEATS = 5  # timed repeats per measurement; the median is reported (the pages' protocol)


def median_call_us(wl_, handle, steps: int, warmup: int, repeats: int = REPEATS) -> tuple:
    """(median µs per call over `repeats` timed runs of `steps` calls, per-repeat µs/call)."""
    ms, _, _ = time_calls(wl_, handle, steps, warmup, repeats=repeats)
    per = [m * 1000.0 / steps for m in ms]
    return statistics.median(per), per


def batch_line(b: int, handle, dev, l2: int, steps: int, warmup: int, H: int = NHEADS,
               seed: int = 0) -> dict:
    """µs per call (median of REPEATS runs of `steps` calls) and TB/s of one batch size."""
    import torch
    w = Workload(b, H, dev, seed=seed, l2_bytes=l2)
    us, per = median_call_us(w, handle, steps, warmup)
    rec = {"us_per_call": round(us, 3),
           "tbps": round(bytes_per_call(b, H=H) / (us * 1e-6) / 1e12, 3),
           "steps": steps, "repeats": len(per), "repeat_us": [round(v, 3) for v in per],
           "sets": w.n_sets}
    del w
    torch.cuda.empty_cache()
    return rec


def run_ours(args) -> None:
    import torch
    import torch.distributed as dist

    import selective_state_update_02_gb300 as ssu
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the kernels have no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    ssu.lib()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    handle = ssu.ssu_create(local)
    if args.launch:
        ssu.ssu_set_launch_override(handle, args.launch)
    ssu.ssu_set_pdl(handle, not args.no_pdl)
    warmup = max(args.warmup, 3)
    bs = args.batch
    N, sdt = args.dstate, args.state_dtype
    eb = 2 if sdt == "bf16" else 4
    default_workload = N == DSTATE and sdt == "f32"
    main = Workload(bs, NHEADS, dev, seed=rank, l2_bytes=l2, packed=True, N=N, state_dtype=sdt)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # The headline: REPEATS timed runs of exactly `steps` calls, each bracketed by a barrier
    # and a device synchronisation; per run the slowest rank's time; the median run reported.
    ms, untimed, clocks = time_calls(main, handle, args.steps, warmup,
                                     clocks_gpu=_smi_index(local), repeats=REPEATS,
                                     barrier=barrier)
    runs = [max(gather_elapsed(m * 1000.0, world, dev)) for m in ms]
    slowest = statistics.median(runs)
    value = aggregate_value([slowest] * world, args.steps)
    per_launch_us = slowest / args.steps
    peaks = load_peaks()
    bpc = bytes_per_call(bs, N=N, state_bytes=eb)
    achieved_gbs = bpc / (per_launch_us * 1e-6) / 1e9
    launch = ssu.ssu_get_launch(handle, main.args[0][1])
    tag = f"batch{bs}"
    if not default_workload:
        tag += f"-n{N}-{sdt}"
    traffic = recorded_traffic(tag)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": warmup, "repeats": REPEATS,
        "repeat_us_per_call": [round(r / args.steps, 3) for r in runs],
        "untimed_calls": untimed,
        "ms_per_step": round(value / 1000.0, 6),
        "higher_is_better": False, "scaling": "weak",
        "vs_baseline": (round(value / PAGE_US[bs], 4)
                        if bs in PAGE_US and world == 1 and default_workload else None),
        "vs_baseline_note": "value / the pages' B200 Triton time for this batch (another "
                            "machine: context, not the target)",
        "dtype": "f32", "data": "synthetic",
        "config": config_for(bs, main.n_sets, N, sdt) | {
            "launch": {"mode": launch[0], "rows_per_warp": launch[1],
                       "warps_per_cta": launch[2], "stages": launch[3],
                       "programmatic_dependent_launch": not args.no_pdl},
            "timing": f"median of {REPEATS} timed runs of {args.steps} graph-replayed calls"},
        "achieved_tbps": round(achieved_gbs / 1000.0, 3),
        "pct_of_nominal_8tbps": round(100.0 * achieved_gbs / NOMINAL_HBM_GBS, 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved_gbs, 1),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved_gbs / peaks["hbm_gbs"], 4),
                     "traffic": traffic, "algorithmic_bytes_per_launch": bpc,
                     "peak_source": peaks["source"],
                     "kernel": "ssu_vec_kernel"},
        "gpu_launches": args.steps * REPEATS,
        "clocks": clocks,
    }
    if not args.skip_ceiling:
        state_bytes = bs * NHEADS * HEADDIM * N * eb
        t_in = same_size_ceiling(state_bytes, dev, l2)
        ceil_gbs = 2 * state_bytes / (t_in * 1e-6) / 1e9
        line["roofline"]["same_size_inplace_gbs"] = round(ceil_gbs, 1)
        line["roofline"]["frac_of_same_size_inplace"] = round(
            (2 * state_bytes / (per_launch_us * 1e-6) / 1e9) / ceil_gbs, 4)
    if not args.skip_extra and world == 1 and default_workload:
        # Batches 8, 128 and 512, each over at least 2000 calls per run (the headline above
        # runs exactly `steps`); then the same with programmatic dependent launch off.
        by, no_pdl = {}, {}
        for b in (8, 128, 512):
            n = max(2000, min(args.steps, int(2e5 / max(b, 1))))
            by[str(b)] = batch_line(b, handle, dev, l2, n, warmup, seed=100 + b) | {
                "pages_b200_us": PAGE_US[b]}
        line["by_batch"] = by
        ssu.ssu_set_pdl(handle, False)
        for b in (8, 128, 512):
            n = max(2000, min(args.steps, int(2e5 / max(b, 1))))
            no_pdl[str(b)] = batch_line(b, handle, dev, l2, n, warmup, seed=100 + b)
        ssu.ssu_set_pdl(handle, not args.no_pdl)
        line["no_pdl"] = no_pdl | {
            "note": "the same calls launched without programmatic dependent launch "
                    "(ssu_set_pdl(h, 0)): each call starts only after the previous one has "
                    "completed"}
    if not args.skip_e2e:
        line["e2e"] = time_e2e(main, handle, min(args.steps, args.e2e_steps), dev)
    if rank == 0 and world == 1 and not args.skip_cpu:
        line["cpu_baseline"] = cpu_baseline(bs, NHEADS, N=N)
    ssu.ssu_destroy(handle)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_head_sweep(args) -> None:
    """The head-count sweep workload: H = 8, 32, 64, 128 at batch 256, headdim 64, dstate
    128, fp32 state, a pool of at least 3x L2 with random non-contiguous indices; one JSON
    line per head count."""
    import torch

    import selective_state_update_02_gb300 as ssu
    dev = torch.device("cuda", 0)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    handle = ssu.ssu_create(0)
    ssu.ssu_set_pdl(handle, not args.no_pdl)
    peaks = load_peaks()
    bs = 256
    warmup = max(args.warmup, 3)
    for H in args.heads:
        w = Workload(bs, H, dev, seed=300 + H, l2_bytes=l2, packed=True)
        n = max(400, min(args.steps, int(4e5 / H)))
        us, per = median_call_us(w, handle, n, warmup)
        bpc = bytes_per_call(bs, H=H)
        gbs = bpc / (us * 1e-6) / 1e9
        launch = ssu.ssu_get_launch(handle, w.args[0][1])
        rec = {"metric": METRIC, "value": round(us, 3), "unit": UNIT, "n_gpus": 1,
               "steps": n, "warmup": warmup, "repeats": len(per),
               "repeat_us_per_call": [round(v, 3) for v in per],
               "higher_is_better": False, "dtype": "f32", "data": "synthetic",
               "config": config_for(bs, w.n_sets, H=H) | {
                   "launch": {"rows_per_warp": launch[1], "warps_per_cta": launch[2],
                              "programmatic_dependent_launch": not args.no_pdl}},
               "achieved_tbps": round(gbs / 1000.0, 3),
               "pct_of_nominal_8tbps": round(100.0 * gbs / NOMINAL_HBM_GBS, 1),
               "roofline": {"bound": "hbm", "achieved": round(gbs, 1),
                            "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": round(gbs / peaks["hbm_gbs"], 4),
                            "traffic": recorded_traffic(f"heads{H}-batch{bs}"),
                            "algorithmic_bytes_per_launch": bpc,
                            "peak_source": peaks["source"], "kernel": "ssu_vec_kernel"}}
        print(json.dumps(rec), flush=True)
        del w
        torch.cuda.empty_cache()
    assert ssu.ssu_get_error(handle) == (0, -1)
    ssu.ssu_destroy(handle)


def _smi_index(local: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        parts = [p for p in vis.split(",") if p.strip()]
        if local < len(parts) and parts[local].strip().isdigit():
            return int(parts[local])
    return local


def graph_time_us(fn, n_sets: int, calls: int = 400, reps: int = 3) -> float:
    """Best-of-`reps` time per call of `fn(i % n_sets)` replayed from one CUDA graph."""
    import torch
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for i in range(n_sets):
            fn(i)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(calls):
            fn(i % n_sets)
    g.replay()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            g.replay()
            e1.record(s)
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) * 1000.0 / calls)
    return best


def same_size_ceiling(nbytes: int, dev, l2_bytes: int, copy: bool = False) -> float:
    """µs per call of PyTorch's own in-place elementwise kernel (`mul_`, read + write of
    `nbytes`) or, with `copy`, of `copy_` between two buffers, over buffers rotated across
    at least 3x the L2: the rate a library kernel reaches at this call size."""
    import torch
    n_sets = max(3, -(-3 * l2_bytes // nbytes))
    bufs = [torch.randn(nbytes // 4, device=dev) for _ in range(n_sets)]
    if copy:
        dst = [torch.empty_like(b) for b in bufs]
        us = graph_time_us(lambda i: dst[i].copy_(bufs[i]), n_sets)
        del dst
    else:
        us = graph_time_us(lambda i: bufs[i].mul_(1.0000001), n_sets)
    del bufs
    torch.cuda.empty_cache()
    return us


def run_calibrate(args) -> None:
    """Library copy / in-place rates at the decode step's state sizes (batch 8, 128, 512)."""
    import torch
    dev = torch.device("cuda", 0)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    for bs in (8, 128, 512):
        nbytes = bs * NHEADS * HEADDIM * DSTATE * 4
        t_copy = same_size_ceiling(nbytes, dev, l2, copy=True)
        t_rmw = same_size_ceiling(nbytes, dev, l2)
        print(json.dumps({"batch": bs, "state_MiB": nbytes >> 20,
                          "copy_us": round(t_copy, 3),
                          "copy_tbps": round(2 * nbytes / t_copy / 1e6, 3),
                          "inplace_us": round(t_rmw, 3),
                          "inplace_tbps": round(2 * nbytes / t_rmw / 1e6, 3)}), flush=True)


# State-block copy workload (vLLM PR #48110, Test Plan / Microbenchmark): per request 24 fp32
# temporal blocks of 2 MiB and 24 bf16 conv blocks of 80 KiB (49.875 MiB copied), distinct
# source and destination blocks, at 1..128 requests.  Its GB200 figures (PR branch, GB/s of
# read + write) are context: another machine.
COPY_TEMPORAL = (32, 128, 128)     # fp32 elements per temporal block: 2 MiB
COPY_CONV = (10240, 4)             # bf16 elements per conv block: 80 KiB
COPY_LAYERS = 24
COPY_REQS = (1, 4, 8, 16, 32, 64, 128)
PAGE_COPY_GBS = {1: 479.4, 4: 1640.6, 8: 3050.0, 16: 4737.9, 32: 5900.6, 64: 5165.9,
                 128: 5788.0}


def copy_bytes_per_request() -> int:
    t = 4 * int(np.prod(COPY_TEMPORAL))
    c = 2 * int(np.prod(COPY_CONV))
    return COPY_LAYERS * (t + c)


class CopyWorkload:
    """48 state tensors whose blocks cover `n_sets` disjoint (src, dst) sets of `reqs`."""

    def __init__(self, reqs: int, dev, l2_bytes: int, seed: int = 0):
        import torch
        per_set = 2 * reqs * copy_bytes_per_request()
        self.n_sets = max(3, -(-3 * l2_bytes // per_set))
        blocks = 2 * reqs * self.n_sets
        gen = torch.Generator(device=dev).manual_seed(seed)
        self.tensors = []
        for _ in range(COPY_LAYERS):
            t = torch.empty((blocks,) + COPY_TEMPORAL, dtype=torch.float32, device=dev)
            t.uniform_(-1, 1, generator=gen)
            self.tensors.append(t)
        for _ in range(COPY_LAYERS):
            c = torch.empty((blocks,) + COPY_CONV, dtype=torch.bfloat16, device=dev)
            c.uniform_(-1, 1, generator=gen)
            self.tensors.append(c)
        perm = torch.from_numpy(np.random.default_rng(seed).permutation(blocks).astype(np.int32))
        perm = perm.view(self.n_sets, 2, reqs).to(dev)
        self.src = [perm[k, 0].contiguous() for k in range(self.n_sets)]
        self.dst = [perm[k, 1].contiguous() for k in range(self.n_sets)]
        self.reqs = reqs

    def call(self, handle, i: int, stream_ptr: int) -> None:
        import selective_state_update_02_gb300 as ssu
        k = i % self.n_sets
        ssu.ssu_copy_blocks(handle, self.tensors, self.src[k], self.dst[k], stream_ptr)


def run_copy(args) -> None:
    """Block-copy throughput (GB/s of read + write) at 1..128 requests, one JSON line each;
    with --sweep, every launch shape at 8, 32 and 128 requests instead."""
    import torch

    import selective_state_update_02_gb300 as ssu
    dev = torch.device("cuda", 0)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    handle = ssu.ssu_create(0)
    ssu.ssu_set_pdl(handle, not args.no_pdl)
    peaks = load_peaks()
    shapes = [None]
    reqs_list = tuple(args.copy_reqs)
    if args.sweep:
        reqs_list = (8, 32, 128)
        shapes = [(ssu.SSU_COPY_VEC, c, v, t) for c in (16, 32, 64) for v in (4, 8, 16)
                  for t in (128, 256)]
    cpu_copy = None
    for reqs in reqs_list:
        w = CopyWorkload(reqs, dev, l2)
        moved = 2 * reqs * copy_bytes_per_request()
        for shape in shapes:
            if shape is None:
                ssu.ssu_copy_set_launch(handle, ssu.SSU_COPY_AUTO)
            else:
                ssu.ssu_copy_set_launch(handle, *shape)
            n = max(w.n_sets * 4, min(400, int(2e5 / (moved / 6e6))))
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for i in range(3):
                    w.call(handle, i, stream.cuda_stream)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                cur = torch.cuda.current_stream().cuda_stream
                for i in range(n):
                    w.call(handle, i, cur)
            g.replay()
            torch.cuda.synchronize()
            best = float("inf")
            for _ in range(3):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    e0.record(stream)
                    g.replay()
                    e1.record(stream)
                torch.cuda.synchronize()
                best = min(best, e0.elapsed_time(e1) * 1000.0 / n)
            gbs = moved / (best * 1e-6) / 1e9
            rec = {"copy_reqs": reqs, "us_per_call": round(best, 3), "gbs": round(gbs, 1),
                   "frac_of_measured_peak": round(gbs / peaks["hbm_gbs"], 4),
                   "pages_gb200_gbs": PAGE_COPY_GBS.get(reqs), "calls": n, "sets": w.n_sets,
                   "launch": list(shape) if shape else "table",
                   "programmatic_dependent_launch": not args.no_pdl}
            if shape is None:
                rec["roofline"] = {
                    "bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                    "traffic": recorded_traffic(f"copy{reqs}", sources=COPY_SOURCES),
                    "algorithmic_bytes_per_launch": moved, "peak_source": peaks["source"],
                    "kernel": "copy_vec_kernel"}
                if not args.skip_cpu:
                    if cpu_copy is None:
                        cpu_copy = cpu_baseline_copy(1)
                    rec["cpu_baseline"] = cpu_copy | {
                        "value": round(cpu_copy["value"] * reqs, 1),
                        "sample": cpu_copy["sample"].replace("scaled to 1 requests",
                                                             f"scaled to {reqs} requests")}
            print(json.dumps(rec), flush=True)
            del g
        del w
        torch.cuda.empty_cache()
    ssu.ssu_copy_set_launch(handle, ssu.SSU_COPY_AUTO)
    assert ssu.ssu_get_error(handle) == (0, -1)
    ssu.ssu_destroy(handle)


def bytes_per_call_tokens(bs: int, T: int, intermediate: bool, H: int = NHEADS,
                          P: int = HEADDIM, N: int = DSTATE, G: int = NGROUPS,
                          state_bytes: int = 4) -> int:
    """Algorithmic bytes of one multi-token call: the state read and written once, T tokens of
    inputs and outputs, and (optionally) T intermediate states written."""
    state = 2 * bs * H * P * N * state_bytes
    per_token = bs * H * P * 2 * 2 + 2 * bs * G * N * 2 + bs * H * 2
    inter = T * bs * H * P * N * state_bytes if intermediate else 0
    return state + T * per_token + bs * 4 + 3 * H * 4 + inter


def run_e2e_only(args) -> None:
    """The e2e object alone (host-buffer paths) for the chosen batch, 16 heads."""
    import torch

    import selective_state_update_02_gb300 as ssu
    dev = torch.device("cuda", 0)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    handle = ssu.ssu_create(0)
    w = Workload(args.batch, NHEADS, dev, seed=5, l2_bytes=l2, packed=True)
    e2e = time_e2e(w, handle, args.e2e_steps, dev)
    print(json.dumps({"batch": args.batch, "e2e": e2e}), flush=True)
    assert ssu.ssu_get_error(handle) == (0, -1)
    ssu.ssu_destroy(handle)


def run_tokens(args) -> None:
    """Multi-token step at batch 128 (cold-L2 rotation): µs per call and GB/s for T = 1..4,
    with and without the intermediate-state output."""
    import torch

    import selective_state_update_02_gb300 as ssu
    import workloads as wl
    dev = torch.device("cuda", 0)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    handle = ssu.ssu_create(0)
    ssu.ssu_set_pdl(handle, not args.no_pdl)
    bs, H = args.batch, NHEADS
    N, sdt = args.dstate, args.state_dtype
    eb = 2 if sdt == "bf16" else 4
    w = Workload(bs, H, dev, seed=5, l2_bytes=l2, N=N, state_dtype=sdt)
    rng = np.random.default_rng(9)
    peaks = load_peaks()
    shapes = [None]
    tokens_list = tuple(args.tokens_list)
    if args.sweep:
        rpi = max(1, 512 // (N * eb))
        nc = (8 if sdt == "bf16" else 4) * max(1, N * eb // 512)
        ks = (2, 4, 8, 16) if (N == DSTATE and sdt == "f32") else (2, 4, 8)
        shapes = [(k * rpi, w) for k in ks if k * nc <= 64 for w in (1, 2, 4)]
        if tokens_list == (1, 2, 3, 4):  # the default list: sweep at 2 and 4 tokens
            tokens_list = (2, 4)
    cpu_by_t = {}
    for T in tokens_list:
        x = torch.from_numpy(wl.f32_to_bf16_bits(rng.standard_normal(
            (w.n_sets, bs, T, H, HEADDIM), dtype=np.float32)).view(np.int16)).view(
            torch.bfloat16).to(dev)
        bc = torch.from_numpy(wl.f32_to_bf16_bits(rng.standard_normal(
            (w.n_sets, 2, bs, T, 1, N), dtype=np.float32)).view(np.int16)).view(
            torch.bfloat16).to(dev)
        dt = torch.from_numpy(wl.f32_to_bf16_bits(rng.uniform(
            -4, 0, (w.n_sets, bs, T, H)).astype(np.float32)).view(np.int16)).view(
            torch.bfloat16).to(dev)
        out = torch.empty(bs, T, H, HEADDIM, dtype=torch.bfloat16, device=dev)
        for shape, with_inter in [(sh, wi) for sh in shapes
                                  for wi in ((False,) if args.sweep else (False, True))]:
            if shape is None:
                ssu.ssu_set_launch_override(handle, args.launch or "auto")
            else:
                ssu.ssu_set_launch(handle, ssu.SSU_MODE_VEC, shape[0], shape[1])
            inter = (torch.empty(bs, T, H, HEADDIM, N, device=dev,
                                 dtype=torch.bfloat16 if sdt == "bf16" else torch.float32)
                     if with_inter else None)

            def call(i, stream_ptr, T=T, x=x, bc=bc, dt=dt, out=out, inter=inter):
                k = i % w.n_sets
                ssu.ssu_update_tokens(handle, w.pool, w.sets[k], x[k], dt[k], w.dt_bias, w.A,
                                      bc[k, 0], bc[k, 1], w.D, out, inter, stream_ptr)

            n = max(w.n_sets * 4, 400)
            us = graph_time_us(lambda i: call(i, torch.cuda.current_stream().cuda_stream),
                               w.n_sets, calls=n)
            moved = bytes_per_call_tokens(bs, T, with_inter, N=N, state_bytes=eb)
            gbs = moved / (us * 1e-6) / 1e9
            rec = {"tokens": T, "batch": bs, "intermediate": with_inter, "dstate": N,
                   "state_dtype": sdt,
                   "launch": list(shape) if shape else (args.launch or "table"),
                   "programmatic_dependent_launch": not args.no_pdl,
                   "us_per_call": round(us, 3), "us_per_token": round(us / T, 3),
                   "gbs": round(gbs, 1),
                   "frac_of_measured_peak": round(gbs / peaks["hbm_gbs"], 4)}
            if shape is None:
                tag = f"tokens{T}-batch{bs}" + ("-inter" if with_inter else "") + (
                    "" if (N == DSTATE and sdt == "f32") else f"-n{N}-{sdt}")
                kern = tokens_kernel(T, with_inter, N, sdt, bool(args.launch))
                rec["roofline"] = {
                    "bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                    "traffic": recorded_traffic(
                        tag, sources=MMA_SOURCES if kern == "ssu_tokens_mma_kernel"
                        else TOKENS_SOURCES),
                    "algorithmic_bytes_per_launch": moved, "peak_source": peaks["source"],
                    "kernel": kern}
                if not args.skip_cpu and N == DSTATE and sdt == "f32":
                    if T not in cpu_by_t:
                        cpu_by_t[T] = cpu_baseline_tokens(bs, H, T)
                    rec["cpu_baseline"] = cpu_by_t[T]
            print(json.dumps(rec), flush=True)
            del inter
        del x, bc, dt, out
        torch.cuda.empty_cache()
    assert ssu.ssu_get_error(handle) == (0, -1)
    ssu.ssu_destroy(handle)


def sweep_shapes(N: int, state_dtype: str) -> list[tuple[int, int, int, int]]:
    """Every launch shape of the bucket: rows per warp = rows per vector instruction x
    {1, 2, 4, 8} (and 16 for an fp32 state of dstate 128), 1 to 8 warps per CTA."""
    rpi = max(1, 512 // (N * (2 if state_dtype == "bf16" else 4)))
    rows = [rpi * k for k in (1, 2, 4, 8)]
    if N == DSTATE and state_dtype == "f32":
        rows.append(16)
    return [(1, r, w, 0) for r in rows for w in (1, 2, 4, 8)]


def run_sweep(args) -> None:
    """Launch-shape sweep: every (rows per warp, warps per CTA) at batch 8, 128 and 512 on the
    cold-L2 rotation workloads; one JSON line per point, then the fastest shape per batch."""
    import torch

    import selective_state_update_02_gb300 as ssu
    dev = torch.device("cuda", 0)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    handle = ssu.ssu_create(0)
    best = {}
    for bs in args.sweep_batches:
        N, sdt = args.dstate, args.state_dtype
        eb = 2 if sdt == "bf16" else 4
        w = Workload(bs, NHEADS, dev, seed=200 + bs, l2_bytes=l2, N=N, state_dtype=sdt)
        shapes = sweep_shapes(N, sdt)
        n = max(1000, int(args.sweep_us_budget / (0.16 * bs + 2.0)))
        for mode, rpw, wpc, stages in shapes:
            ssu.ssu_set_launch(handle, mode, rpw, wpc, stages)
            us, _ = median_call_us(w, handle, n, 5, repeats=3)
            rec = {"batch": bs, "mode": "vec", "rows_per_warp": rpw,
                   "warps_per_cta": wpc, "stages": stages, "us_per_call": round(us, 3),
                   "tbps": round(bytes_per_call(bs, N=N, state_bytes=eb) / (us * 1e-6) / 1e12, 3),
                   "steps": n, "dstate": N, "state_dtype": sdt}
            print(json.dumps(rec), flush=True)
            if bs not in best or us < best[bs]["us_per_call"]:
                best[bs] = rec
        ssu.ssu_set_launch(handle, ssu.SSU_MODE_AUTO)
        us, _ = median_call_us(w, handle, n, 5, repeats=3)
        launch = ssu.ssu_get_launch(handle, w.args[0][1])
        print(json.dumps({"batch": bs, "mode": "table", "launch": launch,
                          "us_per_call": round(us, 3)}), flush=True)
        del w
        torch.cuda.empty_cache()
    print(json.dumps({"best": best}), flush=True)
    ssu.ssu_destroy(handle)


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--batch", type=int, default=DEFAULT_BATCH,
                    help="requests per call (the pages' workloads: 8, 128, 512)")
    ap.add_argument("--head-sweep", action="store_true",
                    help="the head-count sweep instead: H = --heads at batch 256")
    ap.add_argument("--heads", type=int, nargs="+", default=[8, 32, 64, 128],
                    help="head counts timed by --head-sweep")
    ap.add_argument("--dstate", type=int, default=DSTATE, choices=[64, 128, 256])
    ap.add_argument("--state-dtype", default="f32", choices=["f32", "bf16"])
    ap.add_argument("--e2e-steps", type=int, default=5000)
    ap.add_argument("--skip-extra", action="store_true", help="skip the batch 8/512 lines")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--launch", default="",
                    help="force a launch shape 'rows_per_warp,warps_per_cta' (the string "
                         "ssu_set_launch_override takes) instead of the built-in table")
    ap.add_argument("--tokens", action="store_true",
                    help="multi-token step (T = 1..4) at --batch instead")
    ap.add_argument("--copy", action="store_true",
                    help="state-block copy throughput instead (with --sweep: its shapes)")
    ap.add_argument("--no-pdl", action="store_true",
                    help="launch without programmatic dependent launch (ssu_set_pdl(h, 0)); "
                         "it is on by default")
    ap.add_argument("--sweep", action="store_true", help="launch-shape sweep instead")
    ap.add_argument("--calibrate", action="store_true",
                    help="library copy / in-place rates at the call sizes instead")
    ap.add_argument("--copy-reqs", type=int, nargs="+", default=list(COPY_REQS),
                    help="request counts timed by --copy")
    ap.add_argument("--tokens-list", type=int, nargs="+", default=[1, 2, 3, 4],
                    help="token counts timed by --tokens")
    ap.add_argument("--e2e-only", action="store_true",
                    help="only the host-buffer (e2e) measurements at the chosen batch")
    ap.add_argument("--skip-ceiling", action="store_true",
                    help="skip the same-size in-place ceiling measurement")
    ap.add_argument("--sweep-batches", type=int, nargs="+", default=[8, 128, 512])
    ap.add_argument("--sweep-us-budget", type=float, default=60000.0,
                    help="approximate GPU time per sweep point, microseconds")
    args = ap.parse_args()
    if args.steps < 1:
        raise SystemExit("--steps must be >= 1")
    if args.batch < 1:
        raise SystemExit("--batch must be >= 1")
    if args.tokens:
        run_tokens(args)
    elif args.copy:
        run_copy(args)
    elif args.calibrate:
        run_calibrate(args)
    elif args.sweep:
        run_sweep(args)
    elif args.head_sweep:
        run_head_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    elif args.e2e_only:
        run_e2e_only(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
