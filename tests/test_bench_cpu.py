"""Host logic of bench.py: the algorithmic byte count (pinned to the figures the pages print),
clock parsing, the multi-rank aggregation (gloo, world size 2) and the reference arm."""

from __future__ import annotations

import json
import os
import subprocess
import sys
from pathlib import Path

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

ROOT = Path(__file__).resolve().parent.parent
GOLDEN = Path(__file__).resolve().parent / "golden"


def test_bytes_per_request_at_16_heads():
    # state 2*16*64*128*4 + x 2048 + y 2048 + B,C 512 + dt 32 + idx 4 per request
    assert bench.bytes_per_call(1) - 3 * 16 * 4 == 1_053_220
    assert bench.bytes_per_call(128) == 128 * 1_053_220 + 192


def test_bytes_reproduce_the_pages_bandwidths():
    # sglang PR #41223: batch 512 ran at 173.5 us before and 85.7 us after, which its
    # Summary quotes as about 3.1 -> 6.3 TB/s.
    table = json.loads((GOLDEN / "p1_kernel_table.json").read_text())
    row = [r for r in table["rows"] if r["batch"] == 512][0]
    q = table["quoted_tbps_batch512"]
    before = bench.bytes_per_call(512) / (row["baseline_us"] * 1e-6) / 1e12
    after = bench.bytes_per_call(512) / (row["pr_us"] * 1e-6) / 1e12
    assert abs(before - q["baseline"]) <= q["quoted_to"]
    assert abs(after - q["pr"]) <= q["quoted_to"]
    for r in table["rows"]:
        assert bench.PAGE_US[r["batch"]] == r["pr_us"]


def test_parse_clocks():
    csv = "\n".join([
        "0, 1965 MHz, 2070 MHz, 812.40 W, 0x0000000000000000, Not Active, Not Active, "
        "Not Active, Not Active",
        "0, 1980 MHz, 2070 MHz, 830.10 W, 0x0000000000000004, Not Active, Not Active, "
        "Not Active, Active",
        "0, 345 MHz, 2070 MHz, 120.00 W, 0x0000000000000001, Not Active, Not Active, "
        "Not Active, Not Active",
    ])
    c = bench.parse_clocks(csv)
    assert c["sm_mhz"] == pytest.approx(1972.5)
    assert c["sm_max_mhz"] == 2070 and c["reasons"] == ["sw_power_cap"] and c["samples"] == 3
    assert bench.parse_clocks("") is None


def test_aggregate_value_uses_the_slowest_rank():
    assert bench.aggregate_value([1000.0], 100) == 10.0
    assert bench.aggregate_value([1000.0, 1200.0], 100) == 6.0


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.gather_elapsed(100.0 * (rank + 1), world, torch.device("cpu"))
    q.put((rank, got, bench.aggregate_value(got, 10)))
    dist.destroy_process_group()


def test_gather_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, got, agg in res:
        assert got == [100.0, 200.0]
        assert agg == pytest.approx(200.0 / 20)


def test_recorded_traffic_needs_a_matching_source(tmp_path, monkeypatch):
    assert bench.recorded_traffic("no-such-workload") is None


def _run_bench(args, env_extra=None):
    env = dict(os.environ, **(env_extra or {}))
    return subprocess.run([sys.executable, str(ROOT / "bench.py"), *args], capture_output=True,
                          text=True, env=env, timeout=600)


def test_reference_arm_prints_one_line():
    r = _run_bench(["--impl", "reference", "--steps", "3", "--warmup", "1"])
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "us/call" and d["value"] > 0
    assert d["higher_is_better"] is False and d["steps"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_reference_arm_other_ranks_do_nothing():
    r = _run_bench(["--impl", "reference", "--steps", "3", "--warmup", "1"],
                   {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_copy_bytes_reproduce_the_copy_table():
    # 2 x (49.875 MiB per request) x reqs / latency reproduces every GB/s the page prints.
    table = json.loads((GOLDEN / "p2_copy_table.json").read_text())
    per_req = bench.copy_bytes_per_request()
    assert abs(per_req / 2 ** 20 - table["mib_per_request"]) < 0.01
    for r in table["rows"]:
        gbs = 2 * r["reqs"] * per_req / (r["us"] * 1e-6) / 1e9
        assert abs(gbs / r["gbs"] - 1) < 0.003, r
        assert bench.PAGE_COPY_GBS[r["reqs"]] == r["gbs"]


def test_token_bytes_reduce_to_single_step():
    # one token, no intermediate states: the single-step count
    assert bench.bytes_per_call_tokens(128, 1, False) == bench.bytes_per_call(128)
    # each extra token adds only its inputs and outputs; intermediates add T states
    extra = bench.bytes_per_call_tokens(128, 2, False) - bench.bytes_per_call(128)
    assert extra == 128 * (16 * 64 * 2 * 2 + 2 * 128 * 2 + 16 * 2)
    assert (bench.bytes_per_call_tokens(128, 3, True) - bench.bytes_per_call_tokens(128, 3, False)
            == 3 * 128 * 16 * 64 * 128 * 4)


def test_reference_arm_and_cpu_baseline_time_the_oracle_alike(capsys):
    # Both legs time the oracle with one routine (oracle_call_us: the oracle call alone, one
    # persistent thread pool, median over calls), so on the same host they agree; they
    # differed 3.4x when the reference arm's timed loop also held a copy of the pool per step.
    import argparse
    bs = 32
    base = bench.cpu_baseline(bs, 16, budget_s=1.0)
    args = argparse.Namespace(gpus=1, steps=6, warmup=1, batch=bs)
    bench.run_reference(args)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    ratio = line["value"] / base["value"]
    assert 0.6 < ratio < 1.6, (line["value"], base["value"])
    assert line["cpu_baseline"]["cores"] == base["cores"]


def test_token_kernel_names_follow_the_library_rule():
    # ssu_update_tokens: the chunked kernel without intermediates and without a forced shape,
    # fp32 state at dstate 64 / 128 from 5 tokens, bf16 at dstate 128 from 16; else general
    k = bench.tokens_kernel
    assert k(5, False, 128, "f32", False) == "ssu_tokens_mma_kernel"
    assert k(4, False, 128, "f32", False) == "ssu_tokens_kernel"
    assert k(8, False, 64, "f32", False) == "ssu_tokens_mma_kernel"
    assert k(8, True, 128, "f32", False) == "ssu_tokens_kernel"
    assert k(8, False, 128, "f32", True) == "ssu_tokens_kernel"
    assert k(8, False, 256, "f32", False) == "ssu_tokens_kernel"
    assert k(15, False, 128, "bf16", False) == "ssu_tokens_kernel"
    assert k(16, False, 128, "bf16", False) == "ssu_tokens_mma_kernel"
    assert k(64, False, 64, "bf16", False) == "ssu_tokens_kernel"
