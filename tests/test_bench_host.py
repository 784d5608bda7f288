"""Host logic of bench.py on the CPU: arguments, seeds, the algorithmic
byte count, the traffic record's source check (comment-insensitive), the
reference arm's JSON
line, and the multi-rank path (replicas sharded by request, timing taken as
the maximum over ranks) on two gloo ranks."""
import io
import json
import os
import socket
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_parse_args_defaults():
    a = bench.parse_args([])
    assert (a.gpus, a.steps, a.warmup, a.workload, a.impl) == (1, 10000, 50, "c3", "ours")
    assert a.warmup >= 3


def test_rank_seeds_are_distinct_and_reproducible():
    seeds = {bench.rank_seed(2, r, s) for r in range(8) for s in range(4)}
    assert len(seeds) == 32
    assert bench.rank_seed(2, 3, 1) == bench.rank_seed(2, 3, 1)


def test_algorithmic_bytes_by_hand():
    # Two requests, V = 10, bf16: g = 2 accepted all (bonus re-read, no q);
    # g = 3 rejected at 1 with T > 0 (re-read + q row); plus a greedy request
    # (no re-read) and an invalid one (k = -1: rows only).
    V, s = 10, 2
    small = lambda g: g * (4 + 4 + 32) + 4 + 4 + 4 * (g + 1) + 4
    expect = ((3 * V * s + V * s + small(2))
              + (4 * V * s + V * s + V * 4 + small(3))
              + (2 * V * s + small(1))
              + (3 * V * s + small(2)))
    got = bench.algorithmic_bytes([2, 3, 1, 2], [0.8, 1.0, 0.0, 1.0], [2, 1, 0, -1], V, s)
    assert got == expect


def test_recorded_traffic_needs_matching_sources(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "abc")
    f = tmp_path / "profiles" / "traffic_c3.json"
    f.write_text(json.dumps({"source_hash": "abc", "dram_bytes_per_step": 123}))
    assert bench.recorded_traffic("c3") == 123
    f.write_text(json.dumps({"source_hash": "old", "dram_bytes_per_step": 123}))
    assert bench.recorded_traffic("c3") is None
    assert bench.recorded_traffic("c9") is None


def test_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    csrc = tmp_path / "speculative_decoding_verification_75_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "include").mkdir()
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    k = csrc / "k.cuh"
    h = tmp_path / "include" / "a.h"
    h.write_text("/* api */\nint f(int);\n")
    k.write_text("// kernel\n__global__ void g(int *p) { p[0] = 1; }  // store\n")
    base = bench.kernel_source_hash()
    k.write_text("// kernel, reworded\n\n__global__ void g(int *p) { p[0] = 1; }\n")
    h.write_text("/* api,\n   two lines */\nint f(int);  // f\n")
    assert bench.kernel_source_hash() == base
    k.write_text("__global__ void g(int *p) { p[0] = 2; }\n")
    assert bench.kernel_source_hash() != base


def test_reference_arm_prints_one_json_line():
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.main(["--impl", "reference", "--workload", "c1", "--steps", "3",
                           "--warmup", "3"]) == 0
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 3
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1


def test_reference_arm_other_ranks_exit_quietly(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.main(["--impl", "reference", "--workload", "c1", "--steps", "3"]) == 0
    assert buf.getvalue().strip() == ""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.dist_env()
        step_ms = 1.0 + 0.5 * rank                    # per-rank timed region
        rows = 640 * (rank + 1)                       # per-rank work (replicas)
        t_max = bench.aggregate_max(step_ms, w)
        total = bench.aggregate_sum(rows, w)
        dist.barrier()
        results[rank] = (r, lr, w, t_max, total, bench.rank_seed(2, r, 0))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_bench():
    world = 2
    results = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True)
    got = [results[r] for r in range(world)]
    for rank, (r, lr, w, t_max, total, seed) in enumerate(got):
        assert (r, lr, w) == (rank, rank, world)
        assert t_max == 1.5                           # slowest rank sets the time
        assert total == 640 + 1280                    # whole-job work
    assert got[0][5] != got[1][5]                     # each rank draws its own requests
