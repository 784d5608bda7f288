#!/usr/bin/env python
"""Benchmark of the speculative-decoding verification step on GB300.

One *step* is one call of the C-ABI ``spec_verify`` (through the Python
binding) on one batch of the benchmark workload: B=128 requests, gamma=5
drafts, V=151936 (Qwen2.5 vocabulary), bf16 target logits with 1% of each
row boosted by +8 (peaky rows), draft noise 0.7, temperature 0.8.  The metric
is verified draft rows per second (sum of draft lengths per step / step
time); the roofline object reports the achieved HBM bandwidth of the step
against the measured copy bandwidth of the GB300s.

    python bench.py [--steps K] [--warmup W] [--workload c3] [--impl reference]
    torchrun --nproc-per-node N bench.py --gpus N   (weak scaling: B per GPU)

Prints ONE JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
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

L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0
KERNELS_PER_STEP = 1          # one kernel per step (B <= 256 or the cluster path; no histogram)
METRIC = "verified draft rows/sec"
UNIT = "rows/s"


# ------------------------------------------------------------ host logic ----

def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default="c3")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sets", type=int, default=0,
                    help="rotating input sets (0: enough to exceed 3x L2)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=20.0,
                    help="wall time of the CPU baseline (half single-thread, half all cores)")
    ap.add_argument("--sweep-steps", type=int, default=200,
                    help="calls timed per workload of the B x gamma x V sweep")
    ap.add_argument("--no-sweep", action="store_true")
    return ap.parse_args(argv)


def dist_env():
    """(rank, local_rank, world_size) from the torchrun environment."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def rank_seed(base: int, rank: int, set_idx: int) -> int:
    """Distinct, reproducible seed per rank and input set."""
    return base + 1_000_003 * rank + 7919 * set_idx


def algorithmic_bytes(lens, temperature, num_accepted, V, logit_bytes,
                      with_q=True) -> int:
    """Bytes the method must move for one batch: every target logit of the
    g_b+1 rows once, the re-read of the one row each sampled request draws
    from, the q row at each rejection, and the small per-position terms
    (draft id, uniform, one 32-byte sector for the q(x) gather, outputs)."""
    total = 0
    for g, t, k in zip(lens, temperature, num_accepted):
        g, k = int(g), int(k)
        total += (g + 1) * V * logit_bytes
        if t > 0 and k >= 0:
            total += V * logit_bytes
            if k < g and with_q:
                total += V * 4
        total += g * (4 + 4 + 32) + 4 + 4 + 4 * (g + 1) + 4
    return total


def aggregate_max(value: float, world: int) -> float:
    """Maximum of a per-rank float over all ranks (identity for one rank)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_sum(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def measured_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """C/CUDA source without comments or blank-line differences: an edit to
    a comment leaves the compiled kernels, and so this hash, unchanged."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    src = ROOT / "speculative_decoding_verification_75_gb300" / "csrc"
    for f in sorted(src.glob("*")) + sorted((ROOT / "include").glob("*.h")):
        h.update(f.name.encode())
        h.update(_code_only(f.read_text()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per step from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    f = ROOT / "profiles" / f"traffic_{workload}.json"
    if not f.exists():
        return None
    d = json.loads(f.read_text())
    if d.get("source_hash") != kernel_source_hash():
        return None
    return d.get("dram_bytes_per_step")


# ---------------------------------------------------------------- clocks ----

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                    "-i", str(gpu_index), "-lms", str(period_ms)]
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 8]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- our arm ----

def make_sets(W, w, dev, rank, min_bytes, max_sets):
    """Rotating input sets of workload ``w`` until they exceed ``min_bytes``
    (at least two, at most ``max_sets``).  Returns (cases, bytes per set)."""
    cases, set_bytes = [], 0
    while True:
        c = W.make_case(w, device=dev, seed=rank_seed(w.seed, rank, len(cases)))
        cases.append(c)
        set_bytes = sum(t.numel() * t.element_size() for t in c.values() if t is not None)
        if len(cases) >= max_sets or (len(cases) >= 2 and len(cases) * set_bytes >= min_bytes):
            return cases, set_bytes


def step_bytes(case, nacc, V):
    """Algorithmic bytes of one call on ``case`` given its num_accepted."""
    w_g = case["draft_ids"].shape[1]
    lens = (case["draft_lens"].cpu().tolist() if case["draft_lens"] is not None
            else [w_g] * case["draft_ids"].shape[0])
    return algorithmic_bytes(lens, case["temperature"].cpu().tolist(), nacc.cpu().tolist(), V,
                             case["logits"].element_size(), case["draft_probs"] is not None)


def time_workload(api, W, w, dev, steps, warmup, flush_buf=None):
    """Device time of one call of workload ``w``: rotating input sets larger
    than L2 timed back to back, or (sets too small to defeat L2) each call
    timed on its own with an L2 flush between calls.  Returns a dict."""
    import torch
    cases, set_bytes = make_sets(W, w, dev, 0, 3 * L2_BYTES, 32)
    rotate = len(cases) * set_bytes >= 3 * L2_BYTES
    bound = [api.bind(c["logits"], c["draft_ids"], c["draft_probs"], c["u_accept"],
                      c["u_sample"], c["temperature"], c["draft_lens"]) for c in cases]
    n = len(bound)
    for i in range(max(warmup, 3)):
        bound[i % n]()
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    if rotate:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            bound[i % n]()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) * 1e3 / steps
        how = f"{n} rotating input sets of {set_bytes / 1e6:.1f} MB, back to back"
    else:
        times = []
        for i in range(steps):
            flush_buf.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            bound[i % n]()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            times.append(e0.elapsed_time(e1) * 1e3)
        us = statistics.median(times)
        how = (f"median of {steps} single calls, L2 flushed ({flush_buf.numel() / 1e6:.0f} MB "
               f"written) before each")
    by = sum(step_bytes(c, b.out_num_accepted, w.V) for c, b in zip(cases, bound)) / n
    nacc = torch.cat([b.out_num_accepted for b in bound]).float()
    rows = W.verified_rows(cases[0])
    return {"us_per_step": us, "rows_per_s": rows / (us * 1e-6), "bytes_per_step": by,
            "alpha_hat": float(nacc[nacc >= 0].mean()) / max(w.gamma, 1), "timing": how}


def run_ours(args, rank, local_rank, world):
    import torch

    from speculative_decoding_verification_75_gb300 import api, verify_host
    from speculative_decoding_verification_75_gb300 import workloads as W

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    api.load_library()
    w = W.workload(args.workload)
    cases, set_bytes = make_sets(W, w, dev, rank, 3 * L2_BYTES if not args.sets else 0,
                                 args.sets or 64)
    nsets = len(cases)
    rows_per_step = W.verified_rows(cases[0])
    # The tensors of each set are bound once: a timed call is the C-ABI call
    # with marshalled arguments (host cost ~5 us, far below the step).
    bound = [api.bind(c["logits"], c["draft_ids"], c["draft_probs"], c["u_accept"],
                      c["u_sample"], c["temperature"], c["draft_lens"]) for c in cases]

    barrier = (lambda: __import__("torch.distributed").distributed.barrier()) if world > 1 \
        else (lambda: None)
    clocks = ClockSampler(local_rank)
    clocks.start()
    stream = torch.cuda.current_stream(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    # Warm-up directly before the timed region (no host work in between).
    for i in range(max(args.warmup, 3)):
        bound[i % nsets]()
    barrier()
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for i in range(args.steps):
        bound[i % nsets]()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    ms_total = e0.elapsed_time(e1)
    clk = clocks.stop()
    ms_step_local = ms_total / args.steps
    ms_step = aggregate_max(ms_step_local, world)
    rows_all = aggregate_sum(float(rows_per_step), world)
    value = rows_all / (ms_step / 1e3)

    # Algorithmic bytes of each input set (they depend on where requests
    # reject; the outputs of the timed calls are those of the warm-up).
    per_set_bytes = [step_bytes(c, b.out_num_accepted, w.V) for c, b in zip(cases, bound)]
    mean_bytes = sum(per_set_bytes[i % nsets] for i in range(args.steps)) / args.steps
    acc = torch.cat([b.out_num_accepted for b in bound]).float()
    alpha_hat = float(acc.mean()) / w.gamma

    # End to end through the public API from pinned host buffers: each step
    # copies its inputs to the device and reads its outputs back.
    host = []
    for c in cases[:2]:
        host.append({k: (None if v is None else v.cpu().pin_memory()) for k, v in c.items()})
    del bound, cases
    torch.cuda.empty_cache()
    h2d = sum(t.numel() * t.element_size() for t in host[0].values() if t is not None)
    d2h = w.B * (w.gamma + 1) * 4 + w.B * 4
    for i in range(2):
        hc = host[i % len(host)]
        verify_host(hc["logits"], hc["draft_ids"], hc["draft_probs"], hc["u_accept"],
                    hc["u_sample"], hc["temperature"], hc["draft_lens"], device=dev)
    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(args.e2e_steps):
        hc = host[i % len(host)]
        verify_host(hc["logits"], hc["draft_ids"], hc["draft_probs"], hc["u_accept"],
                    hc["u_sample"], hc["temperature"], hc["draft_lens"], device=dev)
    e2e_s = (time.perf_counter() - t0) / args.e2e_steps
    e2e_s = aggregate_max(e2e_s, world)
    e2e_value = rows_all / e2e_s

    peak, peak_src = measured_peaks()
    achieved = mean_bytes / (ms_step_local / 1e3) / 1e9
    traffic = recorded_traffic(args.workload)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (seeded; shapes and value recipe of the workload)",
        "config": {"workload": w.name, "B_per_gpu": w.B, "gamma": w.gamma, "V": w.V,
                   "temperature": list(w.temperatures), "draft_probs": "fp32",
                   "l2": f"inputs larger than L2: {nsets} rotating input sets of "
                         f"{set_bytes / 1e6:.0f} MB",
                   "alpha_hat": alpha_hat, "parallelism": f"replicas x{world} (requests sharded)"},
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"],
                   "reasons": clk["reasons"], "samples": clk["samples"]},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3,
                "h2d_gbs": h2d / e2e_s / 1e9,
                "path": "verify_host: pinned host tensors copied to the device, one call, "
                        "outputs copied back, every step"},
        "gpu_launches": KERNELS_PER_STEP * args.steps,
        "roofline": {"bound": "hbm", "kernel": "spec_verify step (persistent sv_verify_kernel)",
                     "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                     "algorithmic_bytes_per_step": mean_bytes,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s"},
    }
    if rank == 0 and world == 1 and not args.no_sweep:
        line["sweep"] = sweep(api, W, dev, args, peak)
    if rank == 0 and world == 1:
        line["cpu_baseline"] = cpu_baseline(host[0], args.cpu_seconds)
    return line


# The five workloads, c4's gamma 3..8 (B = 64, V = 128256), and c3's shape
# (gamma = 5, peaky rows) along the other two axes: V = 32000 and 128256 at
# B = 128, B = 32 and 256 at V = 151936.
SWEEP = [("c1", {}), ("c2", {}), ("c3", {}), ("c4", {}), ("c5", {})] + \
    [(f"c4_gamma{g}", {"gamma": g}) for g in range(3, 9)] + \
    [("c3_V32000", {"V": 32000}), ("c3_V128256", {"V": 128256}),
     ("c3_B32", {"B": 32}), ("c3_B256", {"B": 256})]


def sweep(api, W, dev, args, peak):
    """The B x gamma x V sweep: every workload (and c4's gamma 3..8 on the
    same seed), each timed on its own inputs.  Throughput in verified draft
    rows/s and algorithmic GB/s with its fraction of the measured HBM rate;
    c1 moves ~1 MB, so its figure of merit is the latency of one call."""
    import torch
    flush = torch.empty(256 * 2 ** 20 // 4, dtype=torch.float32, device=dev)
    out = {}
    for key, over in SWEEP:
        w = W.workload(key.split("_")[0], **over)
        r = time_workload(api, W, w, dev, args.sweep_steps, 3, flush)
        gbs = r["bytes_per_step"] / (r["us_per_step"] * 1e-6) / 1e9
        label = ", ".join(f"{k}={v}" for k, v in over.items())
        out[key] = {"workload": w.name if not over else f"{w.name} ({label})",
                    "B": w.B, "gamma": w.gamma, "V": w.V, "dtype": w.dtype,
                    "us_per_step": r["us_per_step"], "rows_per_s": r["rows_per_s"],
                    "gbs": gbs, "frac": gbs / peak, "alpha_hat": r["alpha_hat"],
                    "timing": r["timing"]}
        if key == "c1":
            out[key]["figure_of_merit"] = "latency (us per call)"
        torch.cuda.empty_cache()
    return out


def cpu_baseline(host, seconds: float):
    """The fp64 oracle, as it stands, on the host cores: whole batches of the
    workload repeated until ``seconds`` of wall time have passed, once on one
    thread and once split by request over every core this process may use."""
    import oracle
    rows = host["draft_ids"].shape[0] * host["draft_ids"].shape[1] \
        if host["draft_lens"] is None else int(host["draft_lens"].sum())
    args = (host["logits"], host["draft_ids"], host["draft_probs"], host["u_accept"],
            host["u_sample"], host["temperature"], host["draft_lens"])

    def timed(nthreads, budget):
        n, t0 = 0, time.perf_counter()
        while True:
            oracle.verify(*args, nthreads=nthreads)
            n += 1
            el = time.perf_counter() - t0
            if el >= budget:
                return n, el

    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    n1, el1 = timed(1, seconds / 2)
    nn, eln = timed(cores, seconds / 2)
    B = host["draft_ids"].shape[0]
    return {"value": nn * rows / eln, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{nn} full batch(es) of {B} requests, fp64 C oracle split by request "
                      f"over {cores} threads, {eln:.1f} s",
            "single_thread": {"value": n1 * rows / el1, "unit": UNIT, "cores": 1,
                              "sample": f"{n1} full batch(es) of {B} requests, one thread, "
                                        f"{el1:.1f} s"}}


# ---------------------------------------------------------- reference arm ----

def run_reference(args, rank, world):
    """The oracle timed on the host cores: each step is one request of the
    workload (a bounded sample), so the whole run ends within minutes."""
    import torch

    import oracle
    from speculative_decoding_verification_75_gb300 import workloads as W
    w = W.workload(args.workload)
    small = w.with_(B=min(w.B, 8))
    case = W.make_case(small, device="cpu", seed=rank_seed(w.seed, 0, 0))
    reqs = []
    for b in range(small.B):
        reqs.append({k: (None if v is None else v[b:b + 1].contiguous()) for k, v in case.items()})

    def step(i):
        r = reqs[i % len(reqs)]
        oracle.verify(r["logits"], r["draft_ids"], r["draft_probs"], r["u_accept"],
                      r["u_sample"], r["temperature"], r["draft_lens"])

    for i in range(max(args.warmup, 3)):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    el = time.perf_counter() - t0
    rows = sum(W.verified_rows(reqs[i % len(reqs)]) for i in range(args.steps))
    value = rows / el
    h2d = sum(t.numel() * t.element_size() for t in reqs[0].values() if t is not None)
    del torch
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; same workload recipe)",
        "config": {"workload": w.name, "B_per_step": 1, "gamma": w.gamma, "V": w.V,
                   "reference": "fp64 C oracle written from the pages (no reference code "
                                "exists: the pages are prose)"},
        "cpu_baseline": {"kind": "oracle", "cores": 1, "value": value, "unit": UNIT,
                         "sample": f"one request of {w.name} per step, {args.steps} steps"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "input_bytes_per_step": h2d,
    }


# -------------------------------------------------------------------- main ----

def main(argv=None):
    args = parse_args(argv)
    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return 0
            world_ref = world
        else:
            import torch
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
    if args.impl == "reference":
        line = run_reference(args, rank, world if world > 1 else 1)
    else:
        line = run_ours(args, rank, local_rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl != "reference":
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
