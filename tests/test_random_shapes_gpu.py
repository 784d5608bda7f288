"""Seeded random batches -- shapes, dtypes, draft lengths, temperatures,
noise levels, peaky rows, deterministic drafts -- on both kernels, each
against the fp64 oracle (needs a GPU).

Every case runs with the small-batch cluster path enabled (batches that
qualify take it) and with every batch sent to the persistent kernel; odd
vocabulary sizes exercise the plain-load variant.  Larger batches (64 to
300 requests: bigger row blocks, and beyond 256 the tables in global
memory) run on the persistent kernel.  The shapes are drawn from a fixed
seed, so a failure names a reproducible case.
"""
import numpy as np
import pytest
import torch

from parity import compare, run_gpu, run_oracle
from speculative_decoding_verification_75_gb300 import api
from speculative_decoding_verification_75_gb300.workloads import Workload, make_case

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
N_CASES = 24


def random_workload(i):
    rng = np.random.default_rng(1000 + i)
    B = int(rng.choice([1, 2, 3, 5, 8, 13, 24, 40]))
    g = int(rng.integers(0, 11))
    V = int(rng.choice([int(rng.integers(1, 64)), int(rng.integers(64, 4096)),
                        int(rng.integers(4096, 70000)), 32000, 50000]))
    if rng.random() < 0.5:
        V = (V + 7) // 8 * 8  # aligned rows: the TMA variants
    dt = "bf16" if rng.random() < 0.6 else "fp32"
    temps = tuple(float(x) for x in rng.choice([0.0, 0.5, 0.8, 1.0, 1.5], size=int(rng.integers(1, 4))))
    lo = float(rng.uniform(0.0, 1.0))
    noise = (lo, lo + float(rng.uniform(0.0, 1.5)))
    ragged = (0, g) if (g > 0 and rng.random() < 0.5) else None
    peaky = rng.random() < 0.3
    w = Workload(f"random#{i} B={B} g={g} V={V} {dt}", B, g, V, dt, float(rng.uniform(1.0, 3.0)),
                 noise, temps, gamma_range=ragged, boost_frac=0.01 if peaky else 0.0,
                 boost=8.0 if peaky else 0.0, seed=2000 + i)
    return w, bool(rng.random() < 0.75)


@pytest.mark.parametrize("small_path", [True, False], ids=["cluster-on", "cluster-off"])
@pytest.mark.parametrize("i", range(N_CASES))
def test_random_batch(i, small_path):
    w, with_q = random_workload(i)
    case = make_case(w, device=DEV, draft_probs=with_q)
    prev = api.set_small_batch_path(small_path)
    try:
        gpu = run_gpu(case)
    finally:
        api.set_small_batch_path(prev)
    rep = compare(case, gpu, run_oracle(case))
    assert rep["borderline"] <= 1, rep
    assert rep["exact"] + rep["draw_border"] + rep["borderline"] + rep["bad"] == w.B


N_LARGE = 8


def random_large_workload(i):
    rng = np.random.default_rng(3000 + i)
    B = int(rng.choice([64, 100, 200, 257, 300]))
    g = int(rng.integers(1, 12))
    V = int(rng.integers(64, 150000 if B <= 64 else (40000 if B <= 200 else 12000)))
    if rng.random() < 0.6:
        V = (V + 7) // 8 * 8
    dt = "bf16" if rng.random() < 0.6 else "fp32"
    temps = tuple(float(x) for x in rng.choice([0.0, 0.5, 0.8, 1.0, 1.5], size=int(rng.integers(1, 4))))
    lo = float(rng.uniform(0.0, 1.0))
    ragged = (0, g) if rng.random() < 0.5 else None
    w = Workload(f"random large#{i} B={B} g={g} V={V} {dt}", B, g, V, dt, float(rng.uniform(1.0, 3.0)),
                 (lo, lo + float(rng.uniform(0.0, 1.5))), temps, gamma_range=ragged, seed=4000 + i)
    return w, bool(rng.random() < 0.75)


@pytest.mark.parametrize("i", range(N_LARGE))
def test_random_large_batch(i):
    w, with_q = random_large_workload(i)
    case = make_case(w, device=DEV, draft_probs=with_q)
    rep = compare(case, run_gpu(case), run_oracle(case))
    assert rep["borderline"] <= 1, rep
    assert rep["exact"] + rep["draw_border"] + rep["borderline"] + rep["bad"] == w.B
