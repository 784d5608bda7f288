"""The small-batch cluster path and the persistent kernel on the same small
batches, each against the fp64 oracle (needs a GPU).

Batches of up to 32 requests with gamma_max < 16 and 16-byte aligned rows
run one thread-block cluster per request unless the path is switched off
(api.set_small_batch_path); every case here runs both ways.  Shapes cover
slices that are empty (V smaller than the cluster), ragged vocabulary
tails, gamma up to 15, greedy / sampled / mixed temperatures, deterministic
drafts, an all-accepting draft (bonus draws) and invalid inputs.
"""
import numpy as np
import pytest
import torch

from parity import compare, run_gpu, run_oracle
from speculative_decoding_verification_75_gb300 import api, workloads
from speculative_decoding_verification_75_gb300.workloads import Workload, make_case

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(params=[True, False], ids=["cluster", "persistent"])
def path(request):
    prev = api.set_small_batch_path(request.param)
    yield "cluster" if request.param else "persistent"
    api.set_small_batch_path(prev)


@pytest.mark.parametrize("key", ["c1", "c2"])
def test_small_workloads(key, path):
    w = workloads.workload(key)
    case = make_case(w, device=DEV)
    rep = compare(case, run_gpu(case), run_oracle(case), label=f"{w.name} ({path})")
    assert rep["borderline"] <= 1
    assert rep["exact"] + rep["draw_border"] + rep["borderline"] + rep["bad"] == w.B


SHAPES = [
    # B, gamma, V, dtype, temperatures, draft lengths, with q
    (1, 5, 8, "fp32", (1.0,), None, True),                 # most slices empty
    (3, 2, 40, "bf16", (0.0, 1.0), (0, 2), True),
    (5, 15, 4096, "bf16", (0.7, 1.0), None, True),         # the longest draft
    (8, 4, 20000, "fp32", (0.0, 0.8, 1.0), (0, 4), False),  # deterministic drafts
    (16, 3, 32000, "bf16", (1.0,), (1, 3), True),
    (32, 2, 50000, "bf16", (0.0, 0.7), None, True),        # the largest batch of the path
    (2, 7, 151936, "bf16", (0.8,), None, True),
    (8, 8, 128256, "bf16", (0.0, 1.0), None, True),        # q_k's slice in other rows' slots
    (4, 1, 3000, "fp32", (1.0,), None, True),              # two rows: q needs an extra slot
    (6, 2, 5000, "bf16", (0.8,), None, True),              # three rows
    (5, 3, 6000, "bf16", (0.8, 1.0), None, True),          # four rows
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"B{s[0]}_g{s[1]}_V{s[2]}_{s[3]}")
def test_small_shapes(shape, path):
    B, g, V, dt, temps, lens, with_q = shape
    w = Workload(f"small B={B} g={g} V={V} {dt}", B, g, V, dt, 2.0, (0.3, 1.5), temps,
                 gamma_range=lens, seed=B * 131 + g)
    case = make_case(w, device=DEV, draft_probs=with_q)
    rep = compare(case, run_gpu(case), run_oracle(case))
    assert rep["bad"] == 0 and rep["borderline"] <= 1


def test_every_draft_accepted(path):
    """q = p exactly: every draft accepted, every token a bonus draw."""
    B, g, V = 6, 4, 3000
    w = Workload("bonus", B, g, V, "fp32", 2.0, (0.0, 0.0), (1.0,), seed=41)
    case = make_case(w, device=DEV)
    p = torch.softmax(case["logits"][:, :g, :].double(), dim=-1).float()
    case["draft_probs"] = p.contiguous()
    gen = torch.Generator(device=DEV).manual_seed(5)
    case["draft_ids"] = torch.multinomial(p.view(-1, V), 1, generator=gen).view(B, g).to(torch.int32)
    case["u_accept"] = torch.rand(B, g, device=DEV, generator=gen) * 0.999
    gpu = run_gpu(case)
    compare(case, gpu, run_oracle(case))
    assert (torch.as_tensor(gpu["num_accepted"]) == g).all()


def test_invalid_inputs(path):
    B, g, V = 8, 2, 304
    w = Workload("bad small", B, g, V, "fp32", 1.0, (0.5, 0.5), (1.0,), seed=42)
    case = make_case(w, device=DEV)
    case["draft_lens"] = torch.full((B,), g, dtype=torch.int32, device=DEV)
    case["draft_lens"][1] = g + 1
    case["temperature"][2] = -1.0
    case["draft_ids"][3, 1] = V
    case["u_accept"][4, 0] = 1.0
    case["u_sample"][5] = float("nan")
    case["logits"][6, 1, 7] = float("inf")
    case["temperature"][7] = 1e-40
    gpu = run_gpu(case)
    ora = run_oracle(case)
    compare(case, gpu, ora)
    assert ora["bad"].tolist() == [0, 1, 2, 4, 8, 16, 32, 2]
    rc, word = api.last_error(api.get_workspace(B, g, V, DEV))
    assert rc == api.SV_ERR_BAD_INPUT_DATA and word == 1 | 2 | 4 | 8 | 16 | 32


def test_greedy_ties_across_slices(path):
    """A greedy row whose maximum appears in several places -- inside one
    slice / chunk and across slices, chunks and clusters' ranks -- takes the
    lowest index, as the oracle does."""
    B, g, V = 4, 3, 40000
    w = Workload("ties", B, g, V, "bf16", 1.0, (0.5, 0.5), (0.0,), seed=43)
    case = make_case(w, device=DEV)
    lg = case["logits"]
    spots = [[39990, 17, 25000], [5, 6, 30001], [20000, 39999, 2500], [12345, 12346, 12347]]
    for b in range(B):
        for i in range(g + 1):
            for j, pos in enumerate(spots[(b + i) % B]):
                lg[b, i, pos] = 50.0  # far above every other logit
    gpu = run_gpu(case)
    ora = run_oracle(case)
    compare(case, gpu, ora)
    for b in range(B):
        k = int(gpu["num_accepted"][b])
        assert gpu["tokens"][b][k] == min(spots[(b + k) % B])


@pytest.mark.parametrize("V", [40000, 151936])
def test_sample_uniform_extremes(path, V):
    """u_sample at 0 (the first token with positive mass) and at the largest
    binary32 value below 1 (u * S at or within rounding of the total: the
    walk may end past every weight and take the last positive one), on
    residual draws and on bonus draws.  At V = 151936 each lane's run of a
    cluster slice is several vectors (the draw walks the one run that holds
    the target); at V = 40000 a run is one vector."""
    B, g = 8, 3
    w = Workload(f"u extremes V={V}", B, g, V, "bf16", 2.0, (0.5, 1.5), (0.8, 1.0), seed=44)
    case = make_case(w, device=DEV)
    top = float(np.nextafter(np.float32(1.0), np.float32(0.0)))
    case["u_sample"][:] = torch.tensor([0.0, top] * (B // 2), device=DEV)
    case["u_accept"][:2] = 0.0  # every draft accepted: bonus draws
    gpu = run_gpu(case)
    rep = compare(case, gpu, run_oracle(case))
    assert rep["bad"] == 0 and rep["borderline"] <= 1
    assert (torch.as_tensor(gpu["num_accepted"][:2]) == g).all()
