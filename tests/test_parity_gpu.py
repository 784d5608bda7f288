"""CUDA path against the fp64 oracle, element by element (needs a GPU).

Covers the five benchmark workloads at full size (every request compared,
not a sample), small multi-chunk cases with ragged vocabulary tails in both
the TMA and the plain-load kernels, and the edge cases of the method:
draft length 0, greedy and mixed temperatures, deterministic drafts, masked
(-inf) logits, an empty residual, invalid inputs, large gamma, misaligned
pointers, repeated calls and a non-default stream.
"""
import numpy as np
import pytest
import torch

from parity import compare, run_gpu, run_oracle, to_np
from speculative_decoding_verification_75_gb300 import api, verify, workloads
from speculative_decoding_verification_75_gb300.workloads import Workload, make_case

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def check(case, **kw):
    gpu = run_gpu(case)
    ora = run_oracle(case)
    return compare(case, gpu, ora, **kw), gpu, ora


@pytest.mark.parametrize("key", ["c1", "c2", "c3", "c4", "c5"])
def test_workload_full_size(key):
    """Every request of the workload: exact, or (draw near a CDF edge) exact
    up to the draw and the draw within its bracket.  An accept decision
    within 1e-5 of its uniform has probability ~2e-5 per decision, so at most
    one such request is tolerated per workload; the counts are reported."""
    w = workloads.workload(key)
    case = make_case(w, device=DEV)
    rep, gpu, ora = check(case, label=w.name)
    assert rep["borderline"] <= 1, rep
    assert rep["exact"] + rep["draw_border"] + rep["borderline"] + rep["bad"] == w.B


@pytest.mark.parametrize("gamma", [3, 4, 5, 6, 7, 8])
def test_gamma_sweep_c4_shape(gamma):
    w = workloads.workload("c4", B=16, gamma=gamma)
    rep, _, _ = check(make_case(w, device=DEV), label=f"c4 shape, B=16, gamma={gamma}")
    assert rep["borderline"] <= 1 and rep["bad"] == 0


SMALL_V = [1, 2, 7, 33, 1000, 1024, 4095, 4096, 4097, 8192, 8200, 20001, 20008]


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("V", SMALL_V)
@pytest.mark.parametrize("with_q", [True, False])
def test_small_vocab_tails(dtype, V, with_q):
    w = Workload("tails", 7, 3, V, dtype, 2.0, (0.3, 1.5), (0.0, 0.7, 1.0),
                 gamma_range=(0, 3), seed=V)
    rep, _, _ = check(make_case(w, device=DEV, draft_probs=with_q))
    assert rep["bad"] == 0


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_misaligned_pointers_use_plain_loads(dtype):
    w = Workload("mis", 5, 4, 4096, dtype, 2.0, (0.5, 0.5), (0.8,), seed=3)
    case = make_case(w, device=DEV)
    lg = case["logits"]
    big = torch.empty(lg.numel() + 8, dtype=lg.dtype, device=DEV)
    view = big[1:1 + lg.numel()].view(lg.shape)
    view.copy_(lg)
    q = case["draft_probs"]
    bigq = torch.empty(q.numel() + 8, dtype=q.dtype, device=DEV)
    qv = bigq[1:1 + q.numel()].view(q.shape)
    qv.copy_(q)
    case2 = dict(case, logits=view, draft_probs=qv)
    r1 = run_gpu(case)
    r2 = run_gpu(case2)
    compare(case2, r2, run_oracle(case2))
    assert np.array_equal(r1["tokens"], r2["tokens"])


def test_zero_drafts_is_plain_sampling():
    w = Workload("g0", 64, 0, 5000, "bf16", 2.0, (1.0, 1.0), (0.0, 1.0), seed=5)
    rep, gpu, _ = check(make_case(w, device=DEV))
    assert (gpu["num_accepted"] == 0).all() and (gpu["tokens"][:, 0] >= 0).all()


def test_large_gamma_multi_round_merge():
    w = Workload("g40", 6, 40, 3000, "fp32", 0.3, (0.01, 0.02), (0.7, 1.0), seed=9)
    case = make_case(w, device=DEV)
    case["u_accept"].mul_(0.2)            # long accepted runs cross the 32-lane rounds
    rep, gpu, _ = check(case)
    assert gpu["num_accepted"].max() > 32


def test_all_accepted_takes_bonus_row():
    w = Workload("bonus", 32, 4, 9000, "bf16", 2.0, (0.5, 0.5), (1.0,), seed=11)
    case = make_case(w, device=DEV)
    case["u_accept"].zero_()
    q = torch.softmax(case["logits"][:, :4].float(), dim=-1)   # q = p: a = 1
    case["draft_probs"] = q.contiguous()
    rep, gpu, _ = check(case)
    assert (gpu["num_accepted"] == 4).all()


# A batch of one request runs the kernel variant whose counter warp runs the
# merge and the search itself; these cover its paths.
@pytest.mark.parametrize("name,T,g,dtype,V,with_q", [
    ("greedy", 0.0, 4, "bf16", 9000, True),
    ("sampled_fp32", 1.0, 3, "fp32", 5000, True),
    ("deterministic", 0.8, 5, "bf16", 12000, False),
    ("gamma0", 1.0, 0, "bf16", 4000, True),
    ("plain_load", 0.7, 3, "fp32", 4097, True),   # V * 4 not a multiple of 16
])
def test_single_request(name, T, g, dtype, V, with_q):
    w = Workload("one_" + name, 1, g, V, dtype, 2.0, (0.5, 0.5), (T,), seed=21)
    for seed in range(4):
        case = make_case(w, device=DEV, seed=100 + seed, draft_probs=with_q)
        check(case)


def test_single_request_bonus_and_invalid():
    w = Workload("one_bonus", 1, 4, 9000, "bf16", 2.0, (0.5, 0.5), (1.0,), seed=22)
    case = make_case(w, device=DEV)
    case["u_accept"].zero_()
    case["draft_probs"] = torch.softmax(case["logits"][:, :4].float(), dim=-1).contiguous()
    rep, gpu, _ = check(case)
    assert int(gpu["num_accepted"][0]) == 4
    case = make_case(w, device=DEV)
    case["u_sample"][0] = float("nan")   # the merge marks it bad; no residual, no search
    gpu = run_gpu(case)
    ora = run_oracle(case)
    compare(case, gpu, ora)
    assert int(gpu["num_accepted"][0]) == -1


def test_empty_residual_draws_from_p():
    w = Workload("empty", 8, 2, 3000, "fp32", 1.5, (0.5, 0.5), (1.0,), seed=12)
    case = make_case(w, device=DEV)
    p = torch.softmax(case["logits"][:, :2].float(), dim=-1)
    case["draft_probs"] = (2.0 * p).contiguous()            # q = 2p: a = 0.5, (p-q)+ = 0
    case["u_accept"].fill_(0.75)                            # every request rejects at 0
    gpu = run_gpu(case)
    ora = run_oracle(case)
    assert (ora["sample_fallback"] == 1).all()
    assert (gpu["resid_mass"] == 0).all()
    compare(case, gpu, ora)


def test_masked_logits():
    V = 20000
    w = Workload("mask", 16, 3, V, "bf16", 2.0, (0.5, 0.5), (0.7, 1.0), seed=13)
    case = make_case(w, device=DEV)
    lg = case["logits"].float()
    lg[:, :, 8192:16384] = float("-inf")                    # a whole bf16 chunk
    lg[:, :, 2:40:3] = float("-inf")
    case["logits"] = lg.to(torch.bfloat16)
    q = torch.softmax(case["logits"][:, :3].float() + 0.3, dim=-1)
    case["draft_probs"] = q.contiguous()
    gen = torch.Generator(device=DEV).manual_seed(13)
    case["draft_ids"] = torch.multinomial(q.view(-1, V), 1, generator=gen).view(16, 3).to(torch.int32)
    check(case)


def test_invalid_inputs_are_isolated():
    B, g, V = 8, 2, 300
    w = Workload("bad", B, g, V, "fp32", 1.0, (0.5, 0.5), (1.0,), seed=14)
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
    assert rc == api.SV_ERR_BAD_INPUT_DATA
    assert word == 1 | 2 | 4 | 8 | 16 | 32


@pytest.mark.parametrize("V,dt", [(300000, "bf16"), (300001, "fp32")])
@pytest.mark.parametrize("small_path", [True, False], ids=["cluster", "persistent"])
def test_very_large_vocabulary(V, dt, small_path):
    """Rows longer than one batch of chunk statistics (more than 16 chunks
    per row: the merge folds two batches) and than 256 segments of 1024 (the
    search walks chunk sums, then the chunk's segment sums, then the
    segment), aligned (TMA) and odd (plain loads), with sample uniforms at 0
    and just below 1 as well as random ones."""
    B, g = 4, 3
    w = Workload(f"large V={V} {dt}", B, g, V, dt, 2.0, (0.5, 1.5), (0.8, 1.0), seed=45)
    case = make_case(w, device=DEV)
    top = float(np.nextafter(np.float32(1.0), np.float32(0.0)))
    case["u_sample"][0] = 0.0
    case["u_sample"][1] = top
    prev = api.set_small_batch_path(small_path)
    try:
        gpu = run_gpu(case)
    finally:
        api.set_small_batch_path(prev)
    rep = compare(case, gpu, run_oracle(case))
    assert rep["bad"] == 0 and rep["borderline"] <= 1


@pytest.mark.parametrize("V", [4096, 40000])
@pytest.mark.parametrize("small_path", [True, False], ids=["cluster", "persistent"])
def test_tiny_temperature_is_invalid_data(V, small_path):
    """A temperature so small that the row maximum in log2 units reaches 2^24
    (in binary32) marks the request bad (SV_BAD_NORMALISER), as the oracle
    does.  The same T with a row maximum of 0 is a valid one-hot request even
    though the other elements' exponents (and, over several chunks or
    slices, their own partial sums) leave the binary32 range; a product just
    below 2^24 is valid too."""
    B, g = 6, 2
    w = Workload("tinyT", B, g, V, "fp32", 1.0, (0.5, 0.5), (1.0,), seed=17)
    case = make_case(w, device=DEV)
    lg = case["logits"]
    lg[0, :, :] = torch.linspace(-3.0, 100.0, V, device=DEV)   # 100 * log2e / 1e-37 overflows
    lg[1, :, :] = torch.linspace(-3.0, 0.0, V, device=DEV)     # maximum 0: offset 0
    lg[2, :, :] = torch.linspace(-3.0, 1.0, V, device=DEV)     # 1.44e7 < 2^24
    lg[3, :, :] = torch.linspace(-3.0, 1.0, V, device=DEV)     # 1.80e7 >= 2^24
    case["temperature"][0:4] = torch.tensor([1e-37, 1e-37, 1e-7, 8e-8], device=DEV)
    prev = api.set_small_batch_path(small_path)
    try:
        gpu = run_gpu(case)
    finally:
        api.set_small_batch_path(prev)
    ora = run_oracle(case)
    compare(case, gpu, ora)
    assert ora["bad"].tolist() == [32, 0, 0, 32, 0, 0]


def test_no_request_with_rows_ends_cleanly():
    """Every draft length out of range: nothing is streamed or merged; the
    call still ends without a timeout and marks every request."""
    B, g, V = 6, 3, 5000
    w = Workload("allbad", B, g, V, "bf16", 1.0, (0.5, 1.0), (0.0, 1.0), seed=15)
    case = make_case(w, device=DEV)
    case["draft_lens"] = torch.tensor([-1, g + 1, g + 5, -3, g + 1, -1], dtype=torch.int32,
                                      device=DEV)
    gpu = run_gpu(case)
    ora = run_oracle(case)
    compare(case, gpu, ora)
    assert (gpu["num_accepted"] == -1).all()
    rc, word = api.last_error(api.get_workspace(B, g, V, DEV))
    assert rc == api.SV_ERR_BAD_INPUT_DATA and word == 1


def test_all_greedy_batch_has_no_residual_work():
    """T = 0 everywhere: requests merge but publish nothing to re-sample."""
    w = Workload("greedy", 24, 4, 70000, "bf16", 2.0, (0.5, 1.0), (0.0,), seed=16)
    rep, gpu, ora = check(make_case(w, device=DEV))
    assert rep["bad"] == 0
    rc, word = api.last_error(api.get_workspace(24, 4, 70000, DEV))
    assert (rc, word) == (api.SV_OK, 0)


def test_bounded_waits_give_up_and_leave_the_context_usable():
    """Failure detection without a GPU fault: an mbarrier phase nobody
    completes and a flag nobody sets, each waited for with a 2 ms limit,
    must time out with SV_FAULT_TIMEOUT; the next call then runs normally."""
    import time
    t0 = time.perf_counter()
    word = api.selftest_wait_timeout(2000)
    assert time.perf_counter() - t0 >= 0.004  # both waits ran to their limit
    assert word == api.SV_FAULT_TIMEOUT | 0x1 | 0x2, hex(word)
    case = make_case(workloads.workload("c1"), device=DEV)
    rep, _, _ = check(case)
    assert rep["exact"] + rep["draw_border"] + rep["borderline"] == 1


def test_clean_call_reports_ok():
    case = make_case(workloads.workload("c1"), device=DEV)
    run_gpu(case)
    rc, word = api.last_error(api.get_workspace(1, 5, 32000, DEV))
    assert (rc, word) == (api.SV_OK, 0)


def test_deterministic_and_stream():
    case = make_case(workloads.workload("c2"), device=DEV)
    a = run_gpu(case)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = run_gpu(case)
    for k in a:
        assert np.array_equal(a[k], b[k], equal_nan=True), k


def test_two_streams_run_concurrently_with_their_own_workspaces():
    """verify() on two streams at once: each stream gets its own cached
    workspace, so the calls may overlap on the GPU; both match the oracle."""
    cases = [make_case(workloads.workload("c2"), device=DEV, seed=s) for s in (31, 32)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    outs = []
    for _ in range(3):  # several rounds so the two streams' calls overlap
        outs = []
        for c, s in zip(cases, streams):
            with torch.cuda.stream(s):
                outs.append(verify(c["logits"], c["draft_ids"], c["draft_probs"],
                                   c["u_accept"], c["u_sample"], c["temperature"],
                                   c["draft_lens"], diag=True, stream=s))
    torch.cuda.synchronize()
    ws = [api.get_workspace(8, 5, 151936, DEV, s) for s in streams]
    assert ws[0].data_ptr() != ws[1].data_ptr()
    for c, (tok, nacc, d) in zip(cases, outs):
        gpu = {"tokens": to_np(tok), "num_accepted": to_np(nacc)}
        gpu.update({k: to_np(v) for k, v in d.items()})
        compare(c, gpu, run_oracle(c))


def test_bound_call_matches_verify():
    """bind(): the arguments are marshalled once; repeated calls give
    verify()'s results and follow the tensors' current contents."""
    c = make_case(workloads.workload("c2"), device=DEV, seed=33)
    args = (c["logits"], c["draft_ids"], c["draft_probs"], c["u_accept"], c["u_sample"],
            c["temperature"], c["draft_lens"])
    ref_tok, ref_nacc = verify(*args)
    bound = api.bind(*args)
    for _ in range(3):
        tok, nacc = bound()
    torch.cuda.synchronize()
    assert torch.equal(tok, ref_tok) and torch.equal(nacc, ref_nacc)
    c["u_sample"].copy_(torch.rand_like(c["u_sample"]))   # new contents, same storage
    tok, nacc = bound()
    ref_tok, ref_nacc = verify(*args)
    torch.cuda.synchronize()
    assert torch.equal(tok, ref_tok) and torch.equal(nacc, ref_nacc)


def test_batch_zero_is_noop():
    lg = torch.empty(0, 3, 10, device=DEV)
    e2 = torch.empty(0, 2, device=DEV)
    tok, nacc = verify(lg, torch.empty(0, 2, dtype=torch.int32, device=DEV), None,
                       e2, torch.empty(0, device=DEV), torch.empty(0, device=DEV))
    assert tok.shape == (0, 3) and nacc.shape == (0,)


def test_gpu_output_is_distributed_as_p():
    """P3 §3.2 on the GPU itself: x ~ q, accept/resample -> emitted ~ p."""
    from scipy import stats
    n, V = 200_000, 6
    gen = torch.Generator(device=DEV).manual_seed(21)
    p0 = torch.tensor([0.30, 0.05, 0.20, 0.25, 0.15, 0.05], device=DEV)
    q0 = torch.tensor([0.10, 0.30, 0.25, 0.05, 0.10, 0.20], device=DEV)
    logits = torch.log(p0).expand(n, 2, V).contiguous()
    q = q0.expand(n, 1, V).contiguous()
    ids = torch.multinomial(q0, n, replacement=True, generator=gen).view(n, 1).to(torch.int32)
    u = torch.rand(n, 1, generator=gen, device=DEV)
    us = torch.rand(n, generator=gen, device=DEV)
    tok, _ = verify(logits, ids, q, u, us, torch.ones(n, device=DEV))
    counts = torch.bincount(tok[:, 0].long(), minlength=V).cpu().numpy()
    pex = torch.softmax(torch.log(p0).double(), 0).cpu().numpy()
    stat = ((counts - n * pex) ** 2 / (n * pex)).sum()
    assert stats.chi2.sf(stat, V - 1) > 1e-4
