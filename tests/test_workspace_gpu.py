"""The workspace protocol on the GPU: one launch per call, counter sets that
alternate by call, epoch-tagged flags, and the certificate that makes a call
clear a workspace it did not leave ready (fresh or foreign bytes, another
layout, a batch too large for the shared tables).  Every case is compared
with the fp64 oracle, or with an oracle-checked run of the same inputs."""
import numpy as np
import pytest
import torch

from parity import compare, run_gpu, run_oracle, to_np
from speculative_decoding_verification_75_gb300 import api, verify, workloads
from speculative_decoding_verification_75_gb300.workloads import Workload, make_case

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def plain(case, **kw):
    """The call without diagnostics: no histogram, so (for B <= 256) one
    launch and no set-up kernel."""
    tok, nacc = verify(case["logits"], case["draft_ids"], case["draft_probs"], case["u_accept"],
                       case["u_sample"], case["temperature"], case["draft_lens"], **kw)
    torch.cuda.synchronize()
    return to_np(tok), to_np(nacc)


@pytest.mark.parametrize("key", ["c1", "c2", "c3", "c4", "c5"])
def test_single_launch_path_matches_checked_path(key):
    """The plain call gives exactly the outputs of the diagnostic call, which
    the parity tests check against the oracle."""
    case = make_case(workloads.workload(key), device=DEV)
    ref = run_gpu(case)
    for _ in range(3):  # consecutive calls alternate the counter sets
        tok, nacc = plain(case)
        assert np.array_equal(tok, ref["tokens"]) and np.array_equal(nacc, ref["num_accepted"])


@pytest.mark.parametrize("fill", [0x00, 0xA5, 0xFF])
def test_workspace_with_arbitrary_bytes(fill):
    """A workspace holding any bytes is cleared by the call that first uses
    it; results match the oracle, with and without diagnostics."""
    w = Workload("junk", 12, 4, 9000, "bf16", 2.0, (0.3, 1.5), (0.0, 0.8, 1.0),
                 gamma_range=(0, 4), seed=21)
    case = make_case(w, device=DEV)
    ora = run_oracle(case)
    nb = api.workspace_bytes(w.B, w.gamma, w.V)
    ws = torch.full((nb,), fill, dtype=torch.uint8, device=DEV)
    gpu = run_gpu(case, workspace=ws)
    compare(case, gpu, ora)
    ws.fill_(fill)
    tok, nacc = plain(case, workspace=ws)
    assert np.array_equal(tok, gpu["tokens"]) and np.array_equal(nacc, gpu["num_accepted"])


def test_layout_changes_on_one_workspace():
    """One buffer serves batches of different shapes in turn (each layout
    places the counters elsewhere); every call still matches the oracle."""
    shapes = [(16, 5, 12000, "bf16"), (3, 2, 700, "fp32"), (40, 8, 5000, "bf16"),
              (1, 5, 32000, "fp32")]
    cases = []
    for i, (B, g, V, dt) in enumerate(shapes):
        w = Workload(f"shape{i}", B, g, V, dt, 2.0, (0.3, 1.5), (0.0, 0.8, 1.0), seed=30 + i)
        case = make_case(w, device=DEV)
        cases.append((w, case, run_oracle(case)))
    nb = max(api.workspace_bytes(w.B, w.gamma, w.V) for w, _, _ in cases)
    ws = torch.zeros(nb, dtype=torch.uint8, device=DEV)
    for order in (range(4), reversed(range(4)), [0, 0, 2, 2, 1, 3, 1]):
        for i in order:
            w, case, ora = cases[i]
            tok, nacc = plain(case, workspace=ws)
            gpu = run_gpu(case, workspace=ws)
            compare(case, gpu, ora)
            assert np.array_equal(tok, gpu["tokens"]) and np.array_equal(nacc, gpu["num_accepted"])


def test_error_word_follows_each_call():
    """The error word read after a call is that call's: a bad call reports its
    bits, the clean call after it reports none, in both counter sets."""
    B, g, V = 4, 2, 600
    w = Workload("errs", B, g, V, "fp32", 1.0, (0.5, 0.5), (1.0,), seed=22)
    good = make_case(w, device=DEV)
    bad = {k: (v.clone() if v is not None else None) for k, v in good.items()}
    bad["draft_ids"][1, 0] = V
    ws = torch.empty(api.workspace_bytes(B, g, V), dtype=torch.uint8, device=DEV)
    for _ in range(3):
        plain(bad, workspace=ws)
        assert api.last_error(ws) == (api.SV_ERR_BAD_INPUT_DATA, 4)
        plain(good, workspace=ws)
        assert api.last_error(ws) == (api.SV_OK, 0)


@pytest.mark.parametrize("B", [257, 2100])
def test_batch_beyond_shared_tables(B):
    """More requests than the kernel keeps in shared memory (256): the set-up
    kernel writes the tables to global memory; ragged drafts, mixed
    temperatures and a few invalid lengths, against the oracle."""
    g, V = 3, 700
    w = Workload("wide", B, g, V, "fp32", 2.0, (0.3, 1.5), (0.0, 0.8, 1.0),
                 gamma_range=(0, 3), seed=23)
    case = make_case(w, device=DEV)
    case["draft_lens"][5] = g + 1
    case["draft_lens"][B - 1] = -1
    ora = run_oracle(case)
    gpu = run_gpu(case)
    rep = compare(case, gpu, ora, label=f"B={B} (tables in global memory)")
    assert rep["bad"] == 2 and rep["borderline"] <= 1
    tok, nacc = plain(case)
    assert np.array_equal(tok, gpu["tokens"]) and np.array_equal(nacc, gpu["num_accepted"])
