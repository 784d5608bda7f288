"""The oracle's test-support views of a draw (CPU), which the GPU parity
checks use for draws near a CDF edge: the weights and their prefix sums
agree exactly, no weight is negative, the rejected token of a deterministic
draft weighs exactly nothing ((p - 1)_+ = 0), and the bonus row's weights
are p itself (they sum to 1)."""
import numpy as np

import oracle
from speculative_decoding_verification_75_gb300.workloads import Workload, make_case


def test_draw_weights_and_prefix_sums_agree():
    B, g, V = 3, 4, 3000
    w = Workload("draw views", B, g, V, "fp32", 2.0, (0.5, 1.0), (0.8,), seed=7)
    o = oracle.default()
    for with_q in (True, False):
        case = make_case(w, draft_probs=with_q)
        ids = case["draft_ids"].numpy()
        for b in range(B):
            for k in range(g + 1):  # k = g: the bonus row
                view = (case["logits"], case["draft_ids"], case["draft_probs"],
                        case["temperature"], b, k, g)
                wts, cdf = o.draw_weights(*view), o.draw_cdf(*view)
                assert wts.shape == cdf.shape == (V,)
                assert (wts >= 0.0).all()
                assert np.array_equal(np.cumsum(wts), cdf)
                if k == g:
                    assert abs(wts.sum() - 1.0) < 1e-12
                elif not with_q:
                    assert wts[ids[b, k]] == 0.0


def test_greedy_request_has_no_draw():
    w = Workload("greedy view", 2, 2, 500, "fp32", 2.0, (0.5, 0.5), (0.0,), seed=8)
    case = make_case(w)
    view = (case["logits"], case["draft_ids"], case["draft_probs"], case["temperature"], 0, 0, 2)
    assert oracle.default().draw_weights(*view) is None
    assert oracle.default().draw_cdf(*view) is None
