"""Acceptance statistics emitted by the verification pass itself.

The tutorial page (P3 §6.2) has the serving layer log the acceptance rate;
§3.3 gives its expectation: with every draft position accepted with
probability alpha = sum_x min(p(x), q(x)) independently, num_accepted is a
truncated geometric variable and E[num_accepted + 1] = (1 - alpha^(g+1)) /
(1 - alpha).  ``sv_diag.accept_hist`` counts requests per num_accepted in
the same pass over the logits; these tests check it against that law on the
GPU over a draft-length sweep, and check the host-side summary.
"""
import math

import numpy as np
import pytest
import torch

from speculative_decoding_verification_75_gb300 import api


def test_acceptance_stats_summary():
    # g = 3; 10 requests with 0 accepted, 20 with 1, 30 with 2, 40 with 3; 5 bad.
    s = api.acceptance_stats([10, 20, 30, 40, 5])
    assert s["n_valid"] == 100 and s["n_bad"] == 5
    assert s["accepted_at"] == [90, 70, 40]
    assert s["reached"] == [100, 90, 70]
    assert s["rate"] == pytest.approx([0.9, 70 / 90, 40 / 70])
    assert s["mean_emitted"] == pytest.approx((10 * 1 + 20 * 2 + 30 * 3 + 40 * 4) / 100)
    with pytest.raises(ValueError):
        api.acceptance_stats([3])


@pytest.mark.gpu
@pytest.mark.parametrize("gamma", [3, 5, 8])
def test_gpu_acceptance_follows_truncated_geometric(gamma):
    dev = torch.device("cuda:0")
    n = 65536
    p0 = torch.tensor([0.5, 0.3, 0.1, 0.1], dtype=torch.float64)
    q0 = torch.tensor([0.3, 0.3, 0.3, 0.1], dtype=torch.float64)
    alpha = float(torch.minimum(p0, q0).sum())  # 0.8
    V = p0.numel()
    gen = torch.Generator(device=dev).manual_seed(31 + gamma)
    logits = torch.log(p0).float().to(dev).expand(n, gamma + 1, V).contiguous()
    q = q0.float().to(dev).expand(n, gamma, V).contiguous()
    ids = torch.multinomial(q0.float().to(dev), n * gamma, replacement=True,
                            generator=gen).view(n, gamma).to(torch.int32)
    u = torch.rand(n, gamma, generator=gen, device=dev)
    us = torch.rand(n, generator=gen, device=dev)
    T = torch.ones(n, device=dev)
    _, nacc, d = api.verify(logits, ids, q, u, us, T, diag=True)
    hist = d["accept_hist"].cpu().numpy().astype(np.int64)
    assert hist[gamma + 1] == 0 and hist[:gamma + 1].sum() == n
    assert np.array_equal(hist[:gamma + 1],
                          np.bincount(nacc.cpu().numpy(), minlength=gamma + 1))
    # The law of num_accepted: alpha^k (1 - alpha) for k < g, alpha^g at g.
    law = np.array([alpha ** k * (1 - alpha) for k in range(gamma)] + [alpha ** gamma])
    from scipy import stats
    chi2 = ((hist[:gamma + 1] - n * law) ** 2 / (n * law)).sum()
    assert stats.chi2.sf(chi2, gamma) > 1e-4, (hist, n * law)
    s = api.acceptance_stats(hist)
    E = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    var = sum((k + 1) ** 2 * w for k, w in enumerate(law)) - E ** 2
    assert abs(s["mean_emitted"] - E) < 5 * math.sqrt(var / n), (s["mean_emitted"], E)
    for i, r in enumerate(s["rate"]):
        assert abs(r - alpha) < 5 * math.sqrt(alpha * (1 - alpha) / s["reached"][i])
