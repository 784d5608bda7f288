"""GPU-versus-oracle comparison with the decision-margin rule.

Integer outputs (accept flags, num_accepted, emitted token ids, the set of
requests with invalid data) must match the fp64 oracle bit for bit, except
for decisions whose margin is below ``MARGIN``: |u - a| for an accept test,
and min(u*S - C_{j-1}, C_j - u*S) (unnormalised residual mass) for a draw.
Such requests are counted and reported (see ``compare``): a near-tie in an
accept decision leaves only a validity check, a near-tie in the draw alone
still pins num_accepted, the accepted drafts and the draw's CDF bracket.
Probabilities must agree within ``REL`` relative error (``ABS`` absolute
floor for values the GPU's flush-to-zero exp2 returns as 0).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from speculative_decoding_verification_75_gb300 import verify

MARGIN = 1e-5
REL = 1e-5
ABS = 1e-30
RESID_ATOL = 1e-5


def to_np(t):
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return t.detach().cpu().numpy()
    return np.asarray(t)


def run_gpu(case, **kw):
    tok, nacc, d = verify(case["logits"], case["draft_ids"], case["draft_probs"],
                          case["u_accept"], case["u_sample"], case["temperature"],
                          case["draft_lens"], diag=True, **kw)
    torch.cuda.synchronize()
    out = {"tokens": to_np(tok), "num_accepted": to_np(nacc)}
    out.update({k: to_np(v) for k, v in d.items()})
    return out


def run_oracle(case):
    return oracle.verify(case["logits"], case["draft_ids"], case["draft_probs"],
                         case["u_accept"], case["u_sample"], case["temperature"],
                         case["draft_lens"])


# Reports of every compare() in this session, printed in the terminal
# summary (tests/conftest.py) so that the borderline counts stay visible.
REPORTS = []


def compare(case, gpu, ora, *, allow_borderline=True, label=None):
    """Check GPU outputs against the oracle; return a small report dict.

    Requests are split three ways:
      exact        every decision clears its margin: num_accepted and every
                   token must equal the oracle's;
      draw_border  every accept decision clears its margin but the draw lies
                   within MARGIN of a CDF edge: num_accepted and the accepted
                   drafts must be exact, and the drawn token j must satisfy
                   C_{j-1} - MARGIN <= u*S <= C_j + MARGIN on the oracle's
                   fp64 CDF of the draw (so the draw is still pinned);
      borderline   an accept decision within MARGIN: only validity is checked
                   (a different decision changes everything after it).
    """
    B, g = ora["flags"].shape
    lens = to_np(case["draft_lens"])
    lens = np.full(B, g) if lens is None else lens
    T = to_np(case["temperature"]).astype(np.float64)
    bad = ora["bad"] != 0
    assert np.array_equal(gpu["num_accepted"] == -1, bad), "bad-input sets differ"
    assert (gpu["tokens"][bad] == -1).all()

    border = np.zeros(B, bool)
    draw_border = np.zeros(B, bool)
    for b in np.nonzero(~bad)[0]:
        gb, k = int(lens[b]), int(ora["num_accepted"][b])
        dec = ora["accept_margin"][b, :min(k + 1, gb)]
        if dec.size and dec.min() < MARGIN:
            border[b] = True
            continue
        if T[b] > 0:
            S = ora["resid_mass"][b]
            draw_border[b] = (ora["sample_margin"][b] < MARGIN
                              or (k < gb and 0.0 < S < MARGIN))
    exact = ~bad & ~border & ~draw_border
    mism = np.nonzero((exact | draw_border) & (gpu["num_accepted"] != ora["num_accepted"]))[0]
    assert mism.size == 0, f"num_accepted differs for requests {mism[:10]}"
    tok_bad = np.nonzero(exact & (gpu["tokens"] != ora["tokens"]).any(axis=1))[0]
    assert tok_bad.size == 0, (
        f"tokens differ for requests {tok_bad[:10]}: gpu {gpu['tokens'][tok_bad[:3]]} "
        f"oracle {ora['tokens'][tok_bad[:3]]}")
    if not allow_borderline:
        assert not border.any(), f"borderline requests {np.nonzero(border)[0]}"

    # Draw-borderline requests: exact up to the draw, the draw within its
    # CDF bracket on the oracle's fp64 weights.
    draw_matching = 0
    us = to_np(case["u_sample"]).astype(np.float64)
    for b in np.nonzero(draw_border)[0]:
        k, gb = int(ora["num_accepted"][b]), int(lens[b])
        assert np.array_equal(gpu["tokens"][b, :k], ora["tokens"][b, :k]), f"request {b}"
        assert (gpu["tokens"][b, k + 1:] == -1).all(), f"request {b}"
        j = int(gpu["tokens"][b, k])
        draw = (case["logits"], case["draft_ids"], case["draft_probs"], case["temperature"],
                b, k, gb)
        cdf = oracle.default().draw_cdf(*draw)
        assert 0 <= j < cdf.size, f"request {b}: token {j}"
        target = us[b] * cdf[-1]
        lo = cdf[j - 1] if j > 0 else 0.0
        # The token's own mass (a positive weight can lie below the
        # resolution of the prefix sums near the total).
        assert oracle.default().draw_weights(*draw)[j] > 0.0, f"request {b}: token {j} has no weight"
        assert lo - MARGIN <= target <= cdf[j] + MARGIN, (
            f"request {b}: token {j} bracket [{lo}, {cdf[j]}) vs u*S {target}")
        draw_matching += int(j == ora["tokens"][b, k])

    # Per-position diagnostics.
    pos = np.arange(g)[None, :] < lens[:, None]
    live = pos & ~bad[:, None]
    fl_ok = live & (ora["accept_margin"] >= MARGIN)
    assert np.array_equal(gpu["flags"][fl_ok], ora["flags"][fl_ok]), "accept flags differ"
    for name in ("p_tok", "accept_prob"):
        a, o = gpu[name][live].astype(np.float64), ora[name][live]
        err = np.abs(a - o) - (REL * np.abs(o) + ABS)
        assert (err <= 0).all(), f"{name}: worst excess {err.max():.3e}"
    assert np.array_equal(gpu["q_tok"][live].astype(np.float64), ora["q_tok"][live])

    rows = np.arange(g + 1)[None, :] <= lens[:, None]
    rlive = rows & ~bad[:, None]
    assert np.array_equal(gpu["row_max"][rlive].astype(np.float64), ora["row_max"][rlive])
    samp = T > 0
    rs = rlive & samp[:, None]
    a, o = gpu["row_sum"][rs].astype(np.float64), ora["row_sum"][rs]
    assert (np.abs(a - o) <= REL * np.abs(o)).all(), "row normalisers differ"
    gr = rlive & ~samp[:, None]
    assert np.array_equal(gpu["row_argmax"][gr], ora["row_argmax"][gr]), "greedy argmax differs"
    sm = ~bad & samp
    a, o = gpu["resid_mass"][sm].astype(np.float64), ora["resid_mass"][sm]
    assert (np.abs(a - o) <= RESID_ATOL + REL * np.abs(o)).all(), "residual mass differs"

    # Acceptance histogram (same pass): the GPU's own num_accepted exactly,
    # and the oracle's except for the borderline requests.
    if "accept_hist" in gpu:
        hist = gpu["accept_hist"].astype(np.int64)
        own = np.bincount(gpu["num_accepted"][~bad], minlength=g + 1)[:g + 1]
        assert np.array_equal(hist[:g + 1], own), "accept_hist differs from num_accepted"
        assert hist[g + 1] == int(bad.sum()), "accept_hist bad-request count differs"
        ref = np.bincount(ora["num_accepted"][~bad], minlength=g + 1)[:g + 1]
        assert np.abs(hist[:g + 1] - ref).sum() <= 2 * int(border.sum()), "accept_hist vs oracle"

    # Inside the band a decision may differ by rounding, but fp32 rounding is
    # far below the band: most borderline requests must still match exactly,
    # so a systematic error cannot hide behind the band.
    bl = np.nonzero(border)[0]
    bl_match = int(sum(np.array_equal(gpu["tokens"][b], ora["tokens"][b]) for b in bl))
    if bl.size >= 4:
        assert bl_match >= 0.75 * bl.size, f"only {bl_match}/{bl.size} borderline match"

    rep = {"requests": int(B), "bad": int(bad.sum()), "exact": int(exact.sum()),
           "draw_border": int(draw_border.sum()), "draw_border_matching": draw_matching,
           "borderline": int(border.sum()), "borderline_matching": bl_match,
           "mean_accepted": float(ora["num_accepted"][~bad].mean()) if (~bad).any() else 0.0}
    if label is not None:
        REPORTS.append((label, rep))
    return rep
