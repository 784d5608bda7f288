"""Pins of the fp64 oracle to facts fixed outside the oracle itself.

Every pin takes an ``oracle.Oracle`` handle and raises ``AssertionError`` if
the oracle disagrees with what the speculative-decoding tutorial page
(dpshk.com/news/5598276, "P3") or plain mathematics fixes:

  worked_example       P3 §4 flow diagram (golden file with hand derivation)
  lossless             P3 §3.2: the emitted token is distributed exactly as p
  expected_emitted     P3 §3.3: E[emitted] = (1 - a^(g+1)) / (1 - a) and the
                       truncated-geometric law behind it
  first_rejection      P3 §5.2 step (4): cumprod keeps only the leading run
  clamp                P3 §5.2 step (2): q is clamped at 1e-10
  bonus                P3 §5.3: all accepted -> g+1 tokens, last from row g
  greedy               P3 §8 pitfall 2: T = 0 is greedy (argmax agreement)
  temperature          closed-form softmax of l / T
  normaliser           scipy's logsumexp (an independent library routine)
  inverse_cdf          numpy searchsorted on the cumulative sum
  deterministic_drafts P3 §7 prompt lookup: q one-hot at the draft, lossless
  empty_residual       the reading for sum (p - q)_+ = 0: draw from p
  bad_inputs / ragged / zero_drafts  the documented edge-case contract
  temperature_range    the reading that a temperature so small that the row
                       maximum in log2 units, m log2(e) / T, reaches 2^24 in
                       binary32 is invalid

``scale`` shrinks the Monte Carlo sizes (the mutation tests use 0.1).
"""
from __future__ import annotations

import json
import math
from pathlib import Path

import numpy as np
from scipy import special, stats

GOLDEN = Path(__file__).resolve().parent / "golden"


def _ln(p):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(p, np.float64)).astype(np.float32)


def _softmax64(row):
    z = np.asarray(row, np.float64)
    e = np.exp(z - z.max())
    return e / e.sum()


def _unit(q):
    q = np.asarray(q, np.float64)
    return q / q.sum()


def _chi2_pvalue(counts, probs):
    counts = np.asarray(counts, np.float64)
    n = counts.sum()
    exp = n * np.asarray(probs, np.float64)
    keep = exp > 0
    assert counts[~keep].sum() == 0, "mass on a zero-probability token"
    stat = ((counts[keep] - exp[keep]) ** 2 / exp[keep]).sum()
    return stats.chi2.sf(stat, keep.sum() - 1)


# ---------------------------------------------------------------- P3 §4 ----
def pin_worked_example(orc, scale=1.0):
    g = json.loads((GOLDEN / "worked_example_p3_s4.json").read_text())
    logits = _ln(g["p_rows"])[None]
    q = np.asarray(g["q_rows"], np.float32)[None]
    r = orc.verify(logits, np.array([g["draft_ids"]]), q,
                   np.array([g["u_accept"]], np.float32),
                   np.array([g["u_sample"]], np.float32),
                   np.array([g["temperature"]], np.float32))
    e = g["expected"]
    np.testing.assert_allclose(r["accept_prob"][0], e["accept_prob"], rtol=1e-6)
    assert r["flags"][0].tolist() == e["flags"]
    assert r["num_accepted"][0] == e["num_accepted"]
    assert r["tokens"][0].tolist() == e["tokens"]
    assert int((r["tokens"][0] >= 0).sum()) == e["emitted"]
    np.testing.assert_allclose(r["resid_mass"][0], e["residual_mass"], rtol=1e-6)
    np.testing.assert_allclose(r["sample_margin"][0], e["sample_margin"], rtol=1e-4)


# -------------------------------------------------------------- P3 §3.2 ----
def pin_lossless(orc, scale=1.0, seed=11):
    """x ~ q, accept with min(1, p/q), else resample: the emitted token at
    position 0 must follow p_0; the bonus token must follow p_1."""
    n = int(1_000_000 * scale)
    rng = np.random.default_rng(seed)
    p0 = np.array([0.30, 0.05, 0.20, 0.25, 0.15, 0.05])
    q0 = np.array([0.10, 0.30, 0.25, 0.05, 0.10, 0.20])
    p1 = np.array([0.05, 0.15, 0.10, 0.30, 0.25, 0.15])
    V = p0.size
    rows = _ln(np.stack([p0, p1]))
    logits = np.ascontiguousarray(np.broadcast_to(rows, (n, 2, V)))
    q32 = q0.astype(np.float32)
    q = np.ascontiguousarray(np.broadcast_to(q32, (n, 1, V)))
    x = rng.choice(V, size=n, p=_unit(q32))
    u_acc = rng.random((n, 1), dtype=np.float32)
    u_smp = rng.random(n, dtype=np.float32)
    r = orc.verify(logits, x.reshape(n, 1), q, u_acc, u_smp,
                   np.ones(n, np.float32))
    p0_exact = _softmax64(rows[0])
    p1_exact = _softmax64(rows[1])
    pv = _chi2_pvalue(np.bincount(r["tokens"][:, 0], minlength=V), p0_exact)
    assert pv > 1e-4, f"emitted token is not distributed as p (p-value {pv:.2e})"
    alpha = np.minimum(p0_exact, _unit(q32)).sum()
    acc = r["flags"][:, 0].mean()
    assert abs(acc - alpha) < 5 * math.sqrt(alpha * (1 - alpha) / n), (acc, alpha)
    bonus = r["tokens"][r["num_accepted"] == 1, 1]
    pv = _chi2_pvalue(np.bincount(bonus, minlength=V), p1_exact)
    assert pv > 1e-4, f"bonus token is not distributed as p_g (p-value {pv:.2e})"


# -------------------------------------------------------------- P3 §3.3 ----
def pin_expected_emitted(orc, scale=1.0, seed=12, gamma=5):
    """Same p, q at every position, x_i ~ q: each draft is kept with
    probability alpha = sum min(p, q), so num_accepted is a truncated
    geometric and E[num_accepted + 1] = (1 - alpha^(g+1)) / (1 - alpha)."""
    n = int(200_000 * scale)
    rng = np.random.default_rng(seed)
    p = np.array([0.40, 0.25, 0.15, 0.10, 0.06, 0.04])
    q = np.array([0.30, 0.30, 0.10, 0.05, 0.05, 0.20])
    V = p.size
    lrow = _ln(p)
    logits = np.ascontiguousarray(np.broadcast_to(lrow, (n, gamma + 1, V)))
    q32 = q.astype(np.float32)
    qq = np.ascontiguousarray(np.broadcast_to(q32, (n, gamma, V)))
    x = rng.choice(V, size=(n, gamma), p=_unit(q32))
    r = orc.verify(logits, x, qq, rng.random((n, gamma), dtype=np.float32),
                   rng.random(n, dtype=np.float32), np.ones(n, np.float32))
    alpha = np.minimum(_softmax64(lrow), _unit(q32)).sum()
    N = r["num_accepted"] + 1
    E = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    assert abs(N.mean() - E) < 5 * N.std() / math.sqrt(n), (N.mean(), E)
    law = np.array([alpha ** k * (1 - alpha) for k in range(gamma)] + [alpha ** gamma])
    pv = _chi2_pvalue(np.bincount(r["num_accepted"], minlength=gamma + 1), law)
    assert pv > 1e-4, f"num_accepted is not truncated-geometric (p-value {pv:.2e})"


# --------------------------------------------------------- P3 §5.2 (4) ----
def pin_first_rejection(orc, scale=1.0):
    """Raw flags 1,1,0,1,1 keep 2 drafts: a later acceptance never counts."""
    V, g = 4, 5
    unif = [0.25] * 4
    p_rows = [unif, unif, [0.1, 0.3, 0.3, 0.3], unif, unif, unif]
    q_rows = [unif, unif, [0.2, 0.2, 0.3, 0.3], unif, unif]
    r = orc.verify(_ln(p_rows)[None], np.array([[3, 1, 0, 2, 2]]),
                   np.array([q_rows], np.float32),
                   np.array([[0.9, 0.9, 0.9, 0.9, 0.9]], np.float32),
                   np.array([0.99], np.float32), np.array([1.0], np.float32))
    assert r["flags"][0].tolist() == [1, 1, 0, 1, 1]
    assert r["num_accepted"][0] == 2
    # the residual (p - q)_+ = [0, 0.1, 0, 0] puts all its mass on token 1
    assert r["tokens"][0].tolist() == [3, 1, 1, -1, -1, -1]
    np.testing.assert_allclose(r["accept_prob"][0], [1, 1, 0.5, 1, 1], rtol=1e-6)


# --------------------------------------------------------- P3 §5.2 (2) ----
def pin_clamp(orc, scale=1.0):
    """a = min(1, p / max(q, 1e-10)): with p(x) = 5e-11 a zero or tiny q gives
    a = 0.5 (not 1 or 0), and q = 2e-10 gives a = 0.25."""
    p = [5e-11, 1 - 5e-11]
    lrow = _ln(p)
    logits = np.ascontiguousarray(np.broadcast_to(lrow, (6, 2, 2)))
    q = np.array([[[0.0, 1.0]], [[0.0, 1.0]], [[1e-12, 1.0]], [[1e-12, 1.0]],
                  [[2e-10, 1.0]], [[2e-10, 1.0]]], np.float32)
    u = np.array([[0.4], [0.6], [0.4], [0.6], [0.2], [0.3]], np.float32)
    r = orc.verify(logits, np.zeros((6, 1), np.int32), q, u,
                   np.full(6, 0.5, np.float32), np.ones(6, np.float32))
    np.testing.assert_allclose(r["accept_prob"][:, 0],
                               [0.5, 0.5, 0.5, 0.5, 0.25, 0.25], rtol=1e-4)
    assert r["flags"][:, 0].tolist() == [1, 0, 1, 0, 1, 0]


# -------------------------------------------------------------- P3 §5.3 ----
def pin_bonus(orc, scale=1.0):
    """Every draft kept -> g+1 tokens; the last is the inverse-CDF draw on
    row g (not row g-1) with the sampling uniform."""
    g = 3
    unif = [0.2] * 5
    p_rows = [unif, unif, unif, [0.1, 0.2, 0.3, 0.25, 0.15]]
    logits = _ln(p_rows)[None]
    q = np.array([[unif, unif, unif]], np.float32)
    for u_s, tok in ((0.35, 2), (0.05, 0), (0.95, 4), (0.31, 2), (0.29, 1)):
        r = orc.verify(logits, np.array([[4, 0, 3]]), q,
                       np.zeros((1, g), np.float32),
                       np.array([u_s], np.float32), np.array([1.0], np.float32))
        assert r["num_accepted"][0] == g
        assert r["tokens"][0].tolist() == [4, 0, 3, tok], (u_s, r["tokens"])


# -------------------------------------------------------- P3 §8 (T = 0) ----
def pin_greedy(orc, scale=1.0):
    """T = 0: a draft is kept iff it is the lowest-index argmax (u = 0 still
    rejects a = 0: the test is strict); the first mismatch emits the argmax;
    all kept emits the argmax of row g."""
    rows = np.array([[0.5, 2.0, 1.0, -1.0],
                     [1.0, 3.0, 3.0, 2.0],      # tie: argmax is index 1
                     [4.0, 1.0, 0.0, 4.5],
                     [0.0, 0.0, 9.0, 0.0]], np.float32)
    onehot = lambda ids: np.eye(4, dtype=np.float32)[ids][None]
    ids = np.array([[1, 1, 0]])
    r = orc.verify(rows[None], ids, onehot(ids[0]), np.zeros((1, 3), np.float32),
                   np.array([0.5], np.float32), np.array([0.0], np.float32))
    assert r["flags"][0].tolist() == [1, 1, 0]
    assert r["tokens"][0].tolist() == [1, 1, 3, -1]
    ids = np.array([[1, 1, 3]])
    r = orc.verify(rows[None], ids, onehot(ids[0]), np.zeros((1, 3), np.float32),
                   np.array([0.5], np.float32), np.array([0.0], np.float32))
    assert r["tokens"][0].tolist() == [1, 1, 3, 2]
    ids = np.array([[1, 2, 3]])   # index 2 ties the max but is not the lowest
    r = orc.verify(rows[None], ids, onehot(ids[0]), np.zeros((1, 3), np.float32),
                   np.array([0.5], np.float32), np.array([0.0], np.float32))
    assert r["tokens"][0].tolist() == [1, 1, -1, -1]
    assert r["num_accepted"][0] == 1


# ------------------------------------------------------ temperature l / T ----
def pin_temperature(orc, scale=1.0):
    """Logits [0, 2 ln 2]: T = 2 gives p = [1/3, 2/3], T = 0.5 gives
    [1/17, 16/17]; T scales the logits before the softmax.  Both tokens are
    checked, so the non-maximal one pins the scaling of l - max as well."""
    lrow = np.array([0.0, 2 * math.log(2)], np.float32)
    logits = np.ascontiguousarray(np.broadcast_to(lrow, (4, 2, 2)))
    q = np.ones((4, 1, 2), np.float32)
    r = orc.verify(logits, np.array([[0], [1], [0], [1]]), q,
                   np.full((4, 1), 0.99, np.float32), np.full(4, 0.5, np.float32),
                   np.array([2.0, 2.0, 0.5, 0.5], np.float32))
    np.testing.assert_allclose(r["p_tok"][:, 0], [1 / 3, 2 / 3, 1 / 17, 16 / 17],
                               rtol=1e-6)
    np.testing.assert_allclose(r["row_sum"][:, 0], [1.5, 1.5, 17 / 16, 17 / 16],
                               rtol=1e-6)


# ----------------------------------------------------- softmax normaliser ----
def pin_normaliser(orc, scale=1.0, seed=13):
    """log(s) + max/T equals scipy's logsumexp(l / T); bf16 rows decode
    exactly (same statistics as their fp32 widening)."""
    import torch
    rng = np.random.default_rng(seed)
    for T in (0.5, 1.0, 2.5):
        row = rng.normal(0.0, 3.0, 5000).astype(np.float32)
        m, s, a = orc.row_stats(row, T)
        assert m == float(row.max()) and a == int(np.argmax(row))
        ref = special.logsumexp(row.astype(np.float64) / T)
        assert abs(math.log(s) + m / T - ref) <= 1e-12 * abs(ref) + 1e-12
        tb = torch.from_numpy(row).to(torch.bfloat16)
        mb, sb, ab = orc.row_stats(tb, T)
        mf, sf, af = orc.row_stats(tb.float().numpy(), T)
        assert (mb, sb, ab) == (mf, sf, af)
    m, s, a = orc.row_stats(np.array([3.0, -1.0, 3.0], np.float32), 0.0)
    assert (m, s, a) == (3.0, 1.0, 0)


# ------------------------------------------------------------ inverse CDF ----
def pin_inverse_cdf(orc, scale=1.0):
    """token = min{j : C_j > u S}; zero-weight tokens are never drawn."""
    for w in ([0.0, 0.2, 0.0, 0.5, 0.3, 0.0], [0.7], [0.0, 0.0, 1e-300, 0.0],
              [0.25, 0.25, 0.25, 0.25]):
        w = np.asarray(w, np.float64)
        c = np.cumsum(w)
        for u in np.linspace(0.0, 0.999999, 397):
            tok, margin = orc.inverse_cdf(w, u)
            assert tok == int(np.searchsorted(c, u * c[-1], side="right")), (w, u)
            assert w[tok] > 0
            lo = c[tok - 1] if tok > 0 else 0.0
            assert abs(margin - min(u * c[-1] - lo, c[tok] - u * c[-1])) < 1e-15


# ------------------------------------------------ P3 §7 prompt lookup ------
def pin_deterministic_drafts(orc, scale=1.0, seed=14):
    """No draft probabilities: q is one-hot at the drafted token, so
    a = p(x) and the residual is p with x removed; still lossless."""
    n = int(400_000 * scale)
    rng = np.random.default_rng(seed)
    p0 = np.array([0.1, 0.2, 0.4, 0.2, 0.1])
    lrow = _ln(p0)
    logits = np.ascontiguousarray(np.broadcast_to(lrow, (n, 2, 5)))
    r = orc.verify(logits, np.full((n, 1), 2), None,
                   rng.random((n, 1), dtype=np.float32),
                   rng.random(n, dtype=np.float32), np.ones(n, np.float32))
    pex = _softmax64(lrow)
    np.testing.assert_allclose(r["accept_prob"][:, 0], pex[2], rtol=1e-6)
    rej = r["num_accepted"] == 0
    assert (r["tokens"][rej, 0] != 2).all()
    pv = _chi2_pvalue(np.bincount(r["tokens"][:, 0], minlength=5), pex)
    assert pv > 1e-4, f"prompt-lookup output not distributed as p ({pv:.2e})"


# -------------------------------------------------- empty residual reading ----
def pin_empty_residual(orc, scale=1.0):
    """q = 2p (inconsistent caller data): a = 0.5 and (p - q)_+ = 0, so the
    reading draws from p itself."""
    p = np.array([0.1, 0.2, 0.3, 0.4])
    lrow = _ln(p)
    logits = np.ascontiguousarray(np.broadcast_to(lrow, (1, 2, 4)))
    q = (2 * p).astype(np.float32)[None, None]
    r = orc.verify(logits, np.array([[3]]), q, np.array([[0.7]], np.float32),
                   np.array([0.45], np.float32), np.array([1.0], np.float32))
    assert r["num_accepted"][0] == 0 and r["resid_mass"][0] == 0.0
    assert r["sample_fallback"][0] == 1
    assert r["tokens"][0].tolist() == [2, -1]   # C = .1 .3 .6 1; 0.45 -> 2


# ------------------------------------------------------ edge-case contract ----
def pin_bad_inputs(orc, scale=1.0):
    """Each invalid input marks only its own request: -1 everywhere."""
    B, g, V = 8, 2, 3
    logits = np.zeros((B, g + 1, V), np.float32)
    logits[6, 1, 0] = np.inf
    ids = np.zeros((B, g), np.int32)
    u = np.full((B, g), 0.5, np.float32)
    us = np.full(B, 0.5, np.float32)
    T = np.ones(B, np.float32)
    lens = np.full(B, g, np.int32)
    lens[1] = g + 1            # BAD_DRAFT_LEN
    T[2] = -1.0                # BAD_TEMP
    ids[3, 1] = V              # BAD_TOKEN
    u[4, 0] = 1.0              # BAD_U_ACCEPT
    us[5] = np.nan             # BAD_U_SAMPLE
    T[7] = 1e-40               # subnormal temperature: BAD_TEMP
    r = orc.verify(logits, ids, None, u, us, T, lens)
    assert r["bad"].tolist() == [0, 1, 2, 4, 8, 16, 32, 2]
    assert (r["num_accepted"][1:] == -1).all() and (r["tokens"][1:] == -1).all()
    assert r["num_accepted"][0] >= 0
    # draft slots past a short draft length are never validated or read
    lens2 = np.array([1], np.int32)
    r = orc.verify(np.zeros((1, g + 1, V), np.float32), np.array([[0, -5]]),
                   None, np.array([[0.5, 7.0]], np.float32),
                   np.array([0.5], np.float32), np.ones(1, np.float32), lens2)
    assert r["bad"][0] == 0


def pin_ragged(orc, scale=1.0, seed=15):
    """A request with draft length g_b < gamma_max gives the same result as
    the same request padded to exactly g_b slots; rows past g_b are unread."""
    rng = np.random.default_rng(seed)
    V, gmax = 7, 5
    for gb in range(gmax + 1):
        logits = rng.normal(0, 2, (1, gmax + 1, V)).astype(np.float32)
        logits[0, gb + 1:] = np.nan
        q = rng.dirichlet(np.ones(V), (1, gmax)).astype(np.float32)
        ids = rng.integers(0, V, (1, gmax)).astype(np.int32)
        u = rng.random((1, gmax), dtype=np.float32)
        us = rng.random(1, dtype=np.float32)
        T = np.array([0.9], np.float32)
        r = orc.verify(logits, ids, q, u, us, T, np.array([gb], np.int32))
        t = orc.verify(np.ascontiguousarray(logits[:, :gb + 1]), ids[:, :gb],
                       np.ascontiguousarray(q[:, :gb]), u[:, :gb], us, T)
        assert r["num_accepted"][0] == t["num_accepted"][0]
        assert r["tokens"][0, :gb + 1].tolist() == t["tokens"][0].tolist()
        assert (r["tokens"][0, gb + 1:] == -1).all()


def pin_zero_drafts(orc, scale=1.0):
    """Draft length 0: the step is one plain draw from row 0."""
    p = np.array([0.5, 0.3, 0.2])
    logits = np.stack([_ln(p), _ln([1 / 3] * 3)])[None]
    r = orc.verify(logits, np.array([[1]]), None, np.array([[0.5]], np.float32),
                   np.array([0.6], np.float32), np.array([1.0], np.float32),
                   np.array([0], np.int32))
    assert r["num_accepted"][0] == 0
    assert r["tokens"][0].tolist() == [1, -1]    # C = .5 .8 1; 0.6 -> 1


def pin_temperature_range(orc, scale=1.0):
    """Reading (the pages' logits are binary32 tensors, so the step runs in
    binary32): a request whose row maximum in log2 units, m * log2(e) / T,
    reaches 2^24 in magnitude (product and quotient rounded to binary32) has
    invalid data (BAD_NORMALISER = 32).  The same tiny T with a row maximum
    of 0 is a valid, one-hot request; so is a product just below 2^24."""
    V = 4
    #   m = 100, T = 1e-37: 1.4e39, beyond binary32 altogether
    #   m = 0,   T = 1e-37: offset 0, every other exponent below -2^24
    #   m = 10,  T = 1e-30: 1.4e31 >= 2^24
    #   m = 1,   T = 1e-7:  1.44e7 < 2^24 = 1.68e7
    #   m = 1,   T = 8e-8:  1.80e7 >= 2^24
    T = np.array([1e-37, 1e-37, 1e-30, 1e-7, 8e-8], np.float32)
    top = [100.0, 0.0, 10.0, 1.0, 1.0]
    logits = np.zeros((5, 2, V), np.float32)
    for r, m in enumerate(top):
        logits[r, :, 0] = m
        logits[r, :, 1:] = m - np.array([1.0, 2.0, 3.0], np.float32)
    ids = np.zeros((5, 1), np.int32)
    r = orc.verify(logits, ids, None, np.full((5, 1), 0.5, np.float32),
                   np.full(5, 0.5, np.float32), T)
    assert r["bad"].tolist() == [32, 0, 32, 0, 32]
    assert r["num_accepted"].tolist() == [-1, 1, -1, 1, -1]
    # the valid rows are one-hot at the maximum: draft 0 accepted, bonus 0
    assert r["tokens"][1].tolist() == [0, 0] and r["tokens"][3].tolist() == [0, 0]


ALL_PINS = [pin_worked_example, pin_lossless, pin_expected_emitted,
            pin_first_rejection, pin_clamp, pin_bonus, pin_greedy,
            pin_temperature, pin_normaliser, pin_inverse_cdf,
            pin_deterministic_drafts, pin_empty_residual, pin_bad_inputs,
            pin_ragged, pin_zero_drafts, pin_temperature_range]
