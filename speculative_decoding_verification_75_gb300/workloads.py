"""Seeded synthetic inputs for the verification step.

This module only draws inputs.  It holds none of the verification step's
arithmetic: the target softmax, the accept test, the residual and the draws
all live in the CUDA library (and, independently, in the test oracle).  It
does synthesise the *draft* model's distribution q, which is an input of the
step: a softmax of noisy copies of the target logits, as a stand-in for a
small draft model aligned with the target (the pages' draft models need
trained weights).

The five workloads mirror the shapes the speculative-decoding pages talk
about: Llama-2 / Llama-3 / Qwen2.5 vocabularies (32000 / 128256 / 151936),
gamma 3..8 draft tokens, batches 1..256, and temperatures 0 (greedy), 0.7,
0.8 and 1.0 (the tutorial's SamplingParams and its temperature pitfall).

Recipe, per request b and row i (all fp32 until the final cast):
  target logits  l[b, i, :] ~ N(0, sigma^2), plus ``boost`` added to
                 floor(boost_frac * V) distinct uniformly chosen entries;
                 cast to the workload's dtype (bf16 or fp32);
  draft logits   d[b, i, :] = float(l[b, i, :]) + N(0, noise_b^2)  (i < gamma)
  draft probs    q = softmax(d / T_b) for T_b > 0, one-hot(argmax d) at T_b = 0
  draft token    x[b, i] ~ q[b, i, :]  (argmax d at T_b = 0)
  uniforms       u_accept[b, i], u_sample[b] ~ U[0, 1)
Positions past a request's draft length hold invalid sentinels (token -1,
uniform 2.0, NaN logits rows) so that any read of them shows up in tests.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Optional, Tuple

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    gamma: int                     # gamma_max: padded number of draft slots
    V: int
    dtype: str                     # "bf16" or "fp32"
    sigma: float                   # std of the target logits
    noise: Tuple[float, float]     # draft noise std, drawn U[lo, hi] per request
    temperatures: Tuple[float, ...]  # per-request T drawn uniformly from these
    gamma_range: Optional[Tuple[int, int]] = None  # ragged draft lengths
    boost_frac: float = 0.0
    boost: float = 0.0
    seed: int = 0
    note: str = ""

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "c1": Workload("c1_B1_g5_V32000_fp32", 1, 5, 32000, "fp32", 2.0, (0.5, 0.5),
                   (1.0,), seed=0, note="single request, Llama-2 vocabulary"),
    "c2": Workload("c2_B8_g5_V151936_bf16", 8, 5, 151936, "bf16", 3.0,
                   (1.0, 1.0), (0.8,), seed=1, note="small batch, Qwen2.5 vocabulary"),
    "c3": Workload("c3_B128_g5_V151936_bf16_peaky", 128, 5, 151936, "bf16", 3.0,
                   (0.7, 0.7), (0.8,), boost_frac=0.01, boost=8.0, seed=2,
                   note="128 concurrent requests, peaky rows"),
    "c4": Workload("c4_B64_g8_V128256_bf16", 64, 8, 128256, "bf16", 2.0,
                   (2.0, 2.0), (1.0,), seed=3, note="low draft alignment, Llama-3 vocabulary"),
    "c5": Workload("c5_B256_g3-7_V151936_bf16_mixedT", 256, 7, 151936, "bf16", 3.0,
                   (0.3, 2.0), (0.0, 0.7, 1.0), gamma_range=(3, 7), seed=4,
                   note="ragged draft lengths, mixed greedy / sampled requests"),
}


def workload(key: str, **overrides) -> Workload:
    w = WORKLOADS[key]
    return w.with_(**overrides) if overrides else w


def _torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "fp32": torch.float32}[name]


@torch.no_grad()
def make_case(w: Workload, device="cpu", seed: Optional[int] = None,
              draft_probs: bool = True) -> dict:
    """Draw one batch of inputs for workload ``w`` on ``device``.

    Returns a dict with ``logits`` [B, g+1, V], ``draft_ids`` [B, g] int32,
    ``draft_probs`` [B, g, V] fp32 (None when ``draft_probs`` is False: the
    drafts are then deterministic and q is one-hot at the drafted token),
    ``u_accept`` [B, g], ``u_sample`` [B], ``temperature`` [B] fp32 and
    ``draft_lens`` [B] int32 (None when every request drafts g tokens).
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    B, g, V = w.B, w.gamma, w.V
    f32 = dict(device=device, dtype=torch.float32)

    def rand(*shape):
        return torch.rand(*shape, generator=gen, **f32)

    # Per-request draft length, noise level and temperature.
    if w.gamma_range is not None:
        lo, hi = w.gamma_range
        lens = torch.randint(lo, hi + 1, (B,), generator=gen, device=device,
                             dtype=torch.int32)
    else:
        lens = torch.full((B,), g, device=device, dtype=torch.int32)
    nlo, nhi = w.noise
    noise = nlo + (nhi - nlo) * rand(B)
    tchoice = torch.tensor(w.temperatures, **f32)
    temperature = tchoice[torch.randint(0, len(w.temperatures), (B,),
                                        generator=gen, device=device)]

    # Target logits.
    logits = w.sigma * torch.randn(B, g + 1, V, generator=gen, **f32)
    nboost = int(w.boost_frac * V)
    if nboost > 0:
        rows = logits.view(B * (g + 1), V)
        for r0 in range(0, rows.shape[0], 64):  # bounded temporary memory
            r1 = min(rows.shape[0], r0 + 64)
            idx = rand(r1 - r0, V).topk(nboost, dim=1).indices
            rows[r0:r1].scatter_add_(1, idx, torch.full(idx.shape, w.boost, **f32))
    logits = logits.to(_torch_dtype(w.dtype))

    # Draft distributions: noisy copies of the (rounded) target rows.
    ids = torch.empty(B, g, device=device, dtype=torch.int32)
    q_all = torch.empty(B, g, V, **f32) if draft_probs else None
    for b in range(B if g > 0 else 0):
        d = logits[b, :g].float() + noise[b] * torch.randn(g, V, generator=gen, **f32)
        T = float(temperature[b])
        if T > 0:
            q = torch.softmax(d / T, dim=-1)
            x = torch.multinomial(q, 1, generator=gen).view(g).to(torch.int32)
        else:
            x = d.argmax(dim=-1).to(torch.int32)
            q = torch.zeros(g, V, **f32)
            q.scatter_(1, x.view(g, 1).long(), 1.0)
        ids[b] = x
        if q_all is not None:
            q_all[b] = q

    u_accept = rand(B, g)
    u_sample = rand(B)

    # Invalid sentinels past each request's draft length.
    if w.gamma_range is not None:
        pos = torch.arange(g, device=device).view(1, g)
        pad = pos >= lens.view(B, 1).long()
        ids[pad] = -1
        u_accept[pad] = 2.0
        row_pad = torch.arange(g + 1, device=device).view(1, g + 1) > lens.view(B, 1).long()
        logits[row_pad] = float("nan")

    return {
        "logits": logits,
        "draft_ids": ids,
        "draft_probs": q_all,
        "u_accept": u_accept,
        "u_sample": u_sample,
        "temperature": temperature,
        "draft_lens": lens if w.gamma_range is not None else None,
    }


def verified_rows(case: dict) -> int:
    """Draft rows one call verifies: the sum of the draft lengths."""
    if case["draft_lens"] is not None:
        return int(case["draft_lens"].sum())
    B, g = case["draft_ids"].shape
    return B * g
