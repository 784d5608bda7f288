"""Each plausible mistake planted in a copy of the oracle (CPU only) must be
caught by at least one pin: this is the evidence that the pins constrain every
step of the oracle, not only its happy path."""
import shutil
import subprocess

import pytest

import oracle
from oracle.build import CFLAGS, SRC
from oracle_pins import ALL_PINS

MUTATIONS = {
    "ratio_transposed": ("P / fmax(q, ORC_Q_FLOOR)", "q / fmax(P, ORC_Q_FLOOR)", 1),
    "accept_not_strict": ("int f = u < a;", "int f = u <= a;", 1),
    "residual_sign": ("r[j] = fmax(p - q, 0.0);", "r[j] = fmax(q - p, 0.0);", 1),
    "residual_unclamped": ("r[j] = fmax(p - q, 0.0);", "r[j] = p - q;", 1),
    "residual_is_q": ("r[j] = fmax(p - q, 0.0);", "r[j] = q;", 1),
    "last_rejection": ("if (f == 0 && k == g)", "if (f == 0)", 1),
    "temperature_multiplies_stats": (
        "s += exp((logit_at(logits, is_bf16, row_offset + (size_t)j) - mx) / T);",
        "s += exp((logit_at(logits, is_bf16, row_offset + (size_t)j) - mx) * T);", 1),
    "temperature_multiplies_prob": ("return exp((l_j - mx) / T) / s;",
                                    "return exp((l_j - mx) * T) / s;", 1),
    "prob_unnormalised": ("return exp((l_j - mx) / T) / s;",
                          "return exp((l_j - mx) / T);", 1),
    "cdf_boundary_inclusive": ("if (c > target) {", "if (c >= target) {", 1),
    "clamp_floor": ("ORC_Q_FLOOR = 1e-10;", "ORC_Q_FLOOR = 1e-12;", 1),
    "argmax_last_tie": ("if (l > mx) {", "if (l >= mx) {", 1),
    "bonus_previous_row": (
        "size_t off = ((size_t)b * rows_per_req + k) * (size_t)V;",
        "size_t off = ((size_t)b * rows_per_req + (k > 0 ? k - 1 : 0)) * (size_t)V;", 1),
    "bf16_decode": ("(uint32_t)h << 16", "(uint32_t)h << 15", 1),
    "sample_uniform_flipped": ("orc_inverse_cdf(resid, V, (double)u_samp[b], &margin)",
                               "orc_inverse_cdf(resid, V, 1.0 - (double)u_samp[b], &margin)", 1),
    "prompt_lookup_keeps_draft": ("q = (j == draft_ids[(size_t)b * gmax + k]) ? 1.0 : 0.0;",
                                  "q = 0.0;", 1),
    "accepted_token_index": ("tok[i] = draft_ids[(size_t)b * gmax + i];",
                             "tok[i] = draft_ids[(size_t)b * gmax];", 1),
    "uniform_closed_interval": ("return u >= 0.0 && u < 1.0;", "return u >= 0.0 && u <= 1.0;", 1),
    "no_fallback": ("if (!(S > 0.0)) {", "if (0) {", 1),
    "greedy_ignored": ("if (T == 0.0)\n        return j == argmax ? 1.0 : 0.0;", "", 1),
    "range_check_dropped": ("!exponent_range_ok(row_m[i], T)", "0", 1),
    "range_limit_off": ("return fabsf(o) < ORC_EXP_LIMIT;", "return isfinite(o);", 1),
}


def _build_mutant(tmp_path, name, old, new, count):
    src = SRC.read_text()
    assert src.count(old) == count, f"{name}: pattern occurs {src.count(old)} times"
    msrc = tmp_path / f"{name}.c"
    msrc.write_text(src.replace(old, new))
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", *CFLAGS, str(msrc), "-o", str(lib), "-lm", "-pthread"], check=True)
    return lib


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(tmp_path, name):
    old, new, count = MUTATIONS[name]
    mutant = oracle.Oracle(_build_mutant(tmp_path, name, old, new, count))
    failed = []
    for pin in ALL_PINS:
        try:
            pin(mutant, scale=0.1)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutation {name!r} passed every pin"
