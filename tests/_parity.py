"""Comparison rules shared by the GPU parity tests.

The method's statement fixes the bars:
  * token ids, accept lengths and l_r are bit-exact, except where the oracle's decision
    sits in the tie band -- the top-two Gumbel scores within TIE of each other, or
    |u - p/q| within TIE -- and such cases must stay below 1e-4 of the positions;
  * probabilities and confidences (q_tok, row max / sum, c, a) agree within RTOL relative.

The band is checked at the decision where the two paths first part: for a draft row, the
first position whose token differs (later positions legitimately follow another path);
for a verification, the first position whose accept / reject outcome differs, or, when
the accept lengths agree, the correction or bonus draw.  Every helper returns the counts
it saw so that a test can report them and hold the rate bound over a whole batch.
"""
from __future__ import annotations

import numpy as np

TIE = 1e-5
RTOL = 1e-5
MAX_TIE_RATE = 1e-4


def draft_rows(got_tokens, ref_tokens, ref_gap, label=""):
    """Draft tokens [n, gamma]: identical up to the first differing position of each row,
    and that position's draw is in the oracle's tie band.

    Returns (diverged rows, mask of the positions before any divergence)."""
    got_tokens = np.asarray(got_tokens)
    ref_tokens = np.asarray(ref_tokens)
    diff = got_tokens != ref_tokens
    diverged = 0
    for i in np.nonzero(diff.any(axis=1))[0]:
        k = int(np.argmax(diff[i]))
        assert ref_gap[i, k] <= TIE, (
            f"{label}: row {i} position {k + 1}: {got_tokens[i, k]} vs {ref_tokens[i, k]} "
            f"(oracle top-two gap {ref_gap[i, k]:.3g} outside the tie band)")
        diverged += 1
    same = np.cumprod(~diff, axis=1).astype(bool)
    return diverged, same


def draft_stats(got, ref, same, keys=("q_tok", "row_max", "row_sumexp"), label=""):
    """Probabilities and row statistics within RTOL on the positions both paths share."""
    for key in keys:
        np.testing.assert_allclose(np.asarray(got[key])[same], np.asarray(ref[key])[same],
                                   rtol=RTOL, err_msg=f"{label}: {key}")


def verify_rows(got, ref, label=""):
    """Verification outputs of the same drafted tokens and verified lengths.

    A row whose accept length or emitted tokens differ must have its first differing
    decision in the tie band: the accept test of position min(accept lengths) + 1 when the
    lengths differ, else the correction / bonus draw.  Returns the number of such rows."""
    diverged = 0
    for i in range(len(ref["accept_len"])):
        ga, ra = int(got["accept_len"][i]), int(ref["accept_len"][i])
        if ga == ra and np.array_equal(got["out_tokens"][i], ref["out_tokens"][i]):
            continue
        if ga != ra:
            j = min(ga, ra)                          # 0-based index of that position
            band = ref["band"][i, j]
            assert np.isfinite(band) and band <= TIE, (
                f"{label}: row {i}: accept length {ga} vs {ra}; the accept test of position "
                f"{j + 1} has |u - p/q| = {band:.3g}, outside the tie band")
        else:
            assert ref["gap"][i] <= TIE, (
                f"{label}: row {i}: {got['out_tokens'][i]} vs {ref['out_tokens'][i]}; the final "
                f"draw's top-two gap {ref['gap'][i]:.3g} is outside the tie band")
        diverged += 1
    return diverged


def band_cases_draft(ref_gap):
    """Draft positions whose draw is in the tie band (the oracle's top-two gap)."""
    return int(np.sum(np.asarray(ref_gap) <= TIE))


def band_cases_verify(ref):
    """Verification decisions in the tie band: accept tests and final draws."""
    band = np.asarray(ref["band"])
    return int(np.sum(np.isfinite(band) & (band <= TIE)) + np.sum(np.asarray(ref["gap"]) <= TIE))


def assert_rate(cases, positions, label=""):
    """Tie-band cases below MAX_TIE_RATE of the positions (no floor)."""
    assert cases <= MAX_TIE_RATE * positions, (
        f"{label}: {cases} tie-band cases in {positions} positions "
        f"(rate {cases / max(1, positions):.2e} >= {MAX_TIE_RATE:g})")
