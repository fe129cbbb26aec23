"""The parity checkers themselves, on the CPU: a planted mistake in a GPU-like
output must make them fail (tie flag inverted, always 0, one flag flipped; an
argmax offset that is not a maximiser)."""
import numpy as np
import pytest
import torch

import synth
from oracle import OracleParams, msa_reference
from parity import TIE_BAND, TIE_MARGIN, check_argmax_row, check_tie_flags


def _tied_case():
    """A small step whose earlier key blocks repeat: block 1 is a copy of
    block 0 and block 3 of block 2, so equal pooled scores straddle the
    selection boundary on many rows (gap 0 < 1e-3)."""
    w = synth.custom([1024], 2, 1, 64, 32, 3, seed=11)
    inp = synth.make_inputs(w)
    kp = inp["k_p"].clone()
    kp[128:256] = kp[0:128]
    kp[384:512] = kp[256:384]
    inp["k_p"] = kp
    ref = msa_reference(inp, OracleParams(w.hq, w.hkv, w.d, w.dp, w.top_k), with_grads=False)
    return ref


def test_tie_flags_accept_the_oracle_reading_and_reject_mistakes():
    gap = _tied_case()["tie_gap"]
    want = (gap < TIE_BAND).astype(np.uint8)
    assert want.sum() > 10 and (want == 0).sum() > 10  # both readings occur
    assert check_tie_flags(want, gap) == 0
    with pytest.raises(AssertionError):
        check_tie_flags(1 - want, gap)  # inverted
    with pytest.raises(AssertionError):
        check_tie_flags(np.zeros_like(want), gap)  # never set
    far = np.nonzero(np.abs(gap.ravel() - TIE_BAND) > TIE_MARGIN)[0]
    one = want.copy().ravel()
    one[far[len(far) // 2]] ^= 1
    with pytest.raises(AssertionError):
        check_tie_flags(one.reshape(want.shape), gap)  # a single flipped flag
    bad = want.copy()
    bad[0, 0] = 2
    with pytest.raises(AssertionError):
        check_tie_flags(bad, gap)  # not a flag


def test_tie_flags_excuse_only_the_margin_around_the_band_edge():
    gap = np.array([[TIE_BAND - TIE_MARGIN / 2, TIE_BAND + TIE_MARGIN / 2, np.inf, 0.0]])
    assert check_tie_flags(np.array([[0, 1, 0, 1]]), gap) == 2
    with pytest.raises(AssertionError):
        check_tie_flags(np.array([[1, 0, 1, 1]]), gap)  # inf gap: no choice, no tie
    with pytest.raises(AssertionError):
        check_tie_flags(np.array([[1, 0, 0, 0]]), gap)  # zero gap must be flagged


def test_argmax_checker_rejects_a_non_maximising_key():
    scores = {(0, 5): 2.0, (0, 9): 2.0 - 5e-4, (0, 1): 1.0, (2, 3): 0.5}
    pooled = np.array([2.0, 0.0, 0.5])

    def score_of(b, a):
        return scores.get((b, a), -np.inf)

    sel, own = [0, 2, -1], [0, 2, -1]
    assert check_argmax_row(sel, [5, 3, 0], own, [5, 3, 0], pooled, score_of) == 0
    assert check_argmax_row(sel, [9, 3, 0], own, [5, 3, 0], pooled, score_of) == 1  # within band
    with pytest.raises(AssertionError):
        check_argmax_row(sel, [1, 3, 0], own, [5, 3, 0], pooled, score_of)
    with pytest.raises(AssertionError):
        check_argmax_row(sel, [5, 4, 0], own, [5, 3, 0], pooled, score_of)  # not causal / unknown
