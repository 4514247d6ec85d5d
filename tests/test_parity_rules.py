"""The parity harness's acceptance rule for a differing H2O victim, on the
CPU: a victim other than the oracle's passes only when it is a live
candidate outside the recent window whose oracle score is within 1e-6
(relative) of the smallest candidate score; a mistake planted in the
device's answer (a slot with a clearly larger score, a slot inside the
window, an append in place of an eviction) must be rejected."""
import numpy as np
import pytest

import oracle
from parity import NEAR_TIE, accept_victims


def _state(scores, pos):
    U, B, d = 1, len(scores), 2
    st = oracle.H2OState(U, B, d)
    st.K[:] = 1.0                       # equal keys: uniform attention, equal added mass
    st.V[0] = np.arange(B * d, dtype=np.float64).reshape(B, d)
    st.score[0] = scores
    st.pos[0] = pos
    st.occ[:] = B
    return st


def _step(st, vic, p=10, r=2):
    q = np.zeros((1, 2)); k = np.ones((1, 2)); v = np.zeros((1, 2))
    return accept_victims(oracle.h2o_decode_step, st, q, k, v, p, r, 1.0, np.array([vic], np.int32))


def test_same_victim_accepted():
    st = _state([1.0, 0.5, 0.5, 2.0], [0, 1, 2, 9])
    after, _, near = _step(st, 1)
    assert near == 0 and after.pos[0].tolist() == [0, 10, 2, 9]
    assert st.pos[0].tolist() == [0, 1, 2, 9]      # the state passed in is left as it was


def test_tied_candidate_followed_and_counted():
    st = _state([1.0, 0.5, 0.5, 2.0], [0, 1, 2, 9])
    after, _, near = _step(st, 2)
    assert near == 1 and after.pos[0].tolist() == [0, 1, 10, 9]


def test_larger_score_rejected():
    st = _state([1.0, 0.5, 0.5, 2.0], [0, 1, 2, 9])
    with pytest.raises(AssertionError, match="not a near tie"):
        _step(st, 0)


def test_victim_inside_window_rejected():
    st = _state([1.0, 0.5, 0.5, 0.1], [0, 1, 2, 9])
    with pytest.raises(AssertionError, match="recent window"):
        _step(st, 3)


def test_append_rejected():
    st = _state([1.0, 0.5, 0.5, 2.0], [0, 1, 2, 9])
    with pytest.raises(AssertionError, match="append"):
        _step(st, -1)


@pytest.mark.parametrize("rel,ok", [(0.5 * NEAR_TIE, True), (2 * NEAR_TIE, False)])
def test_near_tie_threshold(rel, ok):
    # after the step both candidates gain 1/5; the gap is rel of the smaller
    base = 0.5
    st = _state([1.0, base, (base + 0.2) * (1 + rel) - 0.2, 2.0], [0, 1, 2, 9])
    if ok:
        _, _, near = _step(st, 2)
        assert near == 1
    else:
        with pytest.raises(AssertionError, match="not a near tie"):
            _step(st, 2)
