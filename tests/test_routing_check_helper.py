"""The layer tests' routing check (helpers.check_routing_within_tie_band),
pinned on the CPU: it accepts every expert set that some logits within the
device's error of the oracle's would select, and rejects a set that drops a
clearly chosen expert, takes one from below the band, repeats an expert, or
carries wrong or misordered weights."""

import numpy as np
import pytest

import oracle
from tests import helpers

K = 2
# token 0: a clear top-2 (experts 3, 1); token 1: experts 0 and 2 tie at
# 2.0 for the second place behind expert 4 (either is valid)
LOGITS = np.array([[0.0, 2.0, -1.0, 3.0, -2.0],
                   [2.0, -1.0, 2.0, 0.5, 4.0]])
BAND = 1e-3


def _weights(idx):
    w = np.empty(idx.shape)
    for t in range(idx.shape[0]):
        z = LOGITS[t, idx[t]]
        e = np.exp(z - z.max())
        w[t] = e / e.sum()
    return w


def _check(idx):
    idx = np.asarray(idx)
    helpers.check_routing_within_tie_band(LOGITS, K, idx, _weights(idx), BAND)


def test_the_oracles_choice_passes():
    idx, w = oracle.topk_renorm(LOGITS, K)
    helpers.check_routing_within_tie_band(LOGITS, K, idx, w, BAND)


def test_either_side_of_a_tie_passes():
    _check([[3, 1], [4, 0]])
    _check([[3, 1], [4, 2]])


@pytest.mark.parametrize("idx", [
    [[3, 0], [4, 0]],   # drops expert 1, clearly in token 0's top 2
    [[3, 2], [4, 0]],   # takes expert 2, below token 0's band
    [[3, 3], [4, 0]],   # repeats an expert
    [[3, 1], [0, 2]],   # drops expert 4
])
def test_invalid_sets_fail(idx):
    with pytest.raises(AssertionError):
        _check(idx)


def test_wrong_or_misordered_weights_fail():
    idx = np.array([[3, 1], [4, 0]])
    w = _weights(idx)
    bad = w.copy()
    bad[0] = [0.5, 0.5]
    with pytest.raises(AssertionError):
        helpers.check_routing_within_tie_band(LOGITS, K, idx, bad, BAND)
    with pytest.raises(AssertionError):  # slots must be in descending weight
        helpers.check_routing_within_tie_band(LOGITS, K, idx[:, ::-1], w[:, ::-1], BAND)


def test_near_tie_inside_the_band_passes_and_outside_fails():
    lg = np.array([[1.0, 1.0 + 5e-4, 0.0]])  # experts 0 and 1 within the band
    for idx in ([[1]], [[0]]):
        helpers.check_routing_within_tie_band(lg, 1, np.array(idx), np.ones((1, 1)), BAND)
    lg2 = np.array([[1.0, 1.0 + 5e-3, 0.0]])  # now expert 1 is clearly first
    with pytest.raises(AssertionError):
        helpers.check_routing_within_tie_band(lg2, 1, np.array([[0]]), np.ones((1, 1)), BAND)
