"""Pins for the oracle's neighbour expansion of a selected set.  CPU only.

What fixes it, other than the oracle itself: a hand-worked example, the
identity at radius 0, an independent construction by library convolution of
the set's indicator vector, and the bounds of the candidate range.
"""

import numpy as np
import pytest

from oracle import tokenselect as ots


def test_hand_worked_example():
    # n = 40, sink 4, local 8: C = [4, 32)
    got = ots.expand_neighbors([5, 10, 12, 30], 1, 40, 4, 8)
    assert got.tolist() == [4, 5, 6, 9, 10, 11, 12, 13, 29, 30, 31]
    got2 = ots.expand_neighbors([5, 30], 3, 40, 4, 8)
    assert got2.tolist() == [4, 5, 6, 7, 8, 27, 28, 29, 30, 31]


def test_radius_zero_is_identity():
    rng = np.random.default_rng(1)
    S = np.sort(rng.choice(np.arange(4, 900), 120, replace=False))
    assert np.array_equal(ots.expand_neighbors(S, 0, 1000, 4, 100), S)


@pytest.mark.parametrize("radius", [1, 2, 5, 17])
def test_matches_indicator_convolution(radius):
    rng = np.random.default_rng(radius)
    n, sink, local = 3000, 4, 256
    _, c0, c1, _ = ots.regions(n, sink, local)
    S = np.sort(rng.choice(np.arange(c0, c1), 300, replace=False))
    ind = np.zeros(n)
    ind[S] = 1.0
    near = np.convolve(ind, np.ones(2 * radius + 1), mode="same") > 0.5
    near[:c0] = False
    near[c1:] = False
    want = np.nonzero(near)[0]
    got = ots.expand_neighbors(S, radius, n, sink, local)
    assert np.array_equal(got, want)
    assert len(got) <= (2 * radius + 1) * len(S)
    assert set(S.tolist()) <= set(got.tolist())


def test_expansion_never_leaves_the_candidates():
    n, sink, local = 300, 4, 32
    _, c0, c1, _ = ots.regions(n, sink, local)
    got = ots.expand_neighbors([c0, c1 - 1], 10, n, sink, local)
    assert got.min() == c0 and got.max() == c1 - 1
    assert got.tolist() == list(range(c0, c0 + 11)) + list(range(c1 - 11, c1))


def test_planted_half_open_radius_is_caught(monkeypatch):
    def short(S_row, radius, n, sink, local):
        _, c0, c1, _ = ots.regions(n, sink, local)
        out = set()
        for j in np.asarray(S_row).tolist():
            out.update(range(max(c0, j - radius), min(c1, j + radius)))   # drops j + radius
        return np.array(sorted(out), dtype=np.int64)
    monkeypatch.setattr(ots, "expand_neighbors", short)
    with pytest.raises(AssertionError):
        test_hand_worked_example()


def test_planted_unclipped_expansion_is_caught(monkeypatch):
    def unclipped(S_row, radius, n, sink, local):
        out = set()
        for j in np.asarray(S_row).tolist():
            out.update(range(max(0, j - radius), min(n, j + radius + 1)))
        return np.array(sorted(out), dtype=np.int64)
    monkeypatch.setattr(ots, "expand_neighbors", unclipped)
    with pytest.raises(AssertionError):
        test_expansion_never_leaves_the_candidates()
