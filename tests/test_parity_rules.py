"""The comparison rules that decide GPU parity, checked on the CPU: each
accepts the oracle's own answer and differences inside its band, and
rejects a set or an output that is definitely wrong."""

import numpy as np
import pytest

from oracle import snapkv as osnap
from oracle import tokenselect as ots
from tests.parity_rules import (SELECT_EPS_REL, check_attention, check_selection, check_topc, check_topk)


def _oracle_set(sc, K, c0):
    theta = ots.thresholds(sc, K)
    order = ots.rank_order(ots.votes(sc[None], theta[None])[0], ots.score_sums(sc[None])[0], c0)
    return np.sort(order[:K]), theta, order


def _scores(seed, Hq=4, nc=200):
    return np.random.default_rng(seed).standard_normal((Hq, nc))


@pytest.mark.parametrize("seed", range(5))
def test_selection_rule_accepts_the_oracle_set(seed):
    sc, c0, K = _scores(seed), 4, 30
    S, theta, _ = _oracle_set(sc, K, c0)
    check_selection(S, sc, theta, c0, K)


@pytest.mark.parametrize("seed", range(5))
def test_selection_rule_rejects_a_swap_far_from_the_cutoff(seed):
    sc, c0, K = _scores(seed), 4, 30
    S, theta, order = _oracle_set(sc, K, c0)
    wrong = np.sort(np.concatenate([np.setdiff1d(S, [order[0]]), [order[-1]]]))
    with pytest.raises(AssertionError, match="definitely outranks"):
        check_selection(wrong, sc, theta, c0, K)


def test_selection_rule_accepts_a_swap_inside_the_band():
    # One head: theta is the K-th largest score, so the last selected token
    # and the first left out compare by score alone, and a near-tie planted
    # just below the last selected one leaves the thresholds unchanged.
    sc, c0, K = _scores(11, Hq=1), 4, 30
    S, theta, order = _oracle_set(sc, K, c0)
    last_in, first_out = order[K - 1] - c0, order[K] - c0
    eps = SELECT_EPS_REL * np.abs(sc).max()
    sc[:, first_out] = sc[:, last_in] - 0.1 * eps          # the two differ by far less than eps
    S, theta, order = _oracle_set(sc, K, c0)
    assert order[K] - c0 == first_out                       # still just outside in the oracle
    swapped = np.sort(np.concatenate([np.setdiff1d(S, [c0 + last_in]), [c0 + first_out]]))
    stats = {}
    assert check_selection(swapped, sc, theta, c0, K, stats=stats) == 2     # one token out, one in
    assert stats["ndiff"] == 2 and stats["band"] >= 2
    assert check_selection(S, sc, theta, c0, K) == 0
    sc[:, first_out] = sc[:, last_in] - 50 * eps            # now well separated: the swap is wrong
    S, theta, _ = _oracle_set(sc, K, c0)
    swapped = np.sort(np.concatenate([np.setdiff1d(S, [c0 + last_in]), [c0 + first_out]]))
    with pytest.raises(AssertionError):
        check_selection(swapped, sc, theta, c0, K)


def test_selection_rule_rejects_malformed_sets():
    sc, c0, K = _scores(3), 4, 30
    S, theta, _ = _oracle_set(sc, K, c0)
    with pytest.raises(AssertionError, match=r"\|S\|"):
        check_selection(S[:-1], sc, theta, c0, K)
    with pytest.raises(AssertionError, match="ascending"):
        check_selection(S[::-1], sc, theta, c0, K)
    dup = S.copy()
    dup[1] = dup[0]
    with pytest.raises(AssertionError, match="ascending"):
        check_selection(dup, sc, theta, c0, K)
    outside = S.copy()
    outside[-1] = c0 + sc.shape[1]
    with pytest.raises(AssertionError, match="outside"):
        check_selection(outside, sc, theta, c0, K)


def test_topc_rule_accepts_the_oracle_and_rejects_a_far_swap():
    p = np.random.default_rng(5).random(300)
    S = osnap.top_c(p[None], 40)[0]
    check_topc(S, p, 40)
    order = np.lexsort((np.arange(300), -p))
    wrong = np.sort(np.concatenate([np.setdiff1d(S, [order[0]]), [order[-1]]]))
    with pytest.raises(AssertionError, match="outranks"):
        check_topc(wrong, p, 40)
    check_topc(np.arange(300), p, 500)                     # c >= n: every index, ascending


def test_topc_rule_band():
    p = np.random.default_rng(6).random(300)
    order = np.lexsort((np.arange(300), -p))
    eps = SELECT_EPS_REL * p.max()
    p[order[40]] = p[order[39]] - 0.5 * eps
    S = osnap.top_c(p[None], 40)[0]
    swapped = np.sort(np.concatenate([np.setdiff1d(S, [order[39]]), [order[40]]]))
    check_topc(swapped, p, 40)
    p[order[40]] = p[order[39]] - 10 * eps
    S = osnap.top_c(p[None], 40)[0]
    swapped = np.sort(np.concatenate([np.setdiff1d(S, [order[39]]), [order[40]]]))
    with pytest.raises(AssertionError):
        check_topc(swapped, p, 40)


def test_topk_rule_offset_and_band_count():
    key = np.random.default_rng(7).standard_normal(500)
    order = np.lexsort((np.arange(500), -key))
    S = np.sort(order[:50]) + 4
    assert check_topk(S, key, 50, eps=1e-9, offset=4) == 1   # only the cutoff itself lies in a tiny band
    wrong = np.sort(np.concatenate([np.setdiff1d(S - 4, [order[0]]), [order[-1]]])) + 4
    with pytest.raises(AssertionError, match="outranks"):
        check_topk(wrong, key, 50, eps=1e-9, offset=4)


def test_attention_rule_bounds():
    ref = np.random.default_rng(8).standard_normal((2, 8, 128))
    assert check_attention(ref.astype(np.float32), ref)[0] < 1e-6
    bumped = ref.copy()
    bumped[0, 0, 0] += 2e-3
    with pytest.raises(AssertionError, match="max-abs"):
        check_attention(bumped, ref)
    small = 0.1 * ref                                        # every element 9e-4 off: max-abs passes,
    drift = small + 9e-4 * np.sign(small)                    # relative L2 ~ 9e-3 does not
    with pytest.raises(AssertionError, match="relative L2"):
        check_attention(drift, small)


def test_selection_rule_sum_tolerance_is_relative_to_the_head_sums():
    # Independent heads of mixed sign: max|head sum| is far below Hq * max|score|.
    # At the cutoff two tokens with equal votes compare by their head sums: a
    # swap whose sums differ by less than 1e-4 * max|sum| passes; one whose sums
    # differ by 3 times that fails, though that gap is still below Hq * eps.
    Hq, nc, c0, K = 32, 400, 4, 60
    sc = np.random.default_rng(12).standard_normal((Hq, nc))
    S, theta, order = _oracle_set(sc, K, c0)
    vote = ots.votes(sc[None], theta[None])[0]
    last_in, first_out = order[K - 1] - c0, order[K] - c0
    assert vote[last_in] == vote[first_out]
    eps = SELECT_EPS_REL * np.abs(sc).max()
    for gap, ok in ((0.3, True), (3.0, False)):
        sc2 = sc.copy()
        ssum = sc2.sum(0)
        eps_sum = SELECT_EPS_REL * np.abs(ssum).max()
        assert gap * eps_sum < Hq * eps
        shift = (ssum[last_in] - gap * eps_sum) - ssum[first_out]
        # put the shift on the head where first_out lies farthest from theta_h
        h = int(np.argmax(np.abs(sc2[:, first_out] - theta)))
        assert abs(sc2[h, first_out] - theta[h]) > 4 * abs(shift)
        sc2[h, first_out] += shift
        S2, theta2, order2 = _oracle_set(sc2, K, c0)
        assert np.array_equal(theta2, theta) and np.array_equal(S2, S)
        assert order2[K] - c0 == first_out
        swapped = np.sort(np.concatenate([np.setdiff1d(S2, [c0 + last_in]), [c0 + first_out]]))
        if ok:
            assert check_selection(swapped, sc2, theta2, c0, K) == 2
        else:
            with pytest.raises(AssertionError):
                check_selection(swapped, sc2, theta2, c0, K)
