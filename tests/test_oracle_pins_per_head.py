"""Pins for the oracle's per-KV-head selection (TokenSelect without voting)
and its attention.  CPU only.

What fixes them, other than the oracle itself: a library argsort in the case
of one query head per group, brute-force enumeration of K-subsets, a
hand-worked case where a sum and a maximum over the group rank differently,
the grouped-query head mapping, agreement with the voting selection when
there is a single head, and the shared-set attention when every KV head is
given the same set.
"""

import itertools
import math

import numpy as np
import pytest

from oracle import bf16 as obf
from oracle import tokenselect as ots

D, DI = 128, 32


def _case(rng, B, Hq, Hkv, n, dup=False):
    q = obf.round_bf16(rng.standard_normal((B, Hq, D)))
    Kc = obf.round_bf16(rng.standard_normal((B, Hkv, n, D)))
    if dup:                      # exact duplicates force ties in every head
        Kc[:, :, 5] = Kc[:, :, 3]
        Kc[:, :, 6] = Kc[:, :, 3]
    V = obf.round_bf16(rng.standard_normal((B, Hkv, n, D)))
    W = obf.round_bf16(rng.standard_normal((Hkv, D, DI)) / math.sqrt(D))
    return q, Kc, V, W, ots.index_rows(Kc, W)


@pytest.mark.parametrize("seed", range(4))
def test_one_head_per_group_is_plain_topk_per_head(seed):
    rng = np.random.default_rng(700 + seed)
    n, sink, local, H = 200, 4, 16, 3
    q, Kc, V, W, idx = _case(rng, 2, H, H, n, dup=True)
    _, c0, c1, _ = ots.regions(n, sink, local)
    sc = ots.scores(q, W, idx, n, sink, local)
    for K in (1, 5, 60, c1 - c0):
        S, _ = ots.select_per_kv_head(q, W, idx, n, K, sink, local)
        assert S.shape == (2, H, K)
        for b in range(2):
            for g in range(H):
                want = np.sort(np.argsort(-sc[b, g], kind="stable")[:K] + c0)
                assert np.array_equal(S[b, g], want)


@pytest.mark.parametrize("seed", range(6))
def test_per_head_set_is_the_unique_dominating_subset(seed):
    rng = np.random.default_rng(800 + seed)
    n, sink, local, Hkv, Gq = int(rng.integers(8, 15)), 1, 2, 2, 2
    q, Kc, V, W, idx = _case(rng, 1, Hkv * Gq, Hkv, n, dup=seed % 2 == 0)
    _, c0, c1, _ = ots.regions(n, sink, local)
    cand = list(range(c0, c1))
    sc = ots.scores(q, W, idx, n, sink, local)[0]
    for K in range(1, len(cand) + 1):
        S, _ = ots.select_per_kv_head(q, W, idx, n, K, sink, local)
        for g in range(Hkv):
            key = {i: sum(sc[h, i - c0] for h in range(g * Gq, (g + 1) * Gq)) for i in cand}
            winners = [sorted(sub) for sub in itertools.combinations(cand, K)
                       if all((key[a], -a) > (key[x], -x) for a in sub for x in cand if x not in sub)]
            assert len(winners) == 1
            assert S[0, g].tolist() == winners[0]


def _two_head_case():
    """One KV head, two query heads reading index columns 0 and 1.  Token 2
    scores (1, 1) on the two heads, token 3 scores (1.5, 0): the group sum
    ranks token 2 first (2 > 1.5), a maximum would rank token 3 first."""
    n, sink, local = 6, 1, 1
    W = np.zeros((1, D, DI))
    W[0, 0, 0] = 1.0
    W[0, 4, 1] = 1.0
    Kc = np.zeros((1, 1, n, D))
    Kc[0, 0, 2, 0], Kc[0, 0, 2, 4] = 1.0, 1.0
    Kc[0, 0, 3, 0] = 1.5
    Kc[0, 0, 1, 0] = Kc[0, 0, 4, 0] = -1.0
    q = np.zeros((1, 2, D))
    q[0, 0, 0] = 1.0
    q[0, 1, 4] = 1.0
    return q, W, ots.index_rows(Kc, W), n, sink, local


def test_group_sum_hand_worked_case():
    q, W, idx, n, sink, local = _two_head_case()
    S1, info = ots.select_per_kv_head(q, W, idx, n, 1, sink, local)
    assert S1.tolist() == [[[2]]]
    s = 1.0 / math.sqrt(DI)
    assert np.allclose(info["gsum"][0, 0], [-s, 2 * s, 1.5 * s, -s])
    S2, _ = ots.select_per_kv_head(q, W, idx, n, 2, sink, local)
    assert S2.tolist() == [[[2, 3]]]


def test_gqa_groups_are_consecutive_heads():
    # Only query head 6 (group 1 at Gq = 4; an interleaved mapping would put
    # it in group 0) sees a non-zero score: group 0 ranks all candidates
    # equal (lowest indices win), group 1 by head 6.
    n, sink, local, Hq, Hkv = 40, 2, 4, 8, 2
    Kc = np.zeros((1, Hkv, n, D))
    Kc[0, 1, :, 0] = -np.arange(n) / 8.0          # later tokens score lower...
    Kc[0, 1, 30, 0] = 3.0                          # ...except token 30
    W = np.zeros((Hkv, D, DI))
    W[:, 0, 0] = 1.0
    q = np.zeros((1, Hq, D))
    q[0, 6, 0] = 1.0
    idx = ots.index_rows(Kc, W)
    S, _ = ots.select_per_kv_head(q, W, idx, n, 3, sink, local)
    assert S[0, 0].tolist() == [2, 3, 4]
    assert S[0, 1].tolist() == [2, 3, 30]


def test_single_head_agrees_with_voting_selection():
    rng = np.random.default_rng(11)
    n, sink, local = 500, 4, 32
    q, Kc, V, W, idx = _case(rng, 2, 1, 1, n, dup=True)
    _, c0, c1, _ = ots.regions(n, sink, local)
    for K in (1, 2, 50, c1 - c0):
        S_head, _ = ots.select_per_kv_head(q, W, idx, n, K, sink, local)
        S_vote, _ = ots.select(q, W, idx, n, K, sink, local)
        assert np.array_equal(S_head[:, 0], S_vote)


def test_shared_sets_give_the_shared_attention():
    rng = np.random.default_rng(12)
    B, Hq, Hkv, n, sink, local = 2, 8, 2, 300, 4, 32
    q, Kc, V, W, idx = _case(rng, B, Hq, Hkv, n)
    S, _ = ots.select(q, W, idx, n, 40, sink, local)
    S_rep = np.repeat(S[:, None, :], Hkv, axis=1)
    o1, l1 = ots.sparse_attention(q, Kc, V, S, n, sink, local)
    o2, l2 = ots.sparse_attention_per_head(q, Kc, V, S_rep, n, sink, local)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_per_head_attention_uses_each_groups_own_set():
    # Group 1's set holds a dominant key; group 0's does not: only group 1's
    # heads return that key's value.
    n, sink, local, Hq, Hkv = 64, 2, 2, 4, 2
    rng = np.random.default_rng(13)
    q = np.zeros((1, Hq, D))
    q[0, :, 0] = 1.0
    Kc = np.zeros((1, Hkv, n, D))
    V = rng.standard_normal((1, Hkv, n, D))
    Kc[0, :, 20, 0] = 2000.0         # dominant key at token 20 in both KV heads
    S = np.array([[[5, 6], [20, 21]]])
    out, _ = ots.sparse_attention_per_head(q, Kc, V, S, n, sink, local)
    assert np.allclose(out[0, 2], V[0, 1, 20]) and np.allclose(out[0, 3], V[0, 1, 20])
    assert not np.allclose(out[0, 0], V[0, 0, 20])


# ------------------------------------------------------ planted mistakes
def test_planted_group_maximum_is_caught(monkeypatch):
    monkeypatch.setattr(ots, "group_scores",
                        lambda sc, Hkv: sc.reshape(sc.shape[0], Hkv, -1, sc.shape[-1]).max(axis=2))
    with pytest.raises(AssertionError):
        test_group_sum_hand_worked_case()


def test_planted_interleaved_groups_are_caught(monkeypatch):
    def interleaved(sc, Hkv):
        B, Hq, nc = sc.shape
        return sc.reshape(B, Hq // Hkv, Hkv, nc).sum(axis=1)
    monkeypatch.setattr(ots, "group_scores", interleaved)
    with pytest.raises(AssertionError):
        test_gqa_groups_are_consecutive_heads()


def test_planted_descending_tiebreak_is_caught(monkeypatch):
    real = ots.select_per_kv_head

    def desc_ties(q, W, index, n, K, sink, local):
        S, info = real(q, W, index, n, K, sink, local)
        gs, c0 = info["gsum"], info["c0"]
        ids = c0 + np.arange(gs.shape[-1])
        for b in range(S.shape[0]):
            for g in range(S.shape[1]):
                S[b, g] = np.sort(ids[np.lexsort((-ids, -gs[b, g]))][:K])
        return S, info
    monkeypatch.setattr(ots, "select_per_kv_head", desc_ties)
    with pytest.raises(AssertionError):
        test_gqa_groups_are_consecutive_heads()
