"""Pins for the oracle's paged pool and circular local buffer.  CPU only.

What fixes them, other than the oracle itself: hand-worked page and ring
examples whose stored values are the token numbers, an independent
construction of the pool from a contiguous cache by library reshapes, the
invariance under a permutation of the pool's pages, and the round trip of a
ring flush; a swapped page/offset, a shifted ring slot and a flush that
forgets the index are each caught.
"""

import math

import numpy as np
import pytest

from oracle import bf16 as obf
from oracle import paged as opg
from oracle import tokenselect as ots

D, DI = 128, 32


def _token_pool(block_table, P, num_pages, Hkv=1):
    """A pool whose every row stores its own token number (then b * 1000)."""
    pool = np.full((num_pages, Hkv, P, 1), -1.0)
    for b, row in enumerate(block_table):
        for p, page in enumerate(row):
            for r in range(P):
                pool[page, :, r, 0] = 1000 * b + p * P + r
    return pool


def test_hand_worked_pages():
    # P = 2, three pages: tokens 0-1 in pool page 2, 2-3 in page 0, 4-5 in page 1
    pool = np.zeros((3, 1, 2, 1))
    pool[2, 0, :, 0] = [0, 1]
    pool[0, 0, :, 0] = [2, 3]
    pool[1, 0, :, 0] = [4, 5]
    got = opg.logical_rows(pool, [[2, 0, 1]], 2, 6)
    assert got[0, 0, :, 0].tolist() == [0, 1, 2, 3, 4, 5]
    assert opg.page_of([[2, 0, 1]], 2, 0, 3) == (0, 1)
    # n need not fill the last page
    assert opg.logical_rows(pool, [[2, 0, 1]], 2, 5)[0, 0, :, 0].tolist() == [0, 1, 2, 3, 4]


def test_two_sequences_share_a_pool():
    bt = [[3, 0], [1, 2]]
    pool = _token_pool(bt, 4, 4)
    got = opg.logical_rows(pool, bt, 4, 7)
    assert got[0, 0, :, 0].tolist() == list(range(7))
    assert got[1, 0, :, 0].tolist() == [1000 + t for t in range(7)]


def _pool_from_cache(cache, P):
    """Pages cut from a contiguous [B, Hkv, n_cap, w] cache by reshapes:
    pool page b * pps + p holds tokens [p P, (p + 1) P) of sequence b."""
    B, Hkv, n_cap, w = cache.shape
    pps = n_cap // P
    pool = cache.reshape(B, Hkv, pps, P, w).transpose(0, 2, 1, 3, 4).reshape(B * pps, Hkv, P, w)
    table = np.arange(B * pps).reshape(B, pps)
    return pool, table


@pytest.mark.parametrize("P,n", [(4, 37), (8, 64), (16, 17)])
def test_pool_cut_from_a_contiguous_cache(P, n):
    rng = np.random.default_rng(P + n)
    cache = rng.standard_normal((2, 3, 64, 5))
    pool, table = _pool_from_cache(cache, P)
    assert np.array_equal(opg.logical_rows(pool, table, P, n), cache[:, :, :n])
    # moving the pages around the pool (and the table with them) changes nothing
    perm = rng.permutation(pool.shape[0])
    pool2 = np.empty_like(pool)
    pool2[perm] = pool
    assert np.array_equal(opg.logical_rows(pool2, perm[table], P, n), cache[:, :, :n])


def test_hand_worked_ring():
    # R = 5 slots, tokens 0..11 written in order: slot t mod 5 keeps the last
    ring = np.full((1, 1, 5, 1), -1.0)
    for t in range(12):
        ring[0, 0, opg.ring_slot(t, 5), 0] = t
    assert ring[0, 0, :, 0].tolist() == [10, 11, 7, 8, 9]
    main = np.full((1, 1, 12, 1), -2.0)           # the main cache does not hold tokens 8..11
    main[0, 0, :8, 0] = np.arange(8)
    got = opg.attended_rows(main, ring, 5, 12, 0, 4)
    assert got[0, 0, :, 0].tolist() == list(range(12))


def test_ring_local_window_meets_the_sink():
    # n <= sink + local: the local window starts at the end of the sink
    ring = np.zeros((1, 1, 8, 1))
    for t in range(6):
        ring[0, 0, t % 8, 0] = 100 + t
    main = np.zeros((1, 1, 6, 1))
    main[0, 0, :2, 0] = [0, 1]
    got = opg.attended_rows(main, ring, 8, 6, 2, 256)
    assert got[0, 0, :, 0].tolist() == [0, 1, 102, 103, 104, 105]


def _flush_case(seed):
    rng = np.random.default_rng(seed)
    B, Hkv, P, pps, R = 2, 2, 4, 5, 7
    num_pages = B * pps + 2
    bt = rng.permutation(num_pages)[:B * pps].reshape(B, pps)
    K = obf.round_bf16(rng.standard_normal((B, Hkv, P * pps, D)))
    V = obf.round_bf16(rng.standard_normal((B, Hkv, P * pps, D)))
    W = obf.round_bf16(rng.standard_normal((Hkv, D, DI)) / math.sqrt(D))
    return rng, B, Hkv, P, R, num_pages, bt, K, V, W


@pytest.mark.parametrize("start,count", [(0, 7), (5, 3), (13, 7)])
def test_ring_flush_round_trip(start, count):
    rng, B, Hkv, P, R, num_pages, bt, K, V, W = _flush_case(start)
    ring_K = np.zeros((B, Hkv, R, D))
    ring_V = np.zeros((B, Hkv, R, D))
    for t in range(start, start + count):          # the newest R tokens are in the ring
        ring_K[:, :, t % R] = K[:, :, t]
        ring_V[:, :, t % R] = V[:, :, t]
    pK = rng.standard_normal((num_pages, Hkv, P, D))
    pV = rng.standard_normal((num_pages, Hkv, P, D))
    pI = rng.standard_normal((num_pages, Hkv, P, DI))
    K2, V2, I2 = opg.ring_flush(pK, pV, pI, bt, P, ring_K, ring_V, R, W, start, count)
    sl = slice(start, start + count)
    assert np.array_equal(opg.logical_rows(K2, bt, P, start + count)[:, :, sl], K[:, :, sl])
    assert np.array_equal(opg.logical_rows(V2, bt, P, start + count)[:, :, sl], V[:, :, sl])
    assert np.array_equal(opg.logical_rows(I2, bt, P, start + count)[:, :, sl], ots.index_rows(K[:, :, sl], W))
    # every other row is untouched
    written = np.zeros(pK.shape[:3], dtype=bool)
    for b in range(B):
        for t in range(start, start + count):
            page, r = opg.page_of(bt, P, b, t)
            written[page, :, r] = True
    assert np.array_equal(K2[~written], pK[~written]) and np.array_equal(I2[~written], pI[~written])


def test_attention_over_pages_and_ring_equals_the_contiguous_cache():
    rng = np.random.default_rng(21)
    B, Hq, Hkv, n, P, R, sink, local = 2, 4, 2, 50, 8, 16, 4, 12
    K = obf.round_bf16(rng.standard_normal((B, Hkv, 56, D)))
    V = obf.round_bf16(rng.standard_normal((B, Hkv, 56, D)))
    q = obf.round_bf16(rng.standard_normal((B, Hq, D)))
    pK, table = _pool_from_cache(K, P)
    pV, _ = _pool_from_cache(V, P)
    ring_K = np.zeros((B, Hkv, R, D))
    ring_V = np.zeros((B, Hkv, R, D))
    for t in range(n - R, n):
        ring_K[:, :, t % R] = K[:, :, t]
        ring_V[:, :, t % R] = V[:, :, t]
    S = np.sort(np.stack([rng.choice(np.arange(sink, n - local), 9, replace=False) for _ in range(B)]), axis=1)
    Kv = opg.attended_rows(opg.logical_rows(pK, table, P, n), ring_K, R, n, sink, local)
    Vv = opg.attended_rows(opg.logical_rows(pV, table, P, n), ring_V, R, n, sink, local)
    got, got_lse = ots.sparse_attention(q, Kv, Vv, S, n, sink, local)
    want, want_lse = ots.sparse_attention(q, K[:, :, :n], V[:, :, :n], S, n, sink, local)
    assert np.array_equal(got, want) and np.array_equal(got_lse, want_lse)


# ------------------------------------------------------ planted mistakes
def test_planted_swapped_page_and_offset_is_caught(monkeypatch):
    monkeypatch.setattr(opg, "page_of", lambda bt, P, b, t: (int(bt[b][t % P]), t // P))
    with pytest.raises((AssertionError, IndexError)):
        test_hand_worked_pages()


def test_planted_shifted_ring_slot_is_caught(monkeypatch):
    monkeypatch.setattr(opg, "ring_slot", lambda t, R: (t + 1) % R)
    real = opg.attended_rows

    def check():
        ring = np.full((1, 1, 5, 1), -1.0)
        for t in range(12):
            ring[0, 0, t % 5, 0] = t            # written by the true rule
        main = np.zeros((1, 1, 12, 1))
        main[0, 0, :8, 0] = np.arange(8)
        assert real(main, ring, 5, 12, 0, 4)[0, 0, :, 0].tolist() == list(range(12))
    with pytest.raises(AssertionError):
        check()


def test_planted_flush_without_index_is_caught(monkeypatch):
    real = opg.ring_flush

    def no_index(pool_K, pool_V, pool_index, *args):
        K2, V2, _ = real(pool_K, pool_V, pool_index, *args)
        return K2, V2, np.array(pool_index, dtype=np.float64)
    monkeypatch.setattr(opg, "ring_flush", no_index)
    with pytest.raises(AssertionError):
        test_ring_flush_round_trip(5, 3)
