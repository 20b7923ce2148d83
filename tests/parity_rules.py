"""Comparison rules between the CUDA path and the fp64 oracle.

Selection: the selected set must be exactly the oracle's, except for tokens
whose oracle score lies within eps = 1e-4 * max|score| of the cutoff.  In
interval form: with per-token vote bounds counted at theta_h +/- eps and
head-sum bounds sum +/- Hq*eps, no token left out of S may definitely
outrank (lexicographically: vote, sum, then lower index) a token in S.

Attention: max-abs <= 1e-3 and relative L2 <= 1e-3 on the fp32 output,
against the oracle evaluated on the same selected set.
"""

import numpy as np

SELECT_EPS_REL = 1e-4
ATTN_MAX_ABS = 1e-3
ATTN_REL_L2 = 1e-3


def check_selection(S_gpu, sc, theta, c0, K, eps_rel=SELECT_EPS_REL):
    """One sequence.  sc [Hq, |C|] and theta [Hq] are the oracle's (fp64).
    Returns the number of tokens on which GPU and oracle sets differ."""
    S = np.asarray(S_gpu, dtype=np.int64)
    Hq, nc = sc.shape
    assert S.shape == (K,), "|S| = %d, expected K = %d" % (S.shape[0], K)
    if K == 0:
        return 0
    assert np.all(np.diff(S) > 0), "S is not strictly ascending"
    assert S.min() >= c0 and S.max() < c0 + nc, "S has a token outside the candidates"
    eps = eps_rel * np.abs(sc).max()
    vote_lo = (sc > theta[:, None] + eps).sum(0)
    vote_hi = (sc > theta[:, None] - eps).sum(0)
    ssum = sc.sum(0)
    s_lo, s_hi = ssum - Hq * eps, ssum + Hq * eps
    ids = np.arange(nc)
    inS = np.zeros(nc, dtype=bool)
    inS[S - c0] = True
    # worst-case key of each left-out token, best-case key of each chosen one
    out_ids = ids[~inS]
    in_ids = ids[inS]
    if len(out_ids):
        j = out_ids[np.lexsort((out_ids, -s_lo[out_ids], -vote_lo[out_ids]))[0]]   # max L
        i = in_ids[np.lexsort((-in_ids, s_hi[in_ids], vote_hi[in_ids]))[0]]        # min U
        L = (vote_lo[j], s_lo[j], -j)
        U = (vote_hi[i], s_hi[i], -i)
        assert not (L > U), (
            "token %d (vote >= %d, sum >= %.6g) definitely outranks selected token %d (vote <= %d, sum <= %.6g)"
            % (c0 + j, vote_lo[j], s_lo[j], c0 + i, vote_hi[i], s_hi[i]))
    return 0


def selection_difference(S_gpu, S_oracle):
    a = set(np.asarray(S_gpu).tolist())
    b = set(np.asarray(S_oracle).tolist())
    return len(a ^ b)


def check_attention(out_gpu, out_ref, max_abs=ATTN_MAX_ABS, rel_l2=ATTN_REL_L2):
    out_gpu = np.asarray(out_gpu, dtype=np.float64)
    out_ref = np.asarray(out_ref, dtype=np.float64)
    err = out_gpu - out_ref
    ma = np.abs(err).max() if err.size else 0.0
    rl = np.linalg.norm(err) / max(np.linalg.norm(out_ref), 1e-300)
    assert ma <= max_abs, "max-abs error %.3g > %.3g" % (ma, max_abs)
    assert rl <= rel_l2, "relative L2 error %.3g > %.3g" % (rl, rel_l2)
    return ma, rl


def check_topc(S_gpu, p, c, eps_rel=SELECT_EPS_REL):
    """SnapKV selection for one KV head: min(c, n) ascending indices; no index
    left out may definitely outrank (pooled score, then lower index) a kept
    one, with scores known to within eps = 1e-4 * max p."""
    S = np.asarray(S_gpu, dtype=np.int64)
    p = np.asarray(p, dtype=np.float64)
    n = p.shape[0]
    cc = min(c, n)
    assert S.shape == (cc,), "|S| = %d, expected %d" % (S.shape[0], cc)
    assert np.all(np.diff(S) > 0), "S is not strictly ascending"
    assert S.min() >= 0 and S.max() < n
    eps = eps_rel * np.abs(p).max()
    ids = np.arange(n)
    inS = np.zeros(n, dtype=bool)
    inS[S] = True
    out_ids, in_ids = ids[~inS], ids[inS]
    if len(out_ids):
        j = out_ids[np.lexsort((out_ids, -(p[out_ids] - eps)))[0]]
        i = in_ids[np.lexsort((-in_ids, p[in_ids] + eps))[0]]
        assert not ((p[j] - eps, -j) > (p[i] + eps, -i)), (
            "index %d (p >= %.6g) outranks kept index %d (p <= %.6g)" % (j, p[j] - eps, i, p[i] + eps))


def check_topk(S_gpu, key, K, eps, offset=0):
    """Top-K by one scalar key (then lower index) for one row: K strictly
    ascending indices in [offset, offset + len(key)); no index left out may
    definitely outrank a kept one when every key is known to within eps.
    Returns the number of kept indices whose key lies within 2 eps of the
    cutoff (the band where GPU and oracle may legitimately differ)."""
    S = np.asarray(S_gpu, dtype=np.int64) - offset
    key = np.asarray(key, dtype=np.float64)
    n = key.shape[0]
    assert S.shape == (K,), "|S| = %d, expected %d" % (S.shape[0], K)
    assert np.all(np.diff(S) > 0), "S is not strictly ascending"
    assert S.min() >= 0 and S.max() < n, "S has an index outside the candidates"
    ids = np.arange(n)
    inS = np.zeros(n, dtype=bool)
    inS[S] = True
    out_ids, in_ids = ids[~inS], ids[inS]
    if len(out_ids):
        j = out_ids[np.lexsort((out_ids, -(key[out_ids] - eps)))[0]]
        i = in_ids[np.lexsort((-in_ids, key[in_ids] + eps))[0]]
        assert not ((key[j] - eps, -j) > (key[i] + eps, -i)), (
            "index %d (key >= %.6g) outranks kept index %d (key <= %.6g)"
            % (j + offset, key[j] - eps, i + offset, key[i] + eps))
        cut = key[in_ids].min()
        return int((np.abs(key[in_ids] - cut) <= 2 * eps).sum())
    return 0
