"""Comparison rules between the CUDA path and the fp64 oracle.

Selection: the selected set must be exactly the oracle's, except for tokens
whose oracle score lies within eps = 1e-4 * max|score| of the cutoff.  In
interval form: with per-token vote bounds counted at theta_h +/- eps and
head-sum bounds sum +/- 1e-4 * max|sum|, no token left out of S may
definitely outrank (lexicographically: vote, sum, then lower index) a token
in S, and every token where the two sets differ must have an interval that
overlaps the cutoff token's.

Attention: max-abs <= 1e-3 and relative L2 <= 1e-3 on the fp32 output,
against the oracle evaluated on the same selected set.
"""

import numpy as np

SELECT_EPS_REL = 1e-4
ATTN_MAX_ABS = 1e-3
ATTN_REL_L2 = 1e-3


def check_selection(S_gpu, sc, theta, c0, K, eps_rel=SELECT_EPS_REL, stats=None):
    """One sequence.  sc [Hq, |C|] and theta [Hq] are the oracle's (fp64).

    Per-head scores are known to within eps = eps_rel * max|score|, so a
    token's vote lies in [#(score > theta + eps), #(score > theta - eps)];
    its head sum is known to within eps_sum = eps_rel * max|head sum| (the
    same relative rule applied to the second ranking key).  Checks that no
    token left out definitely outranks a selected one, and that every token
    on which the GPU and oracle sets differ has a key interval that overlaps
    the cutoff token's (the oracle's K-th ranked candidate).  Returns the
    number of differing tokens; `stats`, when a dict, receives the number of
    candidates whose interval overlaps the cutoff ('band') and the
    tolerances used."""
    S = np.asarray(S_gpu, dtype=np.int64)
    Hq, nc = sc.shape
    assert S.shape == (K,), "|S| = %d, expected K = %d" % (S.shape[0], K)
    if K == 0:
        return 0
    assert np.all(np.diff(S) > 0), "S is not strictly ascending"
    assert S.min() >= c0 and S.max() < c0 + nc, "S has a token outside the candidates"
    eps = eps_rel * np.abs(sc).max()
    vote = (sc > theta[:, None]).sum(0)
    vote_lo = (sc > theta[:, None] + eps).sum(0)
    vote_hi = (sc > theta[:, None] - eps).sum(0)
    ssum = sc.sum(0)
    eps_sum = eps_rel * np.abs(ssum).max()
    s_lo, s_hi = ssum - eps_sum, ssum + eps_sum
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
    # the oracle's own set and its cutoff token (K-th in its order)
    order = np.lexsort((ids, -ssum, -vote))
    or_in = np.zeros(nc, dtype=bool)
    or_in[order[:K]] = True
    cut = order[K - 1]
    cut_lo, cut_hi = (vote_lo[cut], s_lo[cut]), (vote_hi[cut], s_hi[cut])
    # interval of t overlaps the cutoff's: L(t) <= U(cut) and U(t) >= L(cut), lexicographically
    lo_le = (vote_lo < cut_hi[0]) | ((vote_lo == cut_hi[0]) & (s_lo <= cut_hi[1]))
    hi_ge = (vote_hi > cut_lo[0]) | ((vote_hi == cut_lo[0]) & (s_hi >= cut_lo[1]))
    in_band = lo_le & hi_ge
    diff = np.nonzero(inS != or_in)[0]
    far = diff[~in_band[diff]]
    assert far.size == 0, (
        "%d tokens differ from the oracle's set away from the cutoff band, e.g. token %d (vote %d, sum %.6g; "
        "cutoff vote %d, sum %.6g)" % (far.size, c0 + far[0], vote[far[0]], ssum[far[0]], vote[cut], ssum[cut]))
    if stats is not None:
        stats.update(band=int(in_band.sum()), ndiff=int(diff.size), eps=float(eps), eps_sum=float(eps_sum))
    return int(diff.size)


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
