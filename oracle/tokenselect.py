"""TokenSelect decode step as plain fp64 NumPy, one definition per function.

Test infrastructure only (see the package docstring).

Notation follows the TokenSelect page: per query head h, Score_h(i) on the
compressed key index, a per-head threshold theta_h, Vote(i), the top-K set S,
and attention over S plus the always-included sink and local tokens.

Shapes (all arrays are fp64 values; bf16 inputs are widened exactly):
  q      [B, Hq, d]             current query, one row per query head
  K, V   [B, Hkv, n, d]         cache of n tokens (first n rows of the cache)
  W      [Hkv, d, d_idx]        per-KV-head projection to the index space
  index  [B, Hkv, n, d_idx]     compressed key index (values on the bf16 grid)
Query head h reads KV head g(h) = h // (Hq // Hkv): consecutive query heads
share a KV head (the usual grouped-query convention; the pages do not state
the mapping).

Readings taken where the pages leave a step open are stated at each function.
"""

import numpy as np

from .bf16 import round_bf16


# ---------------------------------------------------------------------------
# Token regions.
# TokenSelect, section "Token-Level Selection と Sparse Attention", table of
# always-included tokens: the first `sink` tokens and the last `local` tokens
# are always attended.  Reading: they are outside the budget, so the candidate
# range C that scoring and voting rank is what lies between them.
# ---------------------------------------------------------------------------
def regions(n, sink, local):
    """Return (sink_end, c0, c1, local_start) for a cache of n tokens.

    sink  = [0, sink_end)          sink_end = min(sink, n)
    C     = [c0, c1)               c0 = sink, c1 = n - local (empty if c1 <= c0)
    local = [local_start, n)       local_start = max(n - local, sink_end)
    """
    sink_end = min(sink, n)
    c0 = sink
    c1 = max(n - local, c0)
    local_start = max(n - local, sink_end)
    return sink_end, c0, c1, local_start


def budget_tokens(n, budget_permille, sink, local):
    """K = min(floor(budget * n), |C|), the floor taken in integers.

    Reading: the budget counts selected tokens only (sink and local are
    extra), as a fraction of the whole context n.
    """
    _, c0, c1, _ = regions(n, sink, local)
    return min((budget_permille * n) // 1000, c1 - c0)


# ---------------------------------------------------------------------------
# Compressed key index.
# TokenSelect, section "Query-Key Dot Product Index": K_index in R^{n x d'},
# d' = d/4, built incrementally during inference.  The page does not say how
# the d' summary is formed; reading: a per-KV-head linear projection W_g of
# shape d x d' (TokenButler, section "Kernarchitektur", projects the real keys
# with a matrix into the same low-dimensional space), stored as bf16.
# ---------------------------------------------------------------------------
def index_rows_exact(K, W):
    """fp64 K_g @ W_g for every (b, g): [B, Hkv, t, d_idx]."""
    K = np.asarray(K, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    B, Hkv = K.shape[:2]
    out = np.empty(K.shape[:3] + (W.shape[-1],))
    for b in range(B):
        for g in range(Hkv):
            out[b, g] = K[b, g] @ W[g]
    return out


def index_rows(K, W):
    """The stored index: round-to-nearest-even bf16 of the fp64 product."""
    return round_bf16(index_rows_exact(K, W))


# ---------------------------------------------------------------------------
# Scores.
# TokenSelect, section "Query-Key Dot Product Index", equation Score_h:
#   Score_h(i) = q_h . k_index,h(i) / sqrt(d').
# The equation dots a d-dimensional query with a d'-dimensional index row;
# the page's own scoring routine takes the query already in d' space.
# Reading: q'_h = W_g(h)^T q_h, kept unrounded.
# ---------------------------------------------------------------------------
def query_index(q, W, Hkv):
    """q'_h = W_{g(h)}^T q_h for every (b, h): [B, Hq, d_idx]."""
    q = np.asarray(q, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    B, Hq, _ = q.shape
    group = Hq // Hkv
    g_of_h = np.arange(Hq) // group
    return np.einsum("bhe,hej->bhj", q, W[g_of_h])


def scores(q, W, index, n, sink, local):
    """Score_h(i) for i in C: [B, Hq, |C|] (column t is token c0 + t)."""
    index = np.asarray(index)
    B, Hkv = index.shape[:2]
    d_idx = index.shape[-1]
    _, c0, c1, _ = regions(n, sink, local)
    qp = query_index(q, W, Hkv)
    Hq = qp.shape[1]
    group = Hq // Hkv
    out = np.empty((B, Hq, c1 - c0))
    for b in range(B):
        for g in range(Hkv):
            rows = np.asarray(index[b, g, c0:c1, :], dtype=np.float64)      # [|C|, d']
            heads = slice(g * group, (g + 1) * group)
            out[b, heads] = (rows @ qp[b, heads].T).T / np.sqrt(d_idx)
    return out


# ---------------------------------------------------------------------------
# Threshold and vote.
# TokenSelect, section "Voting Mechanism": a head-specific threshold theta_h
# and Vote(i) = sum_h 1[Score_h(i) > theta_h] (strict).  The page does not
# define theta_h; reading: theta_h is head h's K-th largest score over C, so
# every head nominates (up to ties) its own top K-1.
# ---------------------------------------------------------------------------
def thresholds(sc, K):
    """theta_h = K-th largest of Score_h over C: [B, Hq]."""
    if K < 1:
        raise ValueError("thresholds need K >= 1")
    return -np.sort(-sc, axis=-1)[..., K - 1]


def votes(sc, theta):
    """Vote(i) = number of heads whose score is strictly above theta_h."""
    return (sc > theta[..., None]).sum(axis=1)


def score_sums(sc):
    """Sum over all query heads of Score_h(i): the second ranking key."""
    return sc.sum(axis=1)


# ---------------------------------------------------------------------------
# Selection.
# TokenSelect, section "Token-Level Selection と Sparse Attention", equation S:
#   S = top-K({i : Vote(i) >= V_min}).
# Readings: one S per sequence and layer, shared by all heads (the equation
# aggregates heads; the page's own selection routine sums votes over heads and
# returns one sorted [batch, k] set).  Ranking is Vote descending, then the
# head-summed score descending, then token index ascending.  When fewer than K
# tokens reach V_min the set is filled from the same order; since Vote leads
# the order, every token with Vote >= V_min ranks ahead of every token below
# it, so the filter only decides which tokens are fill.  S is returned sorted
# ascending.
# ---------------------------------------------------------------------------
def rank_order(vote, ssum, c0):
    """Candidate token ids of one sequence, best first."""
    ids = c0 + np.arange(vote.shape[0])
    # np.lexsort sorts by the last key first.
    return ids[np.lexsort((ids, -ssum, -vote))]


def select(q, W, index, n, K, sink, local, vmin=1):
    """The selected set S (ascending, int64 [B, K]) and the intermediates."""
    if vmin < 1:
        raise ValueError("V_min must be >= 1")
    _, c0, c1, _ = regions(n, sink, local)
    if not 0 <= K <= c1 - c0:
        raise ValueError("K must lie in [0, |C|]")
    sc = scores(q, W, index, n, sink, local)
    B = sc.shape[0]
    if K == 0:
        empty = np.zeros((B, 0), dtype=np.int64)
        return empty, dict(scores=sc, theta=None, vote=None, ssum=None, c0=c0)
    theta = thresholds(sc, K)
    vote = votes(sc, theta)
    ssum = score_sums(sc)
    S = np.stack([np.sort(rank_order(vote[b], ssum[b], c0)[:K]) for b in range(B)])
    return S.astype(np.int64), dict(scores=sc, theta=theta, vote=vote, ssum=ssum, c0=c0)


def select_by_rank_count(vote, ssum, c0, K):
    """Second restatement for small |C|: token i is selected iff fewer than K
    candidates outrank it (pairwise comparison, no sorting).  One sequence."""
    m = vote.shape[0]
    ids = c0 + np.arange(m)
    v_i, v_j = vote[:, None], vote[None, :]
    s_i, s_j = ssum[:, None], ssum[None, :]
    i_i, i_j = ids[:, None], ids[None, :]
    j_beats_i = (v_j > v_i) | ((v_j == v_i) & (s_j > s_i)) | (
        (v_j == v_i) & (s_j == s_i) & (i_j < i_i))
    rank = j_beats_i.sum(axis=1)
    return ids[rank < K]


# ---------------------------------------------------------------------------
# Selection without voting, one set per KV head.
# TokenSelect, ablation table (アブレーション): "w/o Voting" replaces the vote
# by an independent selection per head.  Reading for grouped-query attention:
# KV head g ranks the candidates by the sum of its query heads' scores (its
# own score when the group has one head), ties to the lower token index, and
# keeps the first K, emitted ascending; every query head of the group then
# attends to sink + S_g + local.
# ---------------------------------------------------------------------------
def group_scores(sc, Hkv):
    """Sum of Score_h over the query heads of each KV group: [B, Hkv, |C|]."""
    B, Hq, nc = sc.shape
    return sc.reshape(B, Hkv, Hq // Hkv, nc).sum(axis=2)


def select_per_kv_head(q, W, index, n, K, sink, local):
    """S [B, Hkv, K] (ascending per KV head) and the intermediates."""
    _, c0, c1, _ = regions(n, sink, local)
    if not 0 <= K <= c1 - c0:
        raise ValueError("K must lie in [0, |C|]")
    sc = scores(q, W, index, n, sink, local)
    Hkv = np.asarray(index).shape[1]
    gs = group_scores(sc, Hkv)
    B = sc.shape[0]
    ids = c0 + np.arange(c1 - c0)
    S = np.zeros((B, Hkv, K), dtype=np.int64)
    for b in range(B):
        for g in range(Hkv):
            # best first: larger group score, then lower index
            S[b, g] = np.sort(ids[np.lexsort((ids, -gs[b, g]))][:K])
    return S, dict(scores=sc, gsum=gs, c0=c0)


def sparse_attention_per_head(q, K, V, S, n, sink, local):
    """Attention of each query head over sink + S[b, g(h)] + local: output
    [B, Hq, d] and natural-log LSE [B, Hq]; S is [B, Hkv, K]."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    B, Hq, d = q.shape
    Hkv = K.shape[1]
    group = Hq // Hkv
    out = np.zeros((B, Hq, d))
    lse = np.zeros((B, Hq))
    for b in range(B):
        for h in range(Hq):
            g = h // group
            T = attended_tokens(S[b, g], n, sink, local)
            z = K[b, g, T, :] @ q[b, h] / np.sqrt(d)
            m = z.max()
            p = np.exp(z - m)
            out[b, h] = p @ V[b, g, T, :] / p.sum()
            lse[b, h] = m + np.log(p.sum())
    return out, lse


# ---------------------------------------------------------------------------
# Neighbour expansion of a selected set.
# TokenButler, section "Optimierungen": selected tokens are expanded to their
# spatial neighbours (the prediction interval reuses a selection over several
# steps); SnapKV, section "Top-k Selection と Cluster-based Retention":
# S_final is the union over the selected j of {j - k, ..., j + k}.  Reading
# for the decode step: the union is clipped to the candidates C, since the
# sink and local tokens are attended anyway, and emitted ascending; its size
# varies per set.
# ---------------------------------------------------------------------------
def expand_neighbors(S_row, radius, n, sink, local):
    """Ascending union of [j - radius, j + radius] over j in S_row, within C."""
    _, c0, c1, _ = regions(n, sink, local)
    out = set()
    for j in np.asarray(S_row, dtype=np.int64).tolist():
        out.update(range(max(c0, j - radius), min(c1, j + radius + 1)))
    return np.array(sorted(out), dtype=np.int64)


# ---------------------------------------------------------------------------
# Attention over the selected set.
# TokenSelect, section "Token-Level Selection と Sparse Attention", equation
# Attention: softmax(Q K_S^T / sqrt(d)) V_S, with the sink and local tokens
# always included; section "統合の5ステップ" step 5 merges the sparse and the
# local attention outputs.  Reading: the merge is the log-sum-exp combination,
# which equals one softmax over the disjoint union T = sink u S u local; this
# function computes that single softmax directly.
# ---------------------------------------------------------------------------
def attended_tokens(S_row, n, sink, local):
    """T = sink u S u local for one sequence, ascending."""
    sink_end, _, _, local_start = regions(n, sink, local)
    return np.concatenate([np.arange(sink_end), np.asarray(S_row, dtype=np.int64),
                           np.arange(local_start, n)])


def sparse_attention(q, K, V, S, n, sink, local):
    """Output [B, Hq, d] and natural-log LSE [B, Hq] of attention over T."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    B, Hq, d = q.shape
    Hkv = K.shape[1]
    group = Hq // Hkv
    out = np.zeros((B, Hq, d))
    lse = np.zeros((B, Hq))
    for b in range(B):
        T = attended_tokens(S[b], n, sink, local)
        for h in range(Hq):
            g = h // group
            z = K[b, g, T, :] @ q[b, h] / np.sqrt(d)
            m = z.max()
            p = np.exp(z - m)
            out[b, h] = p @ V[b, g, T, :] / p.sum()
            lse[b, h] = m + np.log(p.sum())
    return out, lse


def dense_attention(q, K, V, n):
    """Plain attention of q over all n cached tokens (the 100 % budget case)."""
    q = np.asarray(q, dtype=np.float64)
    B, Hq, d = q.shape
    empty = np.zeros((B, 0), dtype=np.int64)
    return sparse_attention(q, K, V, empty, n, sink=n, local=0)
