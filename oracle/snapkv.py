"""SnapKV prefill compaction as plain fp64 NumPy.

Test infrastructure only (see the package docstring).

Shapes: q_obs [B, Hq, w, d] (the last w query rows of the prompt),
K, V [B, Hkv, n, d]; query head h reads KV head g(h) = h // (Hq // Hkv).
"""

import numpy as np


def window_attention(q_obs, K, n):
    """A = softmax(Q_obs K^T / sqrt(d_k)) per query head: [B, Hq, w, n].

    SnapKV, section "Attention Score計算とPooling", equation A.  The page's
    code applies no causal mask, so every window row attends to all n prompt
    tokens (reading kept here).
    """
    q = np.asarray(q_obs, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)[:, :, :n, :]
    B, Hq, w, d = q.shape
    Hkv = K.shape[1]
    g_of_h = np.arange(Hq) // (Hq // Hkv)
    x = np.einsum("bhrd,bhjd->bhrj", q, K[:, g_of_h]) / np.sqrt(d)
    x = x - x.max(axis=-1, keepdims=True)
    e = np.exp(x)
    return e / e.sum(axis=-1, keepdims=True)


def window_mean(q_obs, K, n):
    """Importance a_j per KV head: [B, Hkv, n].

    SnapKV, equation a-bar: the mean over the w window rows of A.  The page
    leaves grouped-query attention open; reading: the mean is also taken over
    the Gq query heads that share KV head g, i.e. over all Gq*w rows.
    """
    A = window_attention(q_obs, K, n)
    B, Hq, w, _ = A.shape
    Hkv = np.asarray(K).shape[1]
    group = Hq // Hkv
    return A.reshape(B, Hkv, group * w, n).mean(axis=2)


def pool(a, kernel=3):
    """1-D average pool, stride 1, zero padding kernel//2, divisor `kernel`.

    SnapKV, section "アルゴリズム", step 3 (average pooling with padding
    kernel_size // 2 and stride 1).  Reading: padded zeros count in the
    divisor at the edges (PyTorch's documented default for that call).
    """
    a = np.asarray(a, dtype=np.float64)
    if kernel % 2 != 1 or kernel < 1:
        raise ValueError("kernel must be odd and positive")
    r = kernel // 2
    n = a.shape[-1]
    padded = np.zeros(a.shape[:-1] + (n + 2 * r,))
    padded[..., r:r + n] = a
    out = np.zeros_like(a)
    for t in range(kernel):
        out += padded[..., t:t + n]
    return out / kernel


def top_c(p, c):
    """Indices of the min(c, n) largest pooled scores, ascending.

    SnapKV, section "Top-k SelectionとCluster-based Retention", equation S,
    and step 4-5 of the page's routine (top-k then sort).  Reading for ties,
    which the page leaves to the library: the lower index wins.
    """
    p = np.asarray(p, dtype=np.float64)
    n = p.shape[-1]
    cc = min(c, n)
    flat = p.reshape(-1, n)
    out = np.empty((flat.shape[0], cc), dtype=np.int64)
    ids = np.arange(n)
    for r in range(flat.shape[0]):
        order = np.lexsort((ids, -flat[r]))
        out[r] = np.sort(order[:cc])
    return out.reshape(p.shape[:-1] + (cc,))


def compress(q_obs, K, V, n, c, kernel=3):
    """(idx [B,Hkv,c'], K_c, V_c [B,Hkv,c',d], a, p): the compacted cache."""
    a = window_mean(q_obs, K, n)
    p = pool(a, kernel)
    idx = top_c(p, c)
    K = np.asarray(K)
    V = np.asarray(V)
    B, Hkv = idx.shape[:2]
    Kc = np.stack([np.stack([K[b, g, idx[b, g]] for g in range(Hkv)]) for b in range(B)])
    Vc = np.stack([np.stack([V[b, g, idx[b, g]] for g in range(Hkv)]) for b in range(B)])
    return idx, Kc, Vc, a, p
