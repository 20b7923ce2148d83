"""Where each token's cache rows live: a paged pool and a circular local
buffer, as plain fp64 NumPy.

Test infrastructure only (see the package docstring).

Sources:
  TokenSelect, section "まとめ" (conclusion): integration with vLLM's
  PagedAttention is named as the way to run the method where memory is tight;
  the page shows no layout.
  TokenButler, section "Inferenzstrategie": the cache is held in three
  buffers, the first S tokens, a circular buffer of the newest N tokens and
  the important tokens; section "Optimierungen": the keys are projected in
  batches of N tokens, not at every decode step.

Readings (the pages fix no layout):
  Paged pool.  Fixed pages of P tokens; a page holds the rows of all Hkv KV
  heads, pool [num_pages, Hkv, P, w] (w = d for K and V, d_idx for the
  index).  A block table [B, pages_per_seq] gives the pool page of each
  logical page: token t of sequence b is row t mod P of page
  block_table[b, t // P].  The index uses the same pages and table.
  Circular local buffer.  ring [B, Hkv, R, d] for K and V, R >= local:
  token t sits in slot t mod R.  Attention reads the local tokens from the
  ring and every other token from the main cache.
  Flush.  Tokens enter the main cache in batches: their K and V rows are
  copied out of the ring into their pages and their index rows are projected
  then (once per batch), before they leave the local window.
"""

import numpy as np

from .tokenselect import index_rows, regions


def page_of(block_table, P, b, t):
    """(pool page, row within the page) of token t of sequence b."""
    return int(block_table[b][t // P]), t % P


def logical_rows(pool, block_table, P, n):
    """Rows of tokens 0..n-1 of every sequence: [B, Hkv, n, w], where
    out[b, :, t] = pool[block_table[b, t // P], :, t % P]."""
    pool = np.asarray(pool)
    bt = np.asarray(block_table)
    B = bt.shape[0]
    out = np.empty((B, pool.shape[1], n, pool.shape[3]), dtype=np.float64)
    for b in range(B):
        for t in range(n):
            page, r = page_of(bt, P, b, t)
            out[b, :, t] = pool[page, :, r]
    return out


def ring_slot(t, R):
    """Slot of token t in a circular buffer of R slots."""
    return t % R


def attended_rows(main_rows, ring, R, n, sink, local):
    """The rows that attention reads for a cache of n tokens: the local
    tokens [local_start, n) from the ring, every other token from main_rows
    ([B, Hkv, >= n, w]).  Returns [B, Hkv, n, w]."""
    out = np.array(np.asarray(main_rows, dtype=np.float64)[:, :, :n])
    _, _, _, local_start = regions(n, sink, local)
    ring = np.asarray(ring, dtype=np.float64)
    for t in range(local_start, n):
        out[:, :, t] = ring[:, :, ring_slot(t, R)]
    return out


def ring_flush(pool_K, pool_V, pool_index, block_table, P, ring_K, ring_V, R, W, start, count):
    """Move tokens [start, start + count) of every sequence from the ring
    into their pages, with their index rows; returns new (K, V, index)
    pools, the other rows unchanged."""
    K2 = np.array(pool_K, dtype=np.float64)
    V2 = np.array(pool_V, dtype=np.float64)
    I2 = np.array(pool_index, dtype=np.float64)
    ring_K = np.asarray(ring_K, dtype=np.float64)
    ring_V = np.asarray(ring_V, dtype=np.float64)
    bt = np.asarray(block_table)
    for b in range(bt.shape[0]):
        for t in range(start, start + count):
            page, r = page_of(bt, P, b, t)
            s = ring_slot(t, R)
            K2[page, :, r] = ring_K[b, :, s]
            V2[page, :, r] = ring_V[b, :, s]
            I2[page, :, r] = index_rows(ring_K[b:b + 1, :, s:s + 1], W)[0, :, 0]
    return K2, V2, I2
