"""Query-aware sparse KV selection and attention on GB300 (sm_103a).

Thin Python binding over the C ABI of libqasc (include/qasc.h): every call
checks and marshals torch tensors (device memory) into pointers and sizes and
enqueues the library's CUDA kernels on the current (or given) stream.  No step
of the computation runs in Python or PyTorch; if the library is missing the
calls raise.

Entry points keep the C names:
  ts_index_append, ts_select_workspace_bytes, ts_score_vote_select,
  ts_attn_workspace_bytes, ts_sparse_attn, ts_sparse_attn_noalloc,
  ts_head_select_workspace_bytes, ts_score_select_per_head,
  ts_sparse_attn_per_head, ts_expand_capacity, ts_expand_workspace_bytes,
  ts_expand_neighbors, ts_sparse_attn_ex, ts_index_append_paged,
  ts_score_vote_select_paged, ts_score_select_per_head_paged,
  ts_sparse_attn_paged, ts_ring_flush,
  ts_dense_attn_workspace_bytes, ts_dense_attn, snapkv_workspace_bytes,
  snapkv_compress, qasc_status_string, qasc_last_error, qasc_last_cuda_error, qasc_device_error,
  qasc_selftest_bounded_wait, qasc_version.
"""

import ctypes

import torch

from . import _lib

D = 128
D_IDX = 32


class QascError(RuntimeError):
    def __init__(self, status, message):
        self.status = status
        super().__init__("%s: %s" % (_lib.STATUS_NAMES.get(status, str(status)), message))


def _L():
    return _lib.load()


def _check(status):
    if status != _lib.QASC_OK:
        msg = _L().qasc_last_error()
        raise QascError(status, msg.decode() if msg else "")


def _sized(nbytes):
    """A size query's answer; 0 with a message means the library rejected
    the arguments (the same checks as the call being sized)."""
    if nbytes == 0:
        msg = _L().qasc_last_error()
        if msg:
            raise QascError(_lib.QASC_ERR_INVALID_ARG, msg.decode())
    return int(nbytes)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t, name, dtype):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.device.index != torch.cuda.current_device():
        # The library launches on the current device; another GPU's memory
        # would be dereferenced by its kernels.
        raise ValueError("%s is on %s but the current device is cuda:%d" % (name, t.device,
                                                                             torch.cuda.current_device()))
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return ctypes.c_void_p(t.data_ptr())


def _dims(t, name, dims):
    """Raise unless tensor t (None passes) has these dimensions (None = any).
    The library sees only pointers, so every extent is checked here."""
    if t is None:
        return
    got = tuple(t.shape)
    if len(got) != len(dims) or any(d is not None and g != d for g, d in zip(got, dims)):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple("*" if d is None else d for d in dims), got))


def make_shape(B, Hq, Hkv, n, n_cap):
    return _lib.qasc_shape(B, Hq, Hkv, D, D_IDX, 0, n, n_cap)


def ts_params(K, sink=4, local=256, vmin=1):
    return _lib.qasc_ts_params(K, sink, local, vmin)


def snap_params(c, window=32, pool_k=3):
    return _lib.qasc_snap_params(c, window, pool_k, 0)


def budget_tokens(n, budget_permille, sink=4, local=256):
    """K = min(floor(budget * n), |C|) with the floor taken in integers."""
    c1 = max(n - local, sink)
    return min((budget_permille * n) // 1000, c1 - sink)


def alloc_workspace(nbytes, device=None):
    """Caller-owned workspace (uint8) of at least nbytes, 256-byte aligned."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


# ------------------------------------------------------------------ TokenSelect
def ts_index_append(K, W, index, start, count, *, Hq=None, n=None, stream=None):
    """index[b, g, start:start+count] = RNE_bf16(K[b, g, rows] @ W[g])."""
    _dims(K, "K", (None, None, None, D))
    B, Hkv, n_cap, _ = K.shape
    _dims(W, "W", (Hkv, D, D_IDX))
    _dims(index, "index", (B, Hkv, n_cap, D_IDX))
    shape = make_shape(B, Hq or Hkv, Hkv, n or n_cap, n_cap)
    _check(_L().ts_index_append(ctypes.byref(shape), _ptr(K, "K", torch.bfloat16), _ptr(W, "W", torch.bfloat16),
                                _ptr(index, "index", torch.bfloat16), int(start), int(count), _stream(stream)))


def ts_select_workspace_bytes(B, Hq, Hkv, n, n_cap, K, sink=4, local=256, vmin=1):
    shape = make_shape(B, Hq, Hkv, n, n_cap)
    params = ts_params(K, sink, local, vmin)
    return _sized(_L().ts_select_workspace_bytes(ctypes.byref(shape), ctypes.byref(params)))


def ts_score_vote_select(q, W, index, sel, workspace, *, n, K, sink=4, local=256, vmin=1, stream=None):
    """sel[b, :K] = the selected candidate tokens of sequence b, ascending."""
    _dims(q, "q", (None, None, D))
    B, Hq, _ = q.shape
    _dims(index, "index", (B, None, None, D_IDX))
    _, Hkv, n_cap, _ = index.shape
    _dims(W, "W", (Hkv, D, D_IDX))
    _dims(sel, "sel", (B, K))
    shape = make_shape(B, Hq, Hkv, n, n_cap)
    params = ts_params(K, sink, local, vmin)
    _check(_L().ts_score_vote_select(ctypes.byref(shape), ctypes.byref(params), _ptr(q, "q", torch.bfloat16),
                                     _ptr(W, "W", torch.bfloat16), _ptr(index, "index", torch.bfloat16),
                                     _ptr(sel, "sel", torch.int32), _ptr(workspace, "workspace", torch.uint8),
                                     workspace.numel(), _stream(stream)))


def _attn_dims(q, K, V, out, lse):
    _dims(q, "q", (None, None, D))
    B, Hq, _ = q.shape
    _dims(K, "K", (B, None, None, D))
    _, Hkv, n_cap, _ = K.shape
    _dims(V, "V", (B, Hkv, n_cap, D))
    _dims(out, "out", (B, Hq, D))
    _dims(lse, "lse", (B, Hq))
    return B, Hq, Hkv, n_cap


def ts_attn_workspace_bytes(B, Hq, Hkv, n, n_cap, K, sink=4, local=256):
    shape = make_shape(B, Hq, Hkv, n, n_cap)
    params = ts_params(K, sink, local, 1)
    return _sized(_L().ts_attn_workspace_bytes(ctypes.byref(shape), ctypes.byref(params)))


def ts_sparse_attn(q, K, V, sel, out, workspace, *, n, sink=4, local=256, lse=None, stream=None):
    """out[b, h] = attention of q[b, h] over sink + sel[b] + local tokens."""
    B, Hq, Hkv, n_cap = _attn_dims(q, K, V, out, lse)
    _dims(sel, "sel", (B, None))
    Ksel = sel.shape[1] if sel is not None else 0
    shape = make_shape(B, Hq, Hkv, n, n_cap)
    params = ts_params(Ksel, sink, local, 1)
    _check(_L().ts_sparse_attn(ctypes.byref(shape), ctypes.byref(params), _ptr(q, "q", torch.bfloat16),
                               _ptr(K, "K", torch.bfloat16), _ptr(V, "V", torch.bfloat16),
                               _ptr(sel, "sel", torch.int32) if Ksel else None,
                               _ptr(out, "out", torch.float32), _ptr(lse, "lse", torch.float32),
                               _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream)))


def ts_head_select_workspace_bytes(B, Hq, Hkv, n, n_cap, K, sink=4, local=256):
    shape = make_shape(B, Hq, Hkv, n, n_cap)
    params = ts_params(K, sink, local, 1)
    return _sized(_L().ts_head_select_workspace_bytes(ctypes.byref(shape), ctypes.byref(params)))


def ts_score_select_per_head(q, W, index, sel, workspace, *, n, K, sink=4, local=256, stream=None):
    """sel[b, g, :K] = the candidates with the K largest group-summed scores
    of KV head g, ascending (selection without voting)."""
    _dims(q, "q", (None, None, D))
    B, Hq, _ = q.shape
    _dims(index, "index", (B, None, None, D_IDX))
    _, Hkv, n_cap, _ = index.shape
    _dims(W, "W", (Hkv, D, D_IDX))
    _dims(sel, "sel", (B, Hkv, K))
    shape = make_shape(B, Hq, Hkv, n, n_cap)
    params = ts_params(K, sink, local, 1)
    _check(_L().ts_score_select_per_head(ctypes.byref(shape), ctypes.byref(params), _ptr(q, "q", torch.bfloat16),
                                         _ptr(W, "W", torch.bfloat16), _ptr(index, "index", torch.bfloat16),
                                         _ptr(sel, "sel", torch.int32), _ptr(workspace, "workspace", torch.uint8),
                                         workspace.numel(), _stream(stream)))


def ts_sparse_attn_per_head(q, K, V, sel, out, workspace, *, n, sink=4, local=256, lse=None, stream=None):
    """out[b, h] = attention of q[b, h] over sink + sel[b, g(h)] + local tokens."""
    B, Hq, Hkv, n_cap = _attn_dims(q, K, V, out, lse)
    _dims(sel, "sel", (B, Hkv, None))
    Ksel = sel.shape[2] if sel is not None else 0
    shape = make_shape(B, Hq, Hkv, n, n_cap)
    params = ts_params(Ksel, sink, local, 1)
    _check(_L().ts_sparse_attn_per_head(ctypes.byref(shape), ctypes.byref(params), _ptr(q, "q", torch.bfloat16),
                                        _ptr(K, "K", torch.bfloat16), _ptr(V, "V", torch.bfloat16),
                                        _ptr(sel, "sel", torch.int32) if Ksel else None,
                                        _ptr(out, "out", torch.float32), _ptr(lse, "lse", torch.float32),
                                        _ptr(workspace, "workspace", torch.uint8), workspace.numel(),
                                        _stream(stream)))


def ts_expand_capacity(n, K, radius, sink=4, local=256, n_cap=None, B=1, Hq=1, Hkv=1):
    shape = make_shape(B, Hq, Hkv, n, n_cap or n)
    params = ts_params(K, sink, local, 1)
    return _sized(_L().ts_expand_capacity(ctypes.byref(shape), ctypes.byref(params), radius))


def ts_expand_workspace_bytes(n, K, rows, sink=4, local=256):
    shape = make_shape(1, 1, 1, n, n)
    params = ts_params(K, sink, local, 1)
    return _sized(_L().ts_expand_workspace_bytes(ctypes.byref(shape), ctypes.byref(params), rows))


def ts_expand_neighbors(sel, radius, sel_out, lengths, workspace, *, n, sink=4, local=256, stream=None):
    """sel_out[r, :lengths[r]] = ascending union of [j - radius, j + radius]
    over j in sel[r], within the candidates; sel is [rows, K] (or [B, Hkv, K],
    flattened to rows)."""
    lead = tuple(sel_out.shape[:-1])
    if tuple(sel.shape[:-1]) != lead or tuple(lengths.shape) != lead:
        raise ValueError("sel %s, sel_out %s and lengths %s must share their leading dimensions"
                         % (tuple(sel.shape), tuple(sel_out.shape), tuple(lengths.shape)))
    rows = sel_out.numel() // sel_out.shape[-1]
    K = sel.shape[-1]
    shape = make_shape(1, 1, 1, n, n)
    params = ts_params(K, sink, local, 1)
    _check(_L().ts_expand_neighbors(ctypes.byref(shape), ctypes.byref(params), rows,
                                    _ptr(sel, "sel", torch.int32) if K else None, radius,
                                    _ptr(sel_out, "sel_out", torch.int32), sel_out.shape[-1],
                                    _ptr(lengths, "lengths", torch.int32),
                                    _ptr(workspace, "workspace", torch.uint8), workspace.numel(),
                                    _stream(stream)))


def ts_sparse_attn_ex(q, K, V, sel, out, workspace, *, n, sink=4, local=256, lengths=None, per_kv_head=False,
                      lse=None, stream=None):
    """Attention over sink + sel[b] (or sel[b, g(h)] when per_kv_head) + local,
    using only the first lengths[...] entries of each list when given."""
    B, Hq, Hkv, n_cap = _attn_dims(q, K, V, out, lse)
    _dims(sel, "sel", (B, Hkv, None) if per_kv_head else (B, None))
    _dims(lengths, "lengths", (B, Hkv) if per_kv_head else (B,))
    Ksel = sel.shape[-1] if sel is not None else 0
    shape = make_shape(B, Hq, Hkv, n, n_cap)
    params = ts_params(Ksel, sink, local, 1)
    _check(_L().ts_sparse_attn_ex(ctypes.byref(shape), ctypes.byref(params), _ptr(q, "q", torch.bfloat16),
                                  _ptr(K, "K", torch.bfloat16), _ptr(V, "V", torch.bfloat16),
                                  _ptr(sel, "sel", torch.int32) if Ksel else None,
                                  _ptr(lengths, "lengths", torch.int32), 1 if per_kv_head else 0,
                                  _ptr(out, "out", torch.float32), _ptr(lse, "lse", torch.float32),
                                  _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream)))


def paged_cache(block_table, page_tokens, num_pages):
    """Descriptor of a paged pool: block_table [B, pages_per_seq] int32 on
    the device maps each sequence's logical pages of page_tokens tokens to
    pool pages ([num_pages, Hkv, page_tokens, width] pools)."""
    bt = _ptr(block_table, "block_table", torch.int32)
    if block_table.dim() != 2:
        raise ValueError("block_table must be [B, pages_per_seq]")
    return _lib.qasc_paged_cache(bt.value, int(page_tokens), int(block_table.shape[1]), int(num_pages))


def _pool_geometry(pool, block_table, width=D):
    _dims(pool, "pool", (None, None, None, width))
    _dims(block_table, "block_table", (None, None))
    num_pages, Hkv, P, _ = pool.shape
    B, pps = block_table.shape
    return B, Hkv, P, num_pages, pps * P


def ts_index_append_paged(K_pool, W, index_pool, block_table, start, count, *, Hq=None, n=None, stream=None):
    """Index rows of tokens [start, start + count) of every sequence, in the
    pool page that holds each token."""
    B, Hkv, P, num_pages, n_cap = _pool_geometry(K_pool, block_table)
    _dims(W, "W", (Hkv, D, D_IDX))
    _dims(index_pool, "index_pool", (num_pages, Hkv, P, D_IDX))
    shape = make_shape(B, Hq or Hkv, Hkv, n or n_cap, n_cap)
    cache = paged_cache(block_table, P, num_pages)
    _check(_L().ts_index_append_paged(ctypes.byref(shape), ctypes.byref(cache), _ptr(K_pool, "K_pool", torch.bfloat16),
                                      _ptr(W, "W", torch.bfloat16), _ptr(index_pool, "index_pool", torch.bfloat16),
                                      int(start), int(count), _stream(stream)))


def ts_score_vote_select_paged(q, W, index_pool, block_table, sel, workspace, *, n, K, sink=4, local=256, vmin=1,
                               stream=None):
    """ts_score_vote_select over a paged index pool (workspace:
    ts_select_workspace_bytes with n_cap = pages_per_seq * page_tokens)."""
    B, Hkv, P, num_pages, n_cap = _pool_geometry(index_pool, block_table, D_IDX)
    _dims(q, "q", (B, None, D))
    _dims(W, "W", (Hkv, D, D_IDX))
    _dims(sel, "sel", (B, K))
    shape = make_shape(B, q.shape[1], Hkv, n, n_cap)
    params = ts_params(K, sink, local, vmin)
    cache = paged_cache(block_table, P, num_pages)
    _check(_L().ts_score_vote_select_paged(ctypes.byref(shape), ctypes.byref(params), ctypes.byref(cache),
                                           _ptr(q, "q", torch.bfloat16), _ptr(W, "W", torch.bfloat16),
                                           _ptr(index_pool, "index_pool", torch.bfloat16),
                                           _ptr(sel, "sel", torch.int32), _ptr(workspace, "workspace", torch.uint8),
                                           workspace.numel(), _stream(stream)))


def ts_score_select_per_head_paged(q, W, index_pool, block_table, sel, workspace, *, n, K, sink=4, local=256,
                                   stream=None):
    """ts_score_select_per_head over a paged index pool (workspace:
    ts_head_select_workspace_bytes with n_cap = pages_per_seq * page_tokens)."""
    B, Hkv, P, num_pages, n_cap = _pool_geometry(index_pool, block_table, D_IDX)
    _dims(q, "q", (B, None, D))
    _dims(W, "W", (Hkv, D, D_IDX))
    _dims(sel, "sel", (B, Hkv, K))
    shape = make_shape(B, q.shape[1], Hkv, n, n_cap)
    params = ts_params(K, sink, local, 1)
    cache = paged_cache(block_table, P, num_pages)
    _check(_L().ts_score_select_per_head_paged(ctypes.byref(shape), ctypes.byref(params), ctypes.byref(cache),
                                               _ptr(q, "q", torch.bfloat16), _ptr(W, "W", torch.bfloat16),
                                               _ptr(index_pool, "index_pool", torch.bfloat16),
                                               _ptr(sel, "sel", torch.int32),
                                               _ptr(workspace, "workspace", torch.uint8), workspace.numel(),
                                               _stream(stream)))


def _ring(ring, B, Hkv):
    if ring is None:
        return None
    rk, rv = ring
    if rk.shape != rv.shape or rk.dim() != 4 or tuple(rk.shape[:2]) != (B, Hkv) or rk.shape[3] != D:
        raise ValueError("ring K and V must both be [B=%d, Hkv=%d, R, %d]" % (B, Hkv, D))
    return _lib.qasc_local_ring(_ptr(rk, "ring K", torch.bfloat16).value, _ptr(rv, "ring V", torch.bfloat16).value,
                                int(rk.shape[2]))


def ts_sparse_attn_paged(q, K_pool, V_pool, block_table, sel, out, workspace, *, n, sink=4, local=256, ring=None,
                         lengths=None, per_kv_head=False, lse=None, stream=None):
    """ts_sparse_attn_ex over a paged pool; ring = (ring_K, ring_V), each
    [B, Hkv, R, d] with token t at slot t mod R, supplies the local tokens."""
    B, Hkv, P, num_pages, n_cap = _pool_geometry(K_pool, block_table)
    _dims(V_pool, "V_pool", (num_pages, Hkv, P, D))
    _dims(q, "q", (B, None, D))
    Hq = q.shape[1]
    _dims(out, "out", (B, Hq, D))
    _dims(lse, "lse", (B, Hq))
    _dims(sel, "sel", (B, Hkv, None) if per_kv_head else (B, None))
    _dims(lengths, "lengths", (B, Hkv) if per_kv_head else (B,))
    Ksel = sel.shape[-1] if sel is not None else 0
    shape = make_shape(B, q.shape[1], Hkv, n, n_cap)
    params = ts_params(Ksel, sink, local, 1)
    cache = paged_cache(block_table, P, num_pages)
    rg = _ring(ring, B, Hkv)
    _check(_L().ts_sparse_attn_paged(ctypes.byref(shape), ctypes.byref(params), ctypes.byref(cache),
                                     ctypes.byref(rg) if rg is not None else None, _ptr(q, "q", torch.bfloat16),
                                     _ptr(K_pool, "K_pool", torch.bfloat16), _ptr(V_pool, "V_pool", torch.bfloat16),
                                     _ptr(sel, "sel", torch.int32) if Ksel else None,
                                     _ptr(lengths, "lengths", torch.int32), 1 if per_kv_head else 0,
                                     _ptr(out, "out", torch.float32), _ptr(lse, "lse", torch.float32),
                                     _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream)))


def ts_ring_flush(ring, W, K_pool, V_pool, index_pool, block_table, start, count, *, n=None, stream=None):
    """Tokens [start, start + count) of every sequence from the ring into
    their pages (K and V rows copied, index rows written)."""
    B, Hkv, P, num_pages, n_cap = _pool_geometry(K_pool, block_table)
    _dims(V_pool, "V_pool", (num_pages, Hkv, P, D))
    _dims(index_pool, "index_pool", (num_pages, Hkv, P, D_IDX))
    _dims(W, "W", (Hkv, D, D_IDX))
    shape = make_shape(B, Hkv, Hkv, n or n_cap, n_cap)
    cache = paged_cache(block_table, P, num_pages)
    rg = _ring(ring, B, Hkv)
    _check(_L().ts_ring_flush(ctypes.byref(shape), ctypes.byref(cache), ctypes.byref(rg) if rg is not None else None,
                              _ptr(W, "W", torch.bfloat16), _ptr(K_pool, "K_pool", torch.bfloat16),
                              _ptr(V_pool, "V_pool", torch.bfloat16), _ptr(index_pool, "index_pool", torch.bfloat16),
                              int(start), int(count), _stream(stream)))


def ts_sparse_attn_noalloc(q, K, V, sel, out, *, n, sink=4, local=256, lse=None, stream=None):
    """ts_sparse_attn without a workspace, for callers that cannot allocate
    device memory: the split-K scratch is a fixed 16 MiB area inside the
    library, shared by all calls (serialise calls that could overlap)."""
    B, Hq, Hkv, n_cap = _attn_dims(q, K, V, out, lse)
    _dims(sel, "sel", (B, None))
    Ksel = sel.shape[1] if sel is not None else 0
    shape = make_shape(B, Hq, Hkv, n, n_cap)
    params = ts_params(Ksel, sink, local, 1)
    _check(_L().ts_sparse_attn_noalloc(ctypes.byref(shape), ctypes.byref(params), _ptr(q, "q", torch.bfloat16),
                                       _ptr(K, "K", torch.bfloat16), _ptr(V, "V", torch.bfloat16),
                                       _ptr(sel, "sel", torch.int32) if Ksel else None,
                                       _ptr(out, "out", torch.float32), _ptr(lse, "lse", torch.float32),
                                       _stream(stream)))


def ts_dense_attn_workspace_bytes(B, Hq, Hkv, n, n_cap):
    shape = make_shape(B, Hq, Hkv, n, n_cap)
    return _sized(_L().ts_dense_attn_workspace_bytes(ctypes.byref(shape)))


def ts_dense_attn(q, K, V, out, workspace, *, n, lse=None, stream=None):
    """out[b, h] = attention of q[b, h] over all n cached tokens (the baseline)."""
    B, Hq, Hkv, n_cap = _attn_dims(q, K, V, out, lse)
    shape = make_shape(B, Hq, Hkv, n, n_cap)
    _check(_L().ts_dense_attn(ctypes.byref(shape), _ptr(q, "q", torch.bfloat16), _ptr(K, "K", torch.bfloat16),
                              _ptr(V, "V", torch.bfloat16), _ptr(out, "out", torch.float32),
                              _ptr(lse, "lse", torch.float32), _ptr(workspace, "workspace", torch.uint8),
                              workspace.numel(), _stream(stream)))


# ------------------------------------------------------------------ SnapKV
def snapkv_workspace_bytes(B, Hq, Hkv, n, n_cap, c, window=32, pool_k=3):
    shape = make_shape(B, Hq, Hkv, n, n_cap)
    params = snap_params(c, window, pool_k)
    return _sized(_L().snapkv_workspace_bytes(ctypes.byref(shape), ctypes.byref(params)))


def snapkv_compress(q_obs, K, V, idx, K_out, V_out, workspace, *, n, c, pool_k=3, stream=None):
    """Keep min(c, n) entries per KV head chosen by observation-window attention."""
    _dims(q_obs, "q_obs", (None, None, None, D))
    B, Hq, w, _ = q_obs.shape
    _dims(K, "K", (B, None, None, D))
    _, Hkv, n_cap, _ = K.shape
    _dims(V, "V", (B, Hkv, n_cap, D))
    c_out = min(c, n)
    _dims(idx, "idx", (B, Hkv, c_out))
    _dims(K_out, "K_out", (B, Hkv, c_out, D))
    _dims(V_out, "V_out", (B, Hkv, c_out, D))
    shape = make_shape(B, Hq, Hkv, n, n_cap)
    params = snap_params(c, w, pool_k)
    _check(_L().snapkv_compress(ctypes.byref(shape), ctypes.byref(params), _ptr(q_obs, "q_obs", torch.bfloat16),
                                _ptr(K, "K", torch.bfloat16), _ptr(V, "V", torch.bfloat16),
                                _ptr(idx, "idx", torch.int32), _ptr(K_out, "K_out", torch.bfloat16),
                                _ptr(V_out, "V_out", torch.bfloat16), _ptr(workspace, "workspace", torch.uint8),
                                workspace.numel(), _stream(stream)))


# ------------------------------------------------------------------ status
def qasc_status_string(status):
    return _L().qasc_status_string(int(status)).decode()


def qasc_last_error():
    return _L().qasc_last_error().decode()


def qasc_last_cuda_error():
    return _L().qasc_last_cuda_error().decode()


def qasc_device_error(stream=None):
    _check(_L().qasc_device_error(_stream(stream)))


def qasc_selftest_bounded_wait(limit_us, stream=None):
    """Run one kernel whose bounded wait cannot complete; it gives up after
    limit_us and records a timeout for the next qasc_device_error()."""
    _check(_L().qasc_selftest_bounded_wait(int(limit_us), _stream(stream)))


def qasc_version():
    return int(_L().qasc_version())
