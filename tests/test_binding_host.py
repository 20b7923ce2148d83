"""The Python binding checks every tensor extent before a call reaches the
library (which sees only pointers).  CPU only: the checks run before any
device pointer is taken, so CPU tensors of the wrong shape are enough."""

import pytest
import torch

import query_aware_sparse_compressed_gb300 as qasc

bf, i32, f32 = torch.bfloat16, torch.int32, torch.float32


def t(*shape, dtype=bf):
    return torch.zeros(shape, dtype=dtype)


def test_dims_helper():
    qasc._dims(None, "x", (1, 2))
    qasc._dims(t(2, 3), "x", (2, None))
    with pytest.raises(ValueError, match="x must have shape"):
        qasc._dims(t(2, 3), "x", (2, 4))
    with pytest.raises(ValueError):
        qasc._dims(t(2, 3, 1), "x", (2, 3))


@pytest.mark.parametrize("call", [
    # sel shorter than (B, K)
    lambda: qasc.ts_score_vote_select(t(2, 8, 128), t(2, 128, 32), t(2, 2, 512, 32), t(2, 10, dtype=i32), t(256),
                                      n=512, K=20),
    # W of the wrong KV head count
    lambda: qasc.ts_index_append(t(2, 2, 512, 128), t(3, 128, 32), t(2, 2, 512, 32), 0, 10),
    # out too small
    lambda: qasc.ts_sparse_attn(t(2, 8, 128), t(2, 2, 512, 128), t(2, 2, 512, 128), t(2, 30, dtype=i32),
                                t(2, 4, 128, dtype=f32), t(256), n=512),
    # V not the shape of K
    lambda: qasc.ts_dense_attn(t(2, 8, 128), t(2, 2, 512, 128), t(2, 2, 500, 128), t(2, 8, 128, dtype=f32), t(256),
                               n=512),
    # per-KV-head lengths given as per-sequence
    lambda: qasc.ts_sparse_attn_ex(t(2, 8, 128), t(2, 2, 512, 128), t(2, 2, 512, 128), t(2, 2, 30, dtype=i32),
                                   t(2, 8, 128, dtype=f32), t(256), n=512, lengths=t(2, dtype=i32), per_kv_head=True),
    # expansion lengths not matching the rows
    lambda: qasc.ts_expand_neighbors(t(4, 30, dtype=i32), 1, t(4, 90, dtype=i32), t(3, dtype=i32), t(256), n=512),
    # paged: V pool of another page count
    lambda: qasc.ts_sparse_attn_paged(t(2, 8, 128), t(9, 2, 64, 128), t(8, 2, 64, 128), t(2, 8, dtype=i32),
                                      t(2, 30, dtype=i32), t(2, 8, 128, dtype=f32), t(256), n=500),
    # SnapKV: idx not (B, Hkv, min(c, n))
    lambda: qasc.snapkv_compress(t(1, 8, 32, 128), t(1, 2, 1000, 128), t(1, 2, 1000, 128), t(1, 2, 64, dtype=i32),
                                 t(1, 2, 100, 128), t(1, 2, 100, 128), t(256), n=1000, c=100),
])
def test_wrong_extents_are_rejected_before_the_library(call):
    with pytest.raises(ValueError, match="must have shape|leading dimensions"):
        call()


@pytest.mark.parametrize("query", [
    lambda: qasc.ts_select_workspace_bytes(1, 8, 2, 0, 4096, 409),          # n = 0
    lambda: qasc.ts_attn_workspace_bytes(1, 8, 2, 4096, 4096, 5000),        # K > |C|
    lambda: qasc.ts_head_select_workspace_bytes(1, 8, 3, 4096, 4096, 409),  # Hq not a multiple of Hkv
    lambda: qasc.ts_expand_capacity(4096, 409, -1),
    lambda: qasc.ts_expand_workspace_bytes(4096, 409, 0),
    lambda: qasc.ts_dense_attn_workspace_bytes(1, 8, 2, 5000, 4096),        # n > n_cap
    lambda: qasc.snapkv_workspace_bytes(1, 8, 2, 1000, 1000, 64, window=64),  # 4 x 64 rows > one tile
])
def test_rejected_size_queries_raise(query):
    with pytest.raises(qasc.QascError):
        query()


def test_accepted_size_queries_return_sizes():
    assert qasc.ts_select_workspace_bytes(1, 8, 2, 4096, 4096, 409) > 0
    assert qasc.ts_expand_capacity(4096, 100, 3) == 700


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    # No fallback: without libqasc.so every entry point raises instead of
    # computing anything elsewhere.
    from query_aware_sparse_compressed_gb300 import _lib
    missing = str(tmp_path / "libqasc.so")
    with pytest.raises(RuntimeError, match="not built"):
        _lib.load(missing)
    monkeypatch.setattr(_lib, "LIB_PATH", missing)
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        qasc.ts_select_workspace_bytes(1, 8, 2, 4096, 4096, 409)
