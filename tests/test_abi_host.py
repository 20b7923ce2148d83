"""Host-side checks of the C ABI: the library loads, exports exactly what
include/qasc.h declares, sizes workspaces and rejects bad arguments before
touching a device.  CPU only (no kernel is launched)."""

import ctypes
import os
import re

import pytest

from query_aware_sparse_compressed_gb300 import _lib
from query_aware_sparse_compressed_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qasc.h")


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return _lib.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"QASC_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("ts_index_append", "ts_score_vote_select", "ts_sparse_attn", "snapkv_compress",
                 "ts_select_workspace_bytes", "ts_attn_workspace_bytes", "snapkv_workspace_bytes"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, name


def test_exports_nothing_else(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True).stdout
    exported = sorted(l.split()[-1] for l in out.splitlines() if " T " in l)
    assert exported == declared_symbols()


def shape(B=1, Hq=8, Hkv=2, n=4096, n_cap=4096, d=128, d_idx=32):
    return _lib.qasc_shape(B, Hq, Hkv, d, d_idx, 0, n, n_cap)


def params(K=409, sink=4, local=256, vmin=1):
    return _lib.qasc_ts_params(K, sink, local, vmin)


FAKE = ctypes.c_void_p(0x10000)       # aligned, never dereferenced
MISALIGNED = ctypes.c_void_p(0x10008)


def test_status_strings(lib):
    assert lib.qasc_status_string(0) == b"QASC_OK"
    assert lib.qasc_status_string(3) == b"QASC_ERR_WORKSPACE"
    assert lib.qasc_version() >= 100


def test_workspace_sizes(lib):
    s, p = shape(), params()
    a = lib.ts_select_workspace_bytes(ctypes.byref(s), ctypes.byref(p))
    # scores B*Hq*nc_pad*4 + theta + keys B*nc_pad*8
    nc_pad = -(-(4096 - 260) // 64) * 64
    assert a >= 8 * nc_pad * 4 + nc_pad * 8
    b = lib.ts_attn_workspace_bytes(ctypes.byref(s), ctypes.byref(p))
    assert b >= 8 * 132 * 4
    assert lib.ts_select_workspace_bytes(None, ctypes.byref(p)) == 0


@pytest.mark.parametrize("mutate,code", [
    (lambda s, p: setattr(s, "d", 64), 2),
    (lambda s, p: setattr(s, "d_idx", 16), 2),
    (lambda s, p: setattr(s, "Hkv", 3), 1),
    (lambda s, p: setattr(s, "Hq", 96), 1),
    (lambda s, p: (setattr(s, "Hq", 48), setattr(s, "Hkv", 3)), 2),   # group of 16 not compiled in
    (lambda s, p: setattr(s, "n", 0), 1),
    (lambda s, p: setattr(s, "n", 5000), 1),                            # n > n_cap
    (lambda s, p: setattr(p, "K", 5000), 1),                            # K > |C|
    (lambda s, p: setattr(p, "K", -1), 1),
    (lambda s, p: setattr(p, "vmin", 0), 1),
    (lambda s, p: setattr(p, "sink", -1), 1),
])
def test_select_rejects_bad_arguments(lib, mutate, code):
    s, p = shape(), params()
    mutate(s, p)
    st = lib.ts_score_vote_select(ctypes.byref(s), ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, None)
    assert st == code, lib.qasc_last_error()
    assert lib.qasc_last_error()


def test_select_rejects_null_and_misaligned(lib):
    s, p = shape(), params()
    st = lib.ts_score_vote_select(ctypes.byref(s), ctypes.byref(p), None, FAKE, FAKE, FAKE, FAKE, 1 << 30, None)
    assert st == 1 and b"q is NULL" in lib.qasc_last_error()
    st = lib.ts_score_vote_select(ctypes.byref(s), ctypes.byref(p), MISALIGNED, FAKE, FAKE, FAKE, FAKE, 1 << 30, None)
    assert st == 1 and b"aligned" in lib.qasc_last_error()


def test_select_rejects_small_workspace(lib):
    s, p = shape(), params()
    need = lib.ts_select_workspace_bytes(ctypes.byref(s), ctypes.byref(p))
    st = lib.ts_score_vote_select(ctypes.byref(s), ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, need - 1, None)
    assert st == 3
    st = lib.ts_score_vote_select(ctypes.byref(s), ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, None, need, None)
    assert st == 3


def test_zero_budget_select_is_a_no_op(lib):
    s, p = shape(), params(K=0)
    st = lib.ts_score_vote_select(ctypes.byref(s), ctypes.byref(p), FAKE, FAKE, FAKE, None, None, 0, None)
    assert st == 0


def test_append_rejects_rows_outside_capacity(lib):
    s = shape()
    assert lib.ts_index_append(ctypes.byref(s), FAKE, FAKE, FAKE, 4000, 200, None) == 1
    assert lib.ts_index_append(ctypes.byref(s), FAKE, FAKE, FAKE, -1, 2, None) == 1
    assert lib.ts_index_append(ctypes.byref(s), FAKE, FAKE, FAKE, 10, 0, None) == 0   # empty append


def test_attn_rejects_bad_arguments(lib):
    s, p = shape(), params()
    st = lib.ts_sparse_attn(ctypes.byref(s), ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, None, None, FAKE, 1 << 30,
                            None)
    assert st == 1 and b"out" in lib.qasc_last_error()
    p.K = 9999
    st = lib.ts_sparse_attn(ctypes.byref(s), ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 1 << 30,
                            None)
    assert st == 1


def test_snapkv_rejects_bad_arguments(lib):
    s = shape(Hq=32, Hkv=8, n=1000, n_cap=1000)
    sp = _lib.qasc_snap_params(0, 32, 3, 0)
    assert lib.snapkv_compress(ctypes.byref(s), ctypes.byref(sp), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                               1 << 30, None) == 1
    sp = _lib.qasc_snap_params(64, 32, 4, 0)       # even pooling width
    assert lib.snapkv_compress(ctypes.byref(s), ctypes.byref(sp), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                               1 << 30, None) == 1
    sp = _lib.qasc_snap_params(64, 64, 3, 0)       # 4 heads x 64 rows > one 128-row tile
    assert lib.snapkv_compress(ctypes.byref(s), ctypes.byref(sp), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                               1 << 30, None) == 2
    sp = _lib.qasc_snap_params(64, 32, 67, 0)      # pooling window wider than the supported 65
    assert lib.snapkv_compress(ctypes.byref(s), ctypes.byref(sp), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                               1 << 30, None) == 2


def test_expand_capacity_and_workspace(lib):
    s, p = shape(), params(K=100)
    nc = 4096 - 4 - 256
    assert lib.ts_expand_capacity(ctypes.byref(s), ctypes.byref(p), 0) == 100
    assert lib.ts_expand_capacity(ctypes.byref(s), ctypes.byref(p), 3) == 700
    assert lib.ts_expand_capacity(ctypes.byref(s), ctypes.byref(p), 100) == nc      # capped at |C|
    w1 = lib.ts_expand_workspace_bytes(ctypes.byref(s), ctypes.byref(p), 1)
    w4 = lib.ts_expand_workspace_bytes(ctypes.byref(s), ctypes.byref(p), 4)
    assert w1 >= 512 + 4 + 4 and w4 >= 4 * (512 + 4 + 4) and w1 % 256 == 0
    assert lib.ts_expand_workspace_bytes(ctypes.byref(s), ctypes.byref(p), 0) == 0


@pytest.mark.parametrize("rows,radius,cap,ws_bytes,code", [
    (0, 1, 300, 1 << 20, 1),            # no rows
    (70000, 1, 300, 1 << 20, 1),        # more rows than a grid dimension
    (2, -1, 300, 1 << 20, 1),           # negative radius
    (2, (1 << 20) + 1, 300, 1 << 20, 1),
    (2, 1, 299, 1 << 20, 1),            # cap below (2 r + 1) K
    (2, 1, 300, 16, 3),                 # short workspace
])
def test_expand_rejects_bad_arguments(lib, rows, radius, cap, ws_bytes, code):
    s, p = shape(), params(K=100)
    st = lib.ts_expand_neighbors(ctypes.byref(s), ctypes.byref(p), rows, FAKE, radius, FAKE, cap, FAKE, FAKE,
                                 ws_bytes, None)
    assert st == code, lib.qasc_last_error()


def test_expand_rejects_null_workspace_and_misaligned_lengths(lib):
    s, p = shape(), params(K=100)
    st = lib.ts_expand_neighbors(ctypes.byref(s), ctypes.byref(p), 2, FAKE, 1, FAKE, 300, FAKE, None, 1 << 20, None)
    assert st == 3
    st = lib.ts_expand_neighbors(ctypes.byref(s), ctypes.byref(p), 2, FAKE, 1, FAKE, 300,
                                 ctypes.c_void_p(0x10002), FAKE, 1 << 20, None)
    assert st == 1 and b"aligned" in lib.qasc_last_error()


def test_attn_ex_rejects_misaligned_lengths(lib):
    s, p = shape(), params()
    st = lib.ts_sparse_attn_ex(ctypes.byref(s), ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, ctypes.c_void_p(0x10002), 0,
                               FAKE, None, FAKE, 1 << 30, None)
    assert st == 1 and b"aligned" in lib.qasc_last_error()


def paged(P=256, pps=16, num_pages=64, table=FAKE):
    return _lib.qasc_paged_cache(table.value if table is not None else None, P, pps, num_pages)


def test_bad_table_status_string(lib):
    assert lib.qasc_status_string(6) == b"QASC_ERR_BAD_TABLE"
    assert lib.qasc_status_string(7) == b"QASC_ERR_INTERNAL"


@pytest.mark.parametrize("mutate", [
    lambda s, c: setattr(c, "page_tokens", 100),          # not a power of two
    lambda s, c: setattr(c, "page_tokens", 32),           # below 64
    lambda s, c: setattr(c, "pages_per_seq", 0),
    lambda s, c: setattr(c, "num_pages", 0),
    lambda s, c: setattr(s, "n_cap", 4000),               # n_cap != pages_per_seq * P
    lambda s, c: setattr(c, "num_pages", 1 << 22),        # pool rows beyond 2^31
    lambda s, c: setattr(c, "block_table", None),
    lambda s, c: setattr(c, "block_table", 0x10002),      # misaligned table
])
def test_paged_calls_reject_bad_cache(lib, mutate):
    s, c = shape(n=4000, n_cap=4096), paged()
    mutate(s, c)
    p = params()
    assert lib.ts_index_append_paged(ctypes.byref(s), ctypes.byref(c), FAKE, FAKE, FAKE, 0, 10, None) == 1
    assert lib.ts_score_vote_select_paged(ctypes.byref(s), ctypes.byref(p), ctypes.byref(c), FAKE, FAKE, FAKE, FAKE,
                                          FAKE, 1 << 30, None) == 1
    assert lib.ts_sparse_attn_paged(ctypes.byref(s), ctypes.byref(p), ctypes.byref(c), None, FAKE, FAKE, FAKE, FAKE,
                                    None, 0, FAKE, None, FAKE, 1 << 30, None) == 1
    assert lib.ts_score_select_per_head_paged(ctypes.byref(s), ctypes.byref(p), ctypes.byref(c), FAKE, FAKE, FAKE,
                                              FAKE, FAKE, 1 << 30, None) == 1
    assert lib.qasc_last_error()


def test_paged_calls_reject_null_cache_and_short_ring(lib):
    s, p = shape(n=4000, n_cap=4096), params()
    assert lib.ts_index_append_paged(ctypes.byref(s), None, FAKE, FAKE, FAKE, 0, 10, None) == 1
    c = paged()
    ring = _lib.qasc_local_ring(FAKE.value, FAKE.value, 255)          # below local = 256
    st = lib.ts_sparse_attn_paged(ctypes.byref(s), ctypes.byref(p), ctypes.byref(c), ctypes.byref(ring), FAKE, FAKE,
                                  FAKE, FAKE, None, 0, FAKE, None, FAKE, 1 << 30, None)
    assert st == 1 and b"ring_tokens" in lib.qasc_last_error()
    ring = _lib.qasc_local_ring(MISALIGNED.value, FAKE.value, 512)
    st = lib.ts_sparse_attn_paged(ctypes.byref(s), ctypes.byref(p), ctypes.byref(c), ctypes.byref(ring), FAKE, FAKE,
                                  FAKE, FAKE, None, 0, FAKE, None, FAKE, 1 << 30, None)
    assert st == 1 and b"aligned" in lib.qasc_last_error()


def test_ring_flush_rejects_bad_ranges(lib):
    s, c = shape(n=4000, n_cap=4096), paged()
    ring = _lib.qasc_local_ring(FAKE.value, FAKE.value, 300)
    flush = lambda start, count, r=ring: lib.ts_ring_flush(ctypes.byref(s), ctypes.byref(c), ctypes.byref(r), FAKE,
                                                           FAKE, FAKE, FAKE, start, count, None)
    assert flush(0, 301) == 1                  # more tokens than slots
    assert flush(4000, 200) == 1               # past n_cap
    assert flush(-1, 10) == 1
    assert flush(10, 0) == 0                   # empty flush
    assert lib.ts_ring_flush(ctypes.byref(s), ctypes.byref(c), None, FAKE, FAKE, FAKE, FAKE, 0, 10, None) == 1


def test_selftest_rejects_bad_limits(lib):
    assert lib.qasc_selftest_bounded_wait(0, None) == 1
    assert lib.qasc_selftest_bounded_wait(2000001, None) == 1


INT64_MAX = (1 << 63) - 1
INT32_MAX = (1 << 31) - 1


def test_size_queries_reject_what_their_call_rejects(lib):
    p = params()
    sp = _lib.qasc_snap_params(64, 32, 3, 0)
    queries = {
        "ts_select_workspace_bytes": lambda s, p: lib.ts_select_workspace_bytes(ctypes.byref(s), ctypes.byref(p)),
        "ts_attn_workspace_bytes": lambda s, p: lib.ts_attn_workspace_bytes(ctypes.byref(s), ctypes.byref(p)),
        "ts_head_select_workspace_bytes":
            lambda s, p: lib.ts_head_select_workspace_bytes(ctypes.byref(s), ctypes.byref(p)),
        "ts_expand_capacity": lambda s, p: lib.ts_expand_capacity(ctypes.byref(s), ctypes.byref(p), 1),
        "ts_expand_workspace_bytes": lambda s, p: lib.ts_expand_workspace_bytes(ctypes.byref(s), ctypes.byref(p), 4),
        "ts_dense_attn_workspace_bytes": lambda s, p: lib.ts_dense_attn_workspace_bytes(ctypes.byref(s)),
        "snapkv_workspace_bytes": lambda s, p: lib.snapkv_workspace_bytes(ctypes.byref(s), ctypes.byref(sp)),
    }
    for name, query in queries.items():
        for bad in (shape(n=0), shape(n=5000), shape(d=64), shape(Hkv=3)):
            assert query(bad, p) == 0, name
            assert name.encode() in lib.qasc_last_error(), name
        assert query(shape(), p) > 0, name
        assert lib.qasc_last_error() == b"", name          # an accepted query clears the message
    for name in ("ts_select_workspace_bytes", "ts_attn_workspace_bytes", "ts_head_select_workspace_bytes",
                 "ts_expand_capacity", "ts_expand_workspace_bytes"):
        assert queries[name](shape(), params(K=5000)) == 0, name      # K > |C|
    assert lib.ts_expand_capacity(ctypes.byref(shape()), ctypes.byref(p), -1) == 0
    assert lib.ts_expand_workspace_bytes(ctypes.byref(shape()), ctypes.byref(p), 70000) == 0
    big = _lib.qasc_snap_params(64, INT32_MAX, 3, 0)
    assert lib.snapkv_workspace_bytes(ctypes.byref(shape()), ctypes.byref(big)) == 0


def test_row_ranges_cannot_wrap_around(lib):
    # start + count past 2^63 would wrap to a small value; each must be refused
    # on the host (on a machine without a device an accepted call fails with 4)
    s = shape()
    assert lib.ts_index_append(ctypes.byref(s), FAKE, FAKE, FAKE, 10, INT64_MAX, None) == 1
    assert lib.ts_index_append(ctypes.byref(s), FAKE, FAKE, FAKE, INT64_MAX, 1, None) == 1
    assert lib.ts_index_append(ctypes.byref(s), FAKE, FAKE, FAKE, 4096, 0, None) == 0     # empty, at the end
    s, c = shape(n=4000, n_cap=4096), paged()
    assert lib.ts_index_append_paged(ctypes.byref(s), ctypes.byref(c), FAKE, FAKE, FAKE, 10, INT64_MAX, None) == 1
    ring = _lib.qasc_local_ring(FAKE.value, FAKE.value, 300)
    assert lib.ts_ring_flush(ctypes.byref(s), ctypes.byref(c), ctypes.byref(ring), FAKE, FAKE, FAKE, FAKE,
                             INT64_MAX, 1, None) == 1


def test_pool_size_cannot_wrap_around(lib):
    # num_pages * Hkv * P = 2^69 wraps to 0 in 64 bits
    s, c = shape(n=4000, n_cap=4096), paged(num_pages=1 << 60)
    assert lib.ts_index_append_paged(ctypes.byref(s), ctypes.byref(c), FAKE, FAKE, FAKE, 0, 10, None) == 1
    assert b"2^31" in lib.qasc_last_error()


def test_snapkv_window_product_cannot_wrap_around(lib):
    # 4 heads x (2^31 - 1) rows wraps to a negative int32
    s = shape(Hq=32, Hkv=8, n=1000, n_cap=1000)
    sp = _lib.qasc_snap_params(64, INT32_MAX, 3, 0)
    assert lib.snapkv_compress(ctypes.byref(s), ctypes.byref(sp), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                               1 << 30, None) == 2


def test_valid_call_without_a_device_reports_cuda_error(lib):
    # Arguments that pass every check reach the device lookup, which fails
    # here with a CUDA status and a message; nothing is launched.  On a host
    # with a GPU the fake pointers must never reach a kernel, so skip there.
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    st = lib.ts_index_append(ctypes.byref(shape()), FAKE, FAKE, FAKE, 0, 1, None)
    assert st == 4                                   # QASC_ERR_CUDA
    assert b"no usable CUDA device" in lib.qasc_last_error()


def _documented_select_rules(B, Hq, Hkv, n, n_cap, K, sink, local, vmin):
    """The argument rules qasc.h states for a select call, written out."""
    if B < 1 or Hq < 1 or Hkv < 1 or Hq % Hkv or Hq > 64:
        return False
    if Hq // Hkv not in (1, 2, 4, 8):
        return False
    if not (1 <= n_cap < 2 ** 24 and 1 <= n <= n_cap):
        return False
    if B * Hkv > 65535 or B * Hkv * n_cap >= 2 ** 31:
        return False
    if sink < 0 or local < 0 or vmin < 1:
        return False
    nc = max(n - local, sink) - sink if n > sink else 0
    return 0 <= K <= nc


def test_size_query_accepts_exactly_the_documented_arguments(lib):
    # A valid configuration is drawn, then (half the time) one field is
    # pushed to or across a boundary the header states; the size query must
    # accept (non-zero, or 0 with no message) exactly what the rules allow,
    # and reject the rest with a message.
    import random
    rng = random.Random(20261202)
    seen = {True: 0, False: 0}
    for _ in range(3000):
        Hkv = rng.choice((1, 2, 4, 8))
        Hq = Hkv * rng.choice((1, 2, 4, 8))
        B = rng.choice((1, 2, 4, 64))
        n_cap = rng.choice((1, 300, 4096, 2 ** 17))
        n = rng.randint(1, n_cap)
        sink, local, vmin = rng.choice((0, 4)), rng.choice((0, 256)), 1
        nc = max(n - local, sink) - sink if n > sink else 0
        K = rng.randint(0, nc)
        if rng.random() < 0.5:
            field = rng.randrange(9)
            d = rng.choice((-1, 0, 1))
            if field == 0:
                B = rng.choice((0, 65535 // Hkv + d, (2 ** 31 - 1) // (Hkv * n_cap) + d))
            elif field == 1:
                Hq = rng.choice((0, 3 * Hkv, 16 * Hkv, 64 + d, Hkv - 1))
            elif field == 2:
                Hkv = rng.choice((0, -1, 3, Hq + 1))
            elif field == 3:
                n_cap = rng.choice((0, 2 ** 24 + d, n + d))
            elif field == 4:
                n = rng.choice((0, n_cap + d, sink + local + d))
            elif field == 5:
                K = rng.choice((-1, nc + d))
            elif field == 6:
                sink = rng.choice((-1, n + d))
            elif field == 7:
                local = rng.choice((-1, n + d))
            else:
                vmin = rng.choice((0, -1, 2))
        s = _lib.qasc_shape(B, Hq, Hkv, 128, 32, 0, n, n_cap)
        p = _lib.qasc_ts_params(K, sink, local, vmin)
        got = lib.ts_select_workspace_bytes(ctypes.byref(s), ctypes.byref(p))
        msg = lib.qasc_last_error()
        accepted = got > 0 or msg == b""
        want = _documented_select_rules(B, Hq, Hkv, n, n_cap, K, sink, local, vmin)
        assert accepted == want, (B, Hq, Hkv, n, n_cap, K, sink, local, vmin, got, msg)
        if not accepted:
            assert got == 0 and msg
        seen[want] += 1
    assert min(seen.values()) >= 500, seen


def test_snapkv_size_query_accepts_exactly_the_documented_parameters(lib):
    # The SnapKV rules qasc.h states (c >= 1, window >= 1, pool_k odd in
    # [1, 65], Gq * window <= 128) on a valid shape, each pushed across its
    # boundary half the time.
    import random
    rng = random.Random(7)
    seen = {True: 0, False: 0}
    for _ in range(2000):
        Hkv = rng.choice((1, 2, 8))
        gq = rng.choice((1, 2, 4, 8))
        c = rng.choice((1, 64, 4096))
        window = rng.randint(1, 128 // gq)
        pool_k = rng.choice((1, 3, 5, 65))
        if rng.random() < 0.5:
            field, d = rng.randrange(3), rng.choice((-1, 0, 1))
            if field == 0:
                c = rng.choice((0, -1))
            elif field == 1:
                window = rng.choice((0, -1, 128 // gq + d))
            else:
                pool_k = rng.choice((0, -1, 2, 4, 64, 65 + d, 67))
        s = _lib.qasc_shape(2, Hkv * gq, Hkv, 128, 32, 0, 5000, 5000)
        sp = _lib.qasc_snap_params(c, window, pool_k, 0)
        got = lib.snapkv_workspace_bytes(ctypes.byref(s), ctypes.byref(sp))
        msg = lib.qasc_last_error()
        want = c >= 1 and window >= 1 and pool_k >= 1 and pool_k % 2 == 1 and pool_k <= 65 and gq * window <= 128
        assert (got > 0) == want, (gq, c, window, pool_k, got, msg)
        assert want or msg
        seen[want] += 1
    assert min(seen.values()) >= 300, seen


def test_nvtx_variant_builds_beside_the_default(lib):
    # -DQASC_NVTX wraps each call that enqueues work in an NVTX range; it
    # builds into its own library with the same exports and leaves the
    # default library free of NVTX code.
    import subprocess
    path = qbuild.build(nvtx=True)
    assert path != _lib.LIB_PATH and os.path.exists(path)

    def syms(p, *flags):
        return subprocess.run(["nm", *flags, p], capture_output=True, text=True).stdout

    exported = sorted(l.split()[-1] for l in syms(path, "-D", "--defined-only").splitlines() if " T " in l)
    assert exported == declared_symbols()
    assert "nvtx" in syms(path).lower()
    assert "nvtx" not in syms(_lib.LIB_PATH).lower()
    nv = _lib.load(path)
    s, p = shape(), params()
    assert nv.ts_select_workspace_bytes(ctypes.byref(s), ctypes.byref(p)) == \
        lib.ts_select_workspace_bytes(ctypes.byref(s), ctypes.byref(p))


def test_paged_calls_accept_exactly_the_documented_pools(lib):
    # With no device, a paged call whose arguments pass every check stops at
    # the device lookup (QASC_ERR_CUDA); one that breaks a rule qasc.h
    # states for the pool is refused before it (QASC_ERR_INVALID_ARG).
    # The fake pointers must never reach a kernel, so skip on a GPU host.
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    import random
    rng = random.Random(31)
    seen = {True: 0, False: 0}
    for _ in range(1500):
        Hkv = rng.choice((1, 2, 8))
        P = rng.choice((64, 256, 1024, 65536))
        pages = rng.choice((1, 3, 16))
        num_pages = rng.choice((1, 40, (2 ** 31 - 1) // (Hkv * P)))
        n_cap = pages * P
        if rng.random() < 0.5:
            field, d = rng.randrange(4), rng.choice((-1, 1))
            if field == 0:
                P = rng.choice((0, 32, 63, 65, 96, 131072, P + d))
            elif field == 1:
                pages = rng.choice((0, -1))
            elif field == 2:
                num_pages = rng.choice((0, -1, (2 ** 31) // (Hkv * P) + rng.choice((0, 1)), 2 ** 62))
            else:
                n_cap = n_cap + d
        want = (64 <= P <= 65536 and P & (P - 1) == 0 and pages >= 1 and num_pages >= 1
                and n_cap == pages * P and num_pages * Hkv * P < 2 ** 31)
        if not (1 <= n_cap < 2 ** 24 and 2 * Hkv * n_cap < 2 ** 31):
            continue                                           # a shape rule, not a pool rule
        s = _lib.qasc_shape(2, 4 * Hkv, Hkv, 128, 32, 0, n_cap, n_cap)
        cache = _lib.qasc_paged_cache(FAKE.value, P, pages, num_pages)
        st = lib.ts_index_append_paged(ctypes.byref(s), ctypes.byref(cache), FAKE, FAKE, FAKE, 0, 1, None)
        assert st == (4 if want else 1), (P, pages, num_pages, n_cap, st, lib.qasc_last_error())
        seen[want] += 1
    assert min(seen.values()) >= 300, seen


def test_ring_flush_accepts_exactly_the_documented_rings(lib):
    # Same method as the pool test: valid arguments reach the device lookup
    # (QASC_ERR_CUDA with no device), a ring or range that breaks a stated
    # rule (count <= R <= 2^24, tokens within n_cap) is refused before it.
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    import random
    rng = random.Random(41)
    P, pages = 256, 8
    n_cap = P * pages
    s = _lib.qasc_shape(2, 8, 2, 128, 32, 0, n_cap, n_cap)
    cache = _lib.qasc_paged_cache(FAKE.value, P, pages, 64)
    seen = {True: 0, False: 0}
    for _ in range(1000):
        R = rng.choice((-1, 0, 1, 16, 255, 256, 320, 2 ** 24, 2 ** 24 + 1))
        count = rng.choice((0, 1, 16, 256, 320, R, R + 1))
        start = rng.choice((0, 100, n_cap - count, n_cap - count + 1, -1))
        ring = _lib.qasc_local_ring(FAKE.value, FAKE.value, R)
        st = lib.ts_ring_flush(ctypes.byref(s), ctypes.byref(cache), ctypes.byref(ring), FAKE, FAKE, FAKE, FAKE,
                               start, count, None)
        rows_ok = 0 <= start <= n_cap and 0 <= count <= n_cap - start
        want = 1 <= R <= 2 ** 24 and count <= R and rows_ok
        if want and count == 0:
            assert st in (0, 4), (R, count, start, st)            # an empty flush may return before the lookup
        else:
            assert st == (4 if want else 1), (R, count, start, st, lib.qasc_last_error())
        seen[want] += 1
    assert min(seen.values()) >= 150, seen


def test_expand_size_queries_follow_the_documented_rules(lib):
    # rows in [1, 65535] and radius in [0, 2^20] (qasc.h); the capacity is
    # min(|C|, (2 radius + 1) K) whenever the arguments are accepted.
    import random
    rng = random.Random(53)
    seen = {True: 0, False: 0}
    for _ in range(1500):
        n = rng.choice((261, 300, 5000, 131072))
        nc = max(n - 256, 4) - 4
        K = rng.choice((0, 1, nc // 7, nc))
        rows = rng.choice((-1, 0, 1, 32, 65535, 65536))
        radius = rng.choice((-1, 0, 1, 40, 2 ** 20, 2 ** 20 + 1))
        s = _lib.qasc_shape(1, 1, 1, 128, 32, 0, n, n)
        p = params(K=K)
        ws = lib.ts_expand_workspace_bytes(ctypes.byref(s), ctypes.byref(p), rows)
        assert (ws > 0 or lib.qasc_last_error() == b"") == (1 <= rows <= 65535), (n, K, rows, ws)
        cap = lib.ts_expand_capacity(ctypes.byref(s), ctypes.byref(p), radius)
        ok = 0 <= radius <= 2 ** 20
        if ok:
            assert lib.qasc_last_error() == b"" and cap == min(nc, (2 * radius + 1) * K), (n, K, radius, cap)
        else:
            assert cap == 0 and lib.qasc_last_error()
        seen[ok and 1 <= rows <= 65535] += 1
    assert min(seen.values()) >= 300, seen
