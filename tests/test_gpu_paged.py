"""GPU parity of the paged cache and the circular local buffer
(ts_index_append_paged, ts_score_vote_select_paged, ts_sparse_attn_paged,
ts_ring_flush), against the fp64 oracle and against the contiguous calls.

  index      bit-exact against the oracle's rows of the logical cache
  selection  equal to the contiguous call's set; the band rule against the
             oracle scoring the pool through its own page mapping
  out/lse    equal (bit for bit) to the contiguous call; max-abs and relative
             L2 <= 1e-3 against the oracle on the rows it reads through the
             pages and the ring
  flush      K / V rows bit copies, index rows bit-exact, every other row of
             the pools untouched

Table entries that a call must not touch are poisoned (outside the pool): a
read of one would be reported by qasc_device_error().
"""

import numpy as np
import pytest
import torch

import synth
from oracle import paged as opg
from oracle import tokenselect as ots
from tests.parity_rules import check_attention, check_selection

pytestmark = pytest.mark.gpu

qasc = pytest.importorskip("query_aware_sparse_compressed_gb300")
D = synth.DECODE_CONFIGS
POISON = -5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qasc._lib.load()


def to_pool(cache, P, seed, extra=3):
    """cache [B, Hkv, n_cap, w] on the device -> (pool [num_pages, Hkv, P, w],
    table [B, pps] int32): the logical pages in a seeded random order among
    `extra` spare pages of junk."""
    B, Hkv, n_cap, w = cache.shape
    pps = -(-n_cap // P)
    if pps * P != n_cap:
        cache = torch.cat([cache, torch.zeros((B, Hkv, pps * P - n_cap, w), dtype=cache.dtype, device=cache.device)],
                          dim=2)
    pages = cache.reshape(B, Hkv, pps, P, w).permute(0, 2, 1, 3, 4).reshape(B * pps, Hkv, P, w)
    num_pages = B * pps + extra
    g = torch.Generator().manual_seed(seed)
    slot = torch.randperm(num_pages, generator=g)[:B * pps]
    gd = torch.Generator(device=cache.device).manual_seed(seed)
    pool = (torch.randn((num_pages, Hkv, P, w), generator=gd, device=cache.device) * 100).to(cache.dtype)
    pool[slot.to(cache.device)] = pages
    return pool.contiguous(), slot.reshape(B, pps).to(torch.int32).to(cache.device)


def poison_from(table, first_page):
    t = table.clone()
    if first_page < t.shape[1]:
        t[:, first_page:] = POISON
    return t


def cdiv(a, b):
    return -(-a // b)


def gpu_index(K, W, n, Hq):
    B, Hkv, n_cap, _ = K.shape
    index = torch.zeros((B, Hkv, n_cap, 32), dtype=torch.bfloat16, device="cuda")
    qasc.ts_index_append(K, W, index, 0, n, Hq=Hq, n=n)
    return index


def select_contig(q, W, index, n, K, sink, local):
    B, Hq, _ = q.shape
    _, Hkv, n_cap, _ = index.shape
    sel = torch.empty((B, K), dtype=torch.int32, device="cuda")
    ws = qasc.alloc_workspace(qasc.ts_select_workspace_bytes(B, Hq, Hkv, n, n_cap, K, sink, local))
    qasc.ts_score_vote_select(q, W, index, sel, ws, n=n, K=K, sink=sink, local=local)
    return sel


def select_paged(q, W, index_pool, table, n, K, sink, local):
    B, Hq, _ = q.shape
    Hkv, P = index_pool.shape[1], index_pool.shape[2]
    n_cap = table.shape[1] * P
    sel = torch.empty((B, K), dtype=torch.int32, device="cuda")
    ws = qasc.alloc_workspace(qasc.ts_select_workspace_bytes(B, Hq, Hkv, n, n_cap, K, sink, local))
    qasc.ts_score_vote_select_paged(q, W, index_pool, table, sel, ws, n=n, K=K, sink=sink, local=local)
    return sel


def attn_ws(q, Hkv, n, n_cap, Ksel, sink, local):
    B, Hq, _ = q.shape
    return qasc.alloc_workspace(qasc.ts_attn_workspace_bytes(B, Hq, Hkv, n, n_cap, Ksel, sink, local))


SELECT_CASES = [
    ("tiny", D["tiny"], 64),
    ("tiny", D["tiny"], 1024),
    ("llama8b-6000", D["llama8b"].with_(B=2, n=6000), 128),
    ("llama8b-6000", D["llama8b"].with_(B=2, n=6000), 256),
    ("llama70b-5003", D["llama70b"].with_(B=2, n=5003), 64),
    ("gq1", D["tiny"].with_(Hq=4, Hkv=4, n=3001), 512),
]


@pytest.mark.parametrize("name,cfg,P", SELECT_CASES, ids=["%s-P%d" % (c[0], c[2]) for c in SELECT_CASES])
def test_paged_select(name, cfg, P):
    x_cpu = synth.decode_layer(cfg, 0)
    x = {k: v.cuda() for k, v in x_cpu.items()}
    n, sink, local = cfg.n, cfg.sink, cfg.local
    K = ots.budget_tokens(n, cfg.budget_permille, sink, local)
    _, _, c1, _ = ots.regions(n, sink, local)
    index = gpu_index(x["K"], x["W"], n, cfg.Hq)
    pool, table = to_pool(index, P, seed=P + n)
    table_sel = poison_from(table, cdiv(c1, P))          # pages wholly at or above c1 are never read
    sel_p = select_paged(x["q"], x["W"], pool, table_sel, n, K, sink, local)
    sel_c = select_contig(x["q"], x["W"], index, n, K, sink, local)
    qasc.qasc_device_error()
    assert torch.equal(sel_p, sel_c)
    # the oracle reads the pool through its own page mapping
    idx_logical = opg.logical_rows(synth.to_f64(pool.cpu()), table.cpu().numpy(), P, n)
    q64, W64 = synth.to_f64(x_cpu["q"]), synth.to_f64(x_cpu["W"])
    _, info = ots.select(q64, W64, idx_logical, n, K, sink, local)
    for b in range(cfg.B):
        check_selection(sel_p.cpu().numpy()[b].astype(np.int64), info["scores"][b], info["theta"][b], info["c0"], K)


@pytest.mark.parametrize("P", [128, 512])
def test_paged_per_head_select(P):
    cfg = D["llama8b"].with_(B=2, n=6000)
    x_cpu = synth.decode_layer(cfg, 0)
    x = {k: v.cuda() for k, v in x_cpu.items()}
    n, sink, local = cfg.n, cfg.sink, cfg.local
    K = ots.budget_tokens(n, cfg.budget_permille, sink, local)
    _, _, c1, _ = ots.regions(n, sink, local)
    index = gpu_index(x["K"], x["W"], n, cfg.Hq)
    pool, table = to_pool(index, P, seed=P)
    B, Hq, Hkv, n_cap = cfg.B, cfg.Hq, cfg.Hkv, index.shape[2]
    ws = qasc.alloc_workspace(max(qasc.ts_head_select_workspace_bytes(B, Hq, Hkv, n, n_cap, K, sink, local),
                                  qasc.ts_head_select_workspace_bytes(B, Hq, Hkv, n, table.shape[1] * P, K, sink,
                                                                      local)))
    sel_c = torch.empty((B, Hkv, K), dtype=torch.int32, device="cuda")
    sel_p = torch.empty_like(sel_c)
    qasc.ts_score_select_per_head(x["q"], x["W"], index, sel_c, ws, n=n, K=K, sink=sink, local=local)
    qasc.ts_score_select_per_head_paged(x["q"], x["W"], pool, poison_from(table, cdiv(c1, P)), sel_p, ws, n=n, K=K,
                                        sink=sink, local=local)
    qasc.qasc_device_error()
    assert torch.equal(sel_p, sel_c)


@pytest.mark.parametrize("P", [64, 256])
def test_paged_append_bit_exact(P):
    cfg = D["llama8b"].with_(B=2, n=5000)
    x_cpu = synth.decode_layer(cfg, 0)
    n = cfg.n
    K_pool, table = to_pool(x_cpu["K"].cuda(), P, seed=7)
    idx_pool = (torch.randn((K_pool.shape[0], cfg.Hkv, P, 32)) * 50).to(torch.bfloat16).cuda()
    before = idx_pool.clone()
    W = x_cpu["W"].cuda()
    qasc.ts_index_append_paged(K_pool, W, idx_pool, table, 0, 1777, Hq=cfg.Hq, n=n)   # a bulk append...
    for t in range(1777, 1777 + 5):                                                    # ...single rows...
        qasc.ts_index_append_paged(K_pool, W, idx_pool, table, t, 1, Hq=cfg.Hq, n=n)
    qasc.ts_index_append_paged(K_pool, W, idx_pool, table, 1782, n - 1782, Hq=cfg.Hq, n=n)   # ...and the rest
    qasc.qasc_device_error()
    got = opg.logical_rows(synth.to_f64(idx_pool.cpu()), table.cpu().numpy(), P, n)
    want = ots.index_rows(synth.to_f64(x_cpu["K"][:, :, :n]), synth.to_f64(x_cpu["W"]))
    assert np.array_equal(got, want)
    # rows of tokens >= n and of spare pages are untouched
    written = torch.zeros(idx_pool.shape[:3], dtype=torch.bool)
    tb = table.cpu()
    for b in range(cfg.B):
        for t in range(n):
            written[tb[b, t // P], :, t % P] = True
    assert torch.equal(idx_pool.cpu()[~written], before.cpu()[~written])


def _ring_of(cache, R, n):
    """[B, Hkv, R, d] ring holding tokens [n - R, n) of cache at slot t mod R."""
    B, Hkv, _, d = cache.shape
    ring = torch.empty((B, Hkv, R, d), dtype=cache.dtype, device=cache.device)
    for t in range(n - R, n):
        ring[:, :, t % R] = cache[:, :, t]
    return ring


@pytest.mark.parametrize("per_kv_head", [False, True], ids=["shared", "per-kv-head"])
@pytest.mark.parametrize("ring", [False, True], ids=["pages", "pages+ring"])
@pytest.mark.parametrize("P", [64, 256])
def test_paged_attention(P, ring, per_kv_head):
    cfg = D["llama8b"].with_(B=2, n=6000)
    x_cpu = synth.decode_layer(cfg, 0)
    x = {k: v.cuda() for k, v in x_cpu.items()}
    n, sink, local = cfg.n, cfg.sink, cfg.local
    _, _, _, local_start = ots.regions(n, sink, local)
    Ksel = 700
    rows = cfg.B * cfg.Hkv if per_kv_head else cfg.B
    S = synth.random_selection(rows, n, Ksel, sink, local, 11 + P).cuda()
    S = S.reshape(cfg.B, cfg.Hkv, Ksel) if per_kv_head else S
    g = torch.Generator().manual_seed(3)
    lengths = torch.randint(1, Ksel + 1, S.shape[:-1], generator=g, dtype=torch.int32).cuda() if per_kv_head else None
    n_cap = x["K"].shape[2]

    out_c = torch.empty((cfg.B, cfg.Hq, 128), dtype=torch.float32, device="cuda")
    lse_c = torch.empty((cfg.B, cfg.Hq), dtype=torch.float32, device="cuda")
    qasc.ts_sparse_attn_ex(x["q"], x["K"], x["V"], S, out_c, attn_ws(x["q"], cfg.Hkv, n, n_cap, Ksel, sink, local),
                           n=n, sink=sink, local=local, lengths=lengths, per_kv_head=per_kv_head, lse=lse_c)

    K_pool, table = to_pool(x["K"], P, seed=5)
    V_pool, _ = to_pool(x["V"], P, seed=5)
    R = 300
    ring_kv = (_ring_of(x["K"], R, n), _ring_of(x["V"], R, n)) if ring else None
    # pages past n never hold a read token; with the ring, neither do the pages of the local window
    table_a = poison_from(table, cdiv(local_start, P) if ring else cdiv(n, P))
    out_p = torch.empty_like(out_c)
    lse_p = torch.empty_like(lse_c)
    qasc.ts_sparse_attn_paged(x["q"], K_pool, V_pool, table_a, S, out_p,
                              attn_ws(x["q"], cfg.Hkv, n, table.shape[1] * P, Ksel, sink, local), n=n, sink=sink,
                              local=local, ring=ring_kv, lengths=lengths, per_kv_head=per_kv_head, lse=lse_p)
    qasc.qasc_device_error()
    assert torch.equal(out_p, out_c) and torch.equal(lse_p, lse_c)

    # the oracle on the rows it reads through the pages (and the ring)
    tb = table.cpu().numpy()
    K64 = opg.logical_rows(synth.to_f64(K_pool.cpu()), tb, P, n)
    V64 = opg.logical_rows(synth.to_f64(V_pool.cpu()), tb, P, n)
    if ring:
        K64 = opg.attended_rows(K64, synth.to_f64(ring_kv[0].cpu()), R, n, sink, local)
        V64 = opg.attended_rows(V64, synth.to_f64(ring_kv[1].cpu()), R, n, sink, local)
    q64 = synth.to_f64(x_cpu["q"])
    S_h = S.cpu().numpy().astype(np.int64)
    if per_kv_head:
        Ls = lengths.cpu().numpy()
        S_obj = np.empty(S_h.shape[:2], dtype=object)
        for b in range(cfg.B):
            for gg in range(cfg.Hkv):
                S_obj[b, gg] = S_h[b, gg, :Ls[b, gg]]
        ref, ref_lse = ots.sparse_attention_per_head(q64, K64, V64, S_obj, n, sink, local)
    else:
        ref, ref_lse = ots.sparse_attention(q64, K64, V64, S_h, n, sink, local)
    check_attention(out_p.cpu().numpy(), ref)
    check_attention(lse_p.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("start,count", [(0, 40), (4096 - 40, 40), (1000, 1)])
def test_ring_flush(start, count):
    cfg = D["llama8b"].with_(B=2, n=4096)
    x_cpu = synth.decode_layer(cfg, 0)
    K, V, W = (x_cpu[k].cuda() for k in ("K", "V", "W"))
    P, R = 64, 48
    K_pool, table = to_pool(torch.zeros_like(K), P, seed=9)
    V_pool, _ = to_pool(torch.zeros_like(V), P, seed=9)
    idx_pool = (torch.randn((K_pool.shape[0], cfg.Hkv, P, 32)) * 50).to(torch.bfloat16).cuda()
    pools_before = [p.clone() for p in (K_pool, V_pool, idx_pool)]
    ring_K = torch.zeros((cfg.B, cfg.Hkv, R, 128), dtype=torch.bfloat16, device="cuda")
    ring_V = torch.zeros_like(ring_K)
    for t in range(start, start + count):
        ring_K[:, :, t % R] = K[:, :, t]
        ring_V[:, :, t % R] = V[:, :, t]
    qasc.ts_ring_flush((ring_K, ring_V), W, K_pool, V_pool, idx_pool, table, start, count, n=cfg.n)
    qasc.qasc_device_error()
    tb = table.cpu().numpy()
    e = start + count
    sl = slice(start, e)
    assert np.array_equal(opg.logical_rows(synth.to_f64(K_pool.cpu()), tb, P, e)[:, :, sl],
                          synth.to_f64(x_cpu["K"][:, :, sl]))
    assert np.array_equal(opg.logical_rows(synth.to_f64(V_pool.cpu()), tb, P, e)[:, :, sl],
                          synth.to_f64(x_cpu["V"][:, :, sl]))
    want_idx = ots.index_rows(synth.to_f64(x_cpu["K"][:, :, sl]), synth.to_f64(x_cpu["W"]))
    assert np.array_equal(opg.logical_rows(synth.to_f64(idx_pool.cpu()), tb, P, e)[:, :, sl], want_idx)
    written = torch.zeros(K_pool.shape[:3], dtype=torch.bool)
    for b in range(cfg.B):
        for t in range(start, e):
            written[tb[b, t // P], :, t % P] = True
    for now, before in zip((K_pool, V_pool, idx_pool), pools_before):
        assert torch.equal(now.cpu()[~written], before.cpu()[~written])


def test_flush_then_select_and_attend_equals_contiguous():
    # A decode loop: the newest tokens live in the ring, older ones were
    # flushed into the pages in batches of 16; selection and attention over
    # pages + ring equal the contiguous calls on the whole cache.
    cfg = D["tiny"].with_(n=3000)
    x_cpu = synth.decode_layer(cfg, 0)
    x = {k: v.cuda() for k, v in x_cpu.items()}
    n, sink, local, P, R, batch = cfg.n, cfg.sink, cfg.local, 128, 256 + 32, 16
    K_pool, table = to_pool(torch.zeros_like(x["K"]), P, seed=2)
    V_pool, _ = to_pool(torch.zeros_like(x["V"]), P, seed=2)
    idx_pool = torch.zeros((K_pool.shape[0], cfg.Hkv, P, 32), dtype=torch.bfloat16, device="cuda")
    ring_K = torch.zeros((cfg.B, cfg.Hkv, R, 128), dtype=torch.bfloat16, device="cuda")
    ring_V = torch.zeros_like(ring_K)
    flushed = 0
    for t in range(n):                      # token t arrives in the ring
        ring_K[:, :, t % R] = x["K"][:, :, t]
        ring_V[:, :, t % R] = x["V"][:, :, t]
        # flush a batch once its first token is one step from entering the
        # candidates (it has arrived since local >= batch; it is still in the
        # ring since R >= local + batch)
        while flushed <= t + 1 - local:
            qasc.ts_ring_flush((ring_K, ring_V), x["W"], K_pool, V_pool, idx_pool, table, flushed, batch, n=n)
            flushed += batch
    assert flushed >= n - local
    K = ots.budget_tokens(n, cfg.budget_permille, sink, local)
    _, _, c1, local_start = ots.regions(n, sink, local)
    sel_p = select_paged(x["q"], x["W"], idx_pool, poison_from(table, cdiv(flushed, P)), n, K, sink, local)
    index = gpu_index(x["K"], x["W"], n, cfg.Hq)
    sel_c = select_contig(x["q"], x["W"], index, n, K, sink, local)
    qasc.qasc_device_error()
    assert torch.equal(sel_p, sel_c)
    n_cap = x["K"].shape[2]
    out_c = torch.empty((cfg.B, cfg.Hq, 128), dtype=torch.float32, device="cuda")
    qasc.ts_sparse_attn(x["q"], x["K"], x["V"], sel_c, out_c, attn_ws(x["q"], cfg.Hkv, n, n_cap, K, sink, local), n=n,
                        sink=sink, local=local)
    out_p = torch.empty_like(out_c)
    qasc.ts_sparse_attn_paged(x["q"], K_pool, V_pool, poison_from(table, cdiv(flushed, P)), sel_p, out_p,
                              attn_ws(x["q"], cfg.Hkv, n, table.shape[1] * P, K, sink, local), n=n, sink=sink,
                              local=local, ring=(ring_K, ring_V))
    qasc.qasc_device_error()
    assert torch.equal(out_p, out_c)


def test_table_entry_outside_the_pool_is_reported():
    cfg = D["tiny"].with_(n=3000)
    x = {k: v.cuda() for k, v in synth.decode_layer(cfg, 0).items()}
    n, sink, local, P = cfg.n, cfg.sink, cfg.local, 256
    K = ots.budget_tokens(n, cfg.budget_permille, sink, local)
    index = gpu_index(x["K"], x["W"], n, cfg.Hq)
    pool, table = to_pool(index, P, seed=1)
    bad = table.clone()
    bad[0, 3] = pool.shape[0] + 7            # a page the select reads
    select_paged(x["q"], x["W"], pool, bad, n, K, sink, local)
    with pytest.raises(qasc.QascError) as e:
        qasc.qasc_device_error()
    assert e.value.status == 6
    select_paged(x["q"], x["W"], pool, table, n, K, sink, local)
    qasc.qasc_device_error()                 # the error word was cleared; a clean table reports nothing
    K_pool, ktable = to_pool(x["K"], P, seed=1)
    idx2 = torch.zeros_like(pool)
    bad = ktable.clone()
    bad[0, 1] = -1
    qasc.ts_index_append_paged(K_pool, x["W"], idx2, bad, 0, n, Hq=cfg.Hq, n=n)
    with pytest.raises(qasc.QascError) as e:
        qasc.qasc_device_error()
    assert e.value.status == 6


@pytest.mark.slow
def test_paged_full_size_128k_b4():
    cfg = D["llama8b_long"]
    x = synth.decode_layer(cfg, 0, device="cuda")
    n, sink, local, P = cfg.n, cfg.sink, cfg.local, 256
    K = ots.budget_tokens(n, cfg.budget_permille, sink, local)
    _, _, c1, local_start = ots.regions(n, sink, local)
    index = gpu_index(x["K"], x["W"], n, cfg.Hq)
    sel_c = select_contig(x["q"], x["W"], index, n, K, sink, local)
    idx_pool, table = to_pool(index, P, seed=4)
    del index
    sel_p = select_paged(x["q"], x["W"], idx_pool, poison_from(table, cdiv(c1, P)), n, K, sink, local)
    qasc.qasc_device_error()
    assert torch.equal(sel_p, sel_c)
    del idx_pool
    n_cap = x["K"].shape[2]
    out_c = torch.empty((cfg.B, cfg.Hq, 128), dtype=torch.float32, device="cuda")
    qasc.ts_sparse_attn(x["q"], x["K"], x["V"], sel_c, out_c, attn_ws(x["q"], cfg.Hkv, n, n_cap, K, sink, local), n=n,
                        sink=sink, local=local)
    R = 512
    ring_kv = (_ring_of(x["K"], R, n), _ring_of(x["V"], R, n))
    K_pool, table = to_pool(x["K"], P, seed=6)
    del x["K"]
    V_pool, _ = to_pool(x["V"], P, seed=6)
    del x["V"]
    out_p = torch.empty_like(out_c)
    qasc.ts_sparse_attn_paged(x["q"], K_pool, V_pool, poison_from(table, cdiv(local_start, P)), sel_p, out_p,
                              attn_ws(x["q"], cfg.Hkv, n, table.shape[1] * P, K, sink, local), n=n, sink=sink,
                              local=local, ring=ring_kv)
    qasc.qasc_device_error()
    assert torch.equal(out_p, out_c)
