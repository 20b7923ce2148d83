"""GPU parity of the neighbour expansion and of attention over sets with
lengths (ts_expand_neighbors, ts_sparse_attn_ex), against the fp64 oracle.

  expansion  bit-exact: the in-use entries equal the oracle's union, the
             length its size, the unused entries repeat the last entry
  out/lse    max-abs <= 1e-3 and relative L2 <= 1e-3 against the oracle on the
             expanded (ragged) sets; unused entries never matter
"""

import numpy as np
import pytest
import torch

import synth
from oracle import tokenselect as ots
from tests.parity_rules import check_attention

pytestmark = pytest.mark.gpu

qasc = pytest.importorskip("query_aware_sparse_compressed_gb300")
D = synth.DECODE_CONFIGS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qasc._lib.load()


def gpu_expand(sel, radius, n, sink, local):
    """sel [..., K] on the device -> (sel_out [..., cap], lengths [...])."""
    K = sel.shape[-1]
    cap = max(1, qasc.ts_expand_capacity(n, K, radius, sink, local))
    lead = tuple(sel.shape[:-1])
    out = torch.full(lead + (cap,), -7, dtype=torch.int32, device="cuda")
    lengths = torch.full(lead, -1, dtype=torch.int32, device="cuda")
    rows = out.numel() // cap
    ws = qasc.alloc_workspace(qasc.ts_expand_workspace_bytes(n, K, rows, sink, local))
    qasc.ts_expand_neighbors(sel.contiguous(), radius, out, lengths, ws, n=n, sink=sink, local=local)
    return out, lengths


def check_expansion(sel_h, out_h, len_h, radius, n, sink, local):
    rows = sel_h.reshape(-1, sel_h.shape[-1])
    outs = out_h.reshape(-1, out_h.shape[-1])
    lens = len_h.reshape(-1)
    ref = []
    for r in range(rows.shape[0]):
        want = ots.expand_neighbors(rows[r], radius, n, sink, local)
        L = int(lens[r])
        assert L == len(want), (r, L, len(want))
        assert np.array_equal(outs[r, :L], want), r
        if L < outs.shape[1]:
            assert np.all(outs[r, L:] == (want[-1] if L else sink)), r
        ref.append(want)
    return ref


@pytest.mark.parametrize("radius", [0, 1, 2, 5, 40])
def test_expansion_random_sets(radius):
    n, sink, local, rows, K = 5000, 4, 256, 6, 300
    S = synth.random_selection(rows, n, K, sink, local, 10 + radius)
    out, lengths = gpu_expand(S.cuda(), radius, n, sink, local)
    qasc.qasc_device_error()
    check_expansion(S.numpy(), out.cpu().numpy(), lengths.cpu().numpy(), radius, n, sink, local)


def test_expansion_edges_and_dense_sets():
    n, sink, local = 700, 4, 256
    _, c0, c1, _ = ots.regions(n, sink, local)
    cases = [np.array([c0]), np.array([c1 - 1]), np.array([c0, c0 + 1, c1 - 2, c1 - 1]),
             np.arange(c0, c1, 2), np.arange(c0, c1)]
    for S in cases:
        t = torch.from_numpy(S.astype(np.int32))[None]
        for radius in (1, 3, 1000):
            out, lengths = gpu_expand(t.cuda(), radius, n, sink, local)
            check_expansion(t.numpy(), out.cpu().numpy(), lengths.cpu().numpy(), radius, n, sink, local)


@pytest.mark.parametrize("radius", [0, 3, 7000])
def test_expansion_tokens_outside_candidates_and_duplicates(radius):
    # Sink and local tokens add their neighbours within C; duplicates add
    # nothing twice; 4096 candidates apart is one chunk boundary.
    n, sink, local = 9000, 4, 256
    _, c0, c1, _ = ots.regions(n, sink, local)
    S = np.array([[0, 2, c0 + 10, c1 + 1],
                  [1, 3, c1, n - 1],
                  [c0 - 1, c0 + 4095, c0 + 4096, c1 + 2],
                  [c0 + 100, c0 + 100, c0 + 101, c0 + 5000]], dtype=np.int32)
    t = torch.from_numpy(S)
    out, lengths = gpu_expand(t.cuda(), radius, n, sink, local)
    qasc.qasc_device_error()
    check_expansion(S, out.cpu().numpy(), lengths.cpu().numpy(), radius, n, sink, local)


@pytest.mark.parametrize("radius", [1, 4])
def test_expansion_many_chunks_per_kv_head_rows(radius):
    n, sink, local, B, Hkv, K = 40000, 4, 256, 2, 8, 4000
    S = synth.random_selection(B * Hkv, n, K, sink, local, 77 + radius).reshape(B, Hkv, K)
    out, lengths = gpu_expand(S.cuda(), radius, n, sink, local)
    qasc.qasc_device_error()
    assert out.shape[:2] == (B, Hkv) and lengths.shape == (B, Hkv)
    check_expansion(S.numpy(), out.cpu().numpy(), lengths.cpu().numpy(), radius, n, sink, local)


def _attn_ex(x, sel, lengths, n, sink, local, per_kv_head):
    B, Hq, _ = x["q"].shape
    _, Hkv, n_cap, _ = x["K"].shape
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    ws = qasc.alloc_workspace(qasc.ts_attn_workspace_bytes(B, Hq, Hkv, n, n_cap, sel.shape[-1], sink, local))
    qasc.ts_sparse_attn_ex(x["q"], x["K"], x["V"], sel, out, ws, n=n, sink=sink, local=local, lengths=lengths,
                           per_kv_head=per_kv_head, lse=lse)
    return out, lse


def _select(x, n, K, sink, local, per_head):
    B, Hq, _ = x["q"].shape
    _, Hkv, n_cap, _ = x["K"].shape
    index = torch.zeros((B, Hkv, n_cap, 32), dtype=torch.bfloat16, device="cuda")
    qasc.ts_index_append(x["K"], x["W"], index, 0, n, Hq=Hq, n=n)
    if per_head:
        sel = torch.empty((B, Hkv, K), dtype=torch.int32, device="cuda")
        ws = qasc.alloc_workspace(qasc.ts_head_select_workspace_bytes(B, Hq, Hkv, n, n_cap, K, sink, local))
        qasc.ts_score_select_per_head(x["q"], x["W"], index, sel, ws, n=n, K=K, sink=sink, local=local)
    else:
        sel = torch.empty((B, K), dtype=torch.int32, device="cuda")
        ws = qasc.alloc_workspace(qasc.ts_select_workspace_bytes(B, Hq, Hkv, n, n_cap, K, sink, local))
        qasc.ts_score_vote_select(x["q"], x["W"], index, sel, ws, n=n, K=K, sink=sink, local=local)
    return sel


@pytest.mark.parametrize("per_head", [False, True], ids=["voting", "per-kv-head"])
@pytest.mark.parametrize("radius", [1, 3])
def test_select_expand_attend(per_head, radius):
    cfg = D["llama8b"].with_(B=2, n=6000)
    x_cpu = synth.decode_layer(cfg, 0)
    x = {k: v.cuda() for k, v in x_cpu.items()}
    n, sink, local = cfg.n, cfg.sink, cfg.local
    K = ots.budget_tokens(n, 100, sink, local)
    sel = _select(x, n, K, sink, local, per_head)
    out_sel, lengths = gpu_expand(sel, radius, n, sink, local)
    out, lse = _attn_ex(x, out_sel, lengths, n, sink, local, per_head)
    qasc.qasc_device_error()
    ref_sets = check_expansion(sel.cpu().numpy(), out_sel.cpu().numpy(), lengths.cpu().numpy(), radius, n, sink,
                               local)
    q64, K64, V64 = (synth.to_f64(x_cpu[k]) for k in ("q", "K", "V"))
    if per_head:
        S = np.empty((cfg.B, cfg.Hkv), dtype=object)
        for i, r in enumerate(ref_sets):
            S[i // cfg.Hkv, i % cfg.Hkv] = r
        ref, ref_lse = ots.sparse_attention_per_head(q64, K64[:, :, :n], V64[:, :, :n], S, n, sink, local)
    else:
        ref, ref_lse = ots.sparse_attention(q64, K64[:, :, :n], V64[:, :, :n], ref_sets, n, sink, local)
    check_attention(out.cpu().numpy(), ref)
    check_attention(lse.cpu().numpy(), ref_lse)


def test_unused_entries_are_masked():
    cfg = D["tiny"].with_(n=3000)
    x = {k: v.cuda() for k, v in synth.decode_layer(cfg, 0).items()}
    n, sink, local = cfg.n, cfg.sink, cfg.local
    S = synth.random_selection(cfg.B, n, 200, sink, local, 3).cuda()
    cap = 500
    clean = torch.empty((cfg.B, cap), dtype=torch.int32, device="cuda")
    clean[:, :200] = S
    clean[:, 200:] = S[:, -1:]
    junk = clean.clone()
    g = torch.Generator(device="cpu").manual_seed(4)
    junk[:, 200:] = torch.randint(-10**9, 10**9, (cfg.B, cap - 200), generator=g, dtype=torch.int32).cuda()
    lengths = torch.full((cfg.B,), 200, dtype=torch.int32, device="cuda")
    o1, l1 = _attn_ex(x, clean, lengths, n, sink, local, False)
    o2, l2 = _attn_ex(x, junk, lengths, n, sink, local, False)
    o3, l3 = _attn_ex(x, S, None, n, sink, local, False)
    qasc.qasc_device_error()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    check_attention(o1.cpu().numpy(), o3.cpu().numpy())


def test_ex_without_lengths_equals_sparse_attn():
    cfg = D["llama8b"].with_(B=2, n=5000)
    x = {k: v.cuda() for k, v in synth.decode_layer(cfg, 0).items()}
    S = synth.random_selection(cfg.B, cfg.n, 700, cfg.sink, cfg.local, 6).cuda()
    out_ex, _ = _attn_ex(x, S, None, cfg.n, cfg.sink, cfg.local, False)
    out = torch.empty_like(out_ex)
    ws = qasc.alloc_workspace(qasc.ts_attn_workspace_bytes(cfg.B, cfg.Hq, cfg.Hkv, cfg.n, cfg.n, 700))
    qasc.ts_sparse_attn(x["q"], x["K"], x["V"], S, out, ws, n=cfg.n)
    assert torch.equal(out, out_ex)


@pytest.mark.slow
def test_expand_full_size_128k_b4():
    cfg = D["llama8b_long"]
    x = synth.decode_layer(cfg, 0, device="cuda")
    n, sink, local = cfg.n, cfg.sink, cfg.local
    K = ots.budget_tokens(n, cfg.budget_permille, sink, local)
    sel = _select(x, n, K, sink, local, False)
    out_sel, lengths = gpu_expand(sel, 1, n, sink, local)
    out, _ = _attn_ex(x, out_sel, lengths, n, sink, local, False)
    qasc.qasc_device_error()
    ref_sets = check_expansion(sel.cpu().numpy(), out_sel.cpu().numpy(), lengths.cpu().numpy(), 1, n, sink, local)
    b = 3
    q64 = synth.to_f64(x["q"][b:b + 1].cpu())
    K64 = synth.to_f64(x["K"][b:b + 1, :, :n].cpu())
    V64 = synth.to_f64(x["V"][b:b + 1, :, :n].cpu())
    ref, _ = ots.sparse_attention(q64, K64, V64, [ref_sets[b]], n, sink, local)
    check_attention(out[b:b + 1].cpu().numpy(), ref)
