"""GPU parity of the per-KV-head selection (TokenSelect without voting) and
its attention, against the fp64 oracle.

  S_g      the top-K rule on the group-summed score (parity_rules.check_topk,
           every key known to within Gq * 1e-4 * max|score|); exact on ties
  out/lse  max-abs <= 1e-3 and relative L2 <= 1e-3 against the oracle on the
           GPU's own sets and on the oracle's sets fed to the kernel
"""

import numpy as np
import pytest
import torch

import synth
from oracle import tokenselect as ots
from tests.parity_rules import SELECT_EPS_REL, check_attention, check_topk

pytestmark = pytest.mark.gpu

qasc = pytest.importorskip("query_aware_sparse_compressed_gb300")
D = synth.DECODE_CONFIGS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qasc._lib.load()


def gpu_index(x, n, Hq):
    B, Hkv, n_cap, _ = x["K"].shape
    index = torch.zeros((B, Hkv, n_cap, 32), dtype=torch.bfloat16, device="cuda")
    qasc.ts_index_append(x["K"], x["W"], index, 0, n, Hq=Hq, n=n)
    return index


def gpu_head_select(x, index, n, K, sink, local):
    B, Hq, _ = x["q"].shape
    _, Hkv, n_cap, _ = index.shape
    sel = torch.full((B, Hkv, max(K, 1)), -1, dtype=torch.int32, device="cuda")[:, :, :K].contiguous()
    ws = qasc.alloc_workspace(qasc.ts_head_select_workspace_bytes(B, Hq, Hkv, n, n_cap, K, sink, local))
    qasc.ts_score_select_per_head(x["q"], x["W"], index, sel, ws, n=n, K=K, sink=sink, local=local)
    return sel


def gpu_head_attn(x, sel, n, sink, local):
    B, Hq, _ = x["q"].shape
    _, Hkv, n_cap, _ = x["K"].shape
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    ws = qasc.alloc_workspace(qasc.ts_attn_workspace_bytes(B, Hq, Hkv, n, n_cap, sel.shape[2], sink, local))
    qasc.ts_sparse_attn_per_head(x["q"], x["K"], x["V"], sel, out, ws, n=n, sink=sink, local=local, lse=lse)
    return out, lse


def check_layer(x_cpu, x, n, K, sink, local, bs=None):
    """Select and attend on the GPU; the oracle checks the sequences bs."""
    B, Hq, _ = x["q"].shape
    Hkv = x["K"].shape[1]
    index = gpu_index(x, n, Hq)
    sel = gpu_head_select(x, index, n, K, sink, local)
    out, lse = gpu_head_attn(x, sel, n, sink, local)
    qasc.qasc_device_error()
    bs = range(B) if bs is None else bs
    sel_h = sel.cpu().numpy().astype(np.int64)
    for b in bs:
        q64 = synth.to_f64(x_cpu["q"][b:b + 1])
        K64 = synth.to_f64(x_cpu["K"][b:b + 1, :, :n])
        V64 = synth.to_f64(x_cpu["V"][b:b + 1, :, :n])
        W64 = synth.to_f64(x_cpu["W"])
        idx = ots.index_rows(K64, W64)
        S_ref, info = ots.select_per_kv_head(q64, W64, idx, n, K, sink, local)
        eps = (Hq // Hkv) * SELECT_EPS_REL * np.abs(info["scores"]).max()
        for g in range(Hkv):
            check_topk(sel_h[b, g], info["gsum"][0, g], K, eps, offset=info["c0"])
        # attention on the GPU's own sets, and on the oracle's sets
        ref, ref_lse = ots.sparse_attention_per_head(q64, K64, V64, sel_h[b:b + 1], n, sink, local)
        check_attention(out[b:b + 1].cpu().numpy(), ref)
        check_attention(lse[b:b + 1].cpu().numpy(), ref_lse)
        xb = {k: x[k][b:b + 1].contiguous() for k in ("q", "K", "V")}
        o2, l2 = gpu_head_attn(xb, torch.from_numpy(S_ref.astype(np.int32)).cuda(), n, sink, local)
        ref2, ref2_lse = ots.sparse_attention_per_head(q64, K64, V64, S_ref, n, sink, local)
        check_attention(o2.cpu().numpy(), ref2)
        check_attention(l2.cpu().numpy(), ref2_lse)
    return sel, out


@pytest.mark.parametrize("cfg", [
    D["tiny"],
    D["llama8b"].with_(B=2, n=6000),
    D["llama70b"].with_(B=2, n=5003),
    D["tiny"].with_(Hq=4, Hkv=4, n=3001),
    D["tiny"].with_(Hq=4, Hkv=2, n=2777),
], ids=["tiny", "llama8b-6000", "llama70b-5003", "gq1", "gq2"])
def test_per_head_workloads(cfg):
    x_cpu = synth.decode_layer(cfg, 0)
    x = {k: v.cuda() for k, v in x_cpu.items()}
    K = ots.budget_tokens(cfg.n, cfg.budget_permille, cfg.sink, cfg.local)
    check_layer(x_cpu, x, cfg.n, K, cfg.sink, cfg.local)


@pytest.mark.parametrize("which", ["one", "all"])
def test_per_head_budget_edges(which):
    cfg = D["tiny"].with_(n=1500)
    x_cpu = synth.decode_layer(cfg, 0)
    x = {k: v.cuda() for k, v in x_cpu.items()}
    _, c0, c1, _ = ots.regions(cfg.n, cfg.sink, cfg.local)
    check_layer(x_cpu, x, cfg.n, 1 if which == "one" else c1 - c0, cfg.sink, cfg.local)


def test_per_head_exact_ties_break_to_lower_index():
    cfg = D["tiny"].with_(n=2000, needles_per_qhead=0)
    x_cpu = synth.decode_layer(cfg, 0)
    for dst in range(600, 1400, 7):
        x_cpu["K"][:, :, dst] = x_cpu["K"][:, :, 300]
    x = {k: v.cuda() for k, v in x_cpu.items()}
    n, sink, local = cfg.n, cfg.sink, cfg.local
    q64, K64, W64 = (synth.to_f64(x_cpu[k]) for k in ("q", "K", "W"))
    idx = ots.index_rows(K64[:, :, :n], W64)
    index = gpu_index(x, n, cfg.Hq)
    for K in (1, 50, 113, 400):
        sel = gpu_head_select(x, index, n, K, sink, local)
        S_ref, _ = ots.select_per_kv_head(q64, W64, idx, n, K, sink, local)
        assert np.array_equal(sel.cpu().numpy(), S_ref), K


@pytest.mark.parametrize("n", [3000, 20000])
def test_per_head_zero_query_selects_lowest_indices(n):
    """Every group sum is zero (of either sign): all keys of a row are equal,
    so the select has no digit to resolve and the lowest indices win; the
    cluster's CTAs exchange only their counts (n = 20000 spans several CTAs
    per row)."""
    cfg = D["tiny"].with_(n=n)
    x = {k: v.cuda() for k, v in synth.decode_layer(cfg, 0).items()}
    x["q"].zero_()
    x["q"][:, ::2] = -0.0
    index = gpu_index(x, n, cfg.Hq)
    for K in (1, 300, 2000):
        sel = gpu_head_select(x, index, n, K, cfg.sink, cfg.local)
        qasc.qasc_device_error()
        want = torch.arange(cfg.sink, cfg.sink + K, dtype=torch.int32).expand(cfg.B, cfg.Hkv, K)
        assert torch.equal(sel.cpu(), want), (n, K)


def test_shared_sets_match_the_shared_attention():
    cfg = D["llama8b"].with_(B=2, n=5000)
    x = {k: v.cuda() for k, v in synth.decode_layer(cfg, 0).items()}
    S = synth.random_selection(cfg.B, cfg.n, 700, cfg.sink, cfg.local, 5).cuda()
    S_rep = S[:, None, :].expand(cfg.B, cfg.Hkv, 700).contiguous()
    o1 = torch.empty((cfg.B, cfg.Hq, 128), dtype=torch.float32, device="cuda")
    ws = qasc.alloc_workspace(qasc.ts_attn_workspace_bytes(cfg.B, cfg.Hq, cfg.Hkv, cfg.n, cfg.n, 700))
    qasc.ts_sparse_attn(x["q"], x["K"], x["V"], S, o1, ws, n=cfg.n)
    o2, _ = gpu_head_attn(x, S_rep, cfg.n, cfg.sink, cfg.local)
    assert torch.equal(o1, o2)


def test_per_head_deterministic_repeat():
    cfg = D["llama8b"].with_(B=2, n=8000)
    x = {k: v.cuda() for k, v in synth.decode_layer(cfg, 0).items()}
    K = ots.budget_tokens(cfg.n, cfg.budget_permille, cfg.sink, cfg.local)
    index = gpu_index(x, cfg.n, cfg.Hq)
    s1 = gpu_head_select(x, index, cfg.n, K, cfg.sink, cfg.local)
    s2 = gpu_head_select(x, index, cfg.n, K, cfg.sink, cfg.local)
    assert torch.equal(s1, s2)


@pytest.mark.slow
def test_per_head_full_size_128k_b4():
    cfg = D["llama8b_long"]
    x = synth.decode_layer(cfg, 0, device="cuda")
    x_cpu = {k: v.cpu() for k, v in x.items()}
    K = ots.budget_tokens(cfg.n, cfg.budget_permille, cfg.sink, cfg.local)
    check_layer(x_cpu, x, cfg.n, K, cfg.sink, cfg.local, bs=[2])
