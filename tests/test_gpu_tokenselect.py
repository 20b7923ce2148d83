"""GPU parity of the TokenSelect decode path against the fp64 oracle.

Every case draws seeded synthetic inputs (synth), runs the CUDA path through
the C ABI (Python binding) and compares with the oracle on the same inputs:
  index    bit-exact (RNE bf16 of the exact product)
  S        the band rule in parity_rules.check_selection
  out/lse  max-abs <= 1e-3 and relative L2 <= 1e-3 against the oracle
           evaluated on the GPU's own selected set; also on the oracle's S
           (passed to the kernel as input) and on seeded random sets.
"""

import math

import numpy as np
import pytest
import torch

import synth
from oracle import tokenselect as ots
from tests.parity_rules import check_attention, check_selection, selection_difference

pytestmark = pytest.mark.gpu

qasc = pytest.importorskip("query_aware_sparse_compressed_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qasc._lib.load()   # raises if the library was not built


def to_dev(x):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def gpu_index(x, n, Hq):
    K, W = x["K"], x["W"]
    B, Hkv, n_cap, _ = K.shape
    index = torch.zeros((B, Hkv, n_cap, 32), dtype=torch.bfloat16, device="cuda")
    qasc.ts_index_append(K, W, index, 0, n, Hq=Hq, n=n)
    return index


# Output buffers sit inside larger ones filled with a canary value; after
# each call the canaries either side must be intact (no write outside the
# output).  GUARD elements keep the output 16-byte aligned.
GUARD = 64


def guarded(shape, dtype, fill):
    n = math.prod(shape)
    buf = torch.full((n + 2 * GUARD,), fill, dtype=dtype, device="cuda")
    return buf, buf[GUARD:GUARD + n].view(shape)


def assert_guard(buf, view, fill, what):
    torch.cuda.synchronize()
    n = view.numel()
    assert bool((buf[:GUARD] == fill).all()) and bool((buf[GUARD + n:] == fill).all()), \
        "%s: a call wrote outside its output buffer" % what


def gpu_select(x, index, n, K, sink, local):
    q, W = x["q"], x["W"]
    B, Hq, _ = q.shape
    _, Hkv, n_cap, _ = index.shape
    buf, sel = guarded((B, K), torch.int32, -7)
    ws = qasc.alloc_workspace(qasc.ts_select_workspace_bytes(B, Hq, Hkv, n, n_cap, K, sink, local))
    qasc.ts_score_vote_select(q, W, index, sel, ws, n=n, K=K, sink=sink, local=local)
    assert_guard(buf, sel, -7, "ts_score_vote_select sel")
    return sel


def gpu_attn(x, sel, n, sink, local):
    q, K, V = x["q"], x["K"], x["V"]
    B, Hq, _ = q.shape
    _, Hkv, n_cap, _ = K.shape
    Ksel = sel.shape[1]
    obuf, out = guarded((B, Hq, 128), torch.float32, -7777.0)
    lbuf, lse = guarded((B, Hq), torch.float32, -7777.0)
    ws = qasc.alloc_workspace(qasc.ts_attn_workspace_bytes(B, Hq, Hkv, n, n_cap, Ksel, sink, local))
    qasc.ts_sparse_attn(q, K, V, sel if Ksel else None, out, ws, n=n, sink=sink, local=local, lse=lse)
    assert_guard(obuf, out, -7777.0, "ts_sparse_attn out")
    assert_guard(lbuf, lse, -7777.0, "ts_sparse_attn lse")
    return out, lse


def run_case(cfg, budget_permille=None, layer=0, check_index=True):
    x_cpu = synth.decode_layer(cfg, layer)
    x = to_dev(x_cpu)
    n, sink, local = cfg.n, cfg.sink, cfg.local
    bp = cfg.budget_permille if budget_permille is None else budget_permille
    K = ots.budget_tokens(n, bp, sink, local)
    index = gpu_index(x, n, cfg.Hq)
    sel = gpu_select(x, index, n, K, sink, local)
    out, lse = gpu_attn(x, sel, n, sink, local)
    qasc.qasc_device_error()
    torch.cuda.synchronize()

    q64, K64, V64, W64 = (synth.to_f64(x_cpu[k]) for k in ("q", "K", "V", "W"))
    idx_ref = ots.index_rows(K64[:, :, :n], W64)
    if check_index:
        got = synth.to_f64(index[:, :, :n])
        assert np.array_equal(got, idx_ref), "index differs in %d places" % int((got != idx_ref).sum())
    S_ref, info = ots.select(q64, W64, idx_ref, n, K, sink, local)
    S_gpu = sel.cpu().numpy().astype(np.int64)
    ndiff = 0
    for b in range(cfg.B):
        if K > 0:
            d = check_selection(S_gpu[b], info["scores"][b], info["theta"][b], info["c0"], K)
            assert d == selection_difference(S_gpu[b], S_ref[b])
            ndiff += d
    # The GPU's output against the oracle evaluated on the GPU's own set.
    own_out, own_lse = ots.sparse_attention(q64, K64[:, :, :n], V64[:, :, :n], S_gpu, n, sink, local)
    check_attention(out.cpu().numpy(), own_out)
    check_attention(lse.cpu().numpy(), own_lse)
    # Attention parity on the oracle's set, run through the kernel as input.
    sel_ref = torch.from_numpy(S_ref.astype(np.int32)).cuda()
    out_o, lse_o = gpu_attn(x, sel_ref, n, sink, local)
    ref_out, ref_lse = ots.sparse_attention(q64, K64[:, :, :n], V64[:, :, :n], S_ref, n, sink, local)
    check_attention(out_o.cpu().numpy(), ref_out)
    check_attention(lse_o.cpu().numpy(), ref_lse)
    return dict(ndiff=ndiff, S_gpu=S_gpu, S_ref=S_ref, x=x, out=out, lse=lse, K=K)


D = synth.DECODE_CONFIGS


def test_tiny_workload_exact():
    r = run_case(D["tiny"])
    assert r["ndiff"] == 0


@pytest.mark.parametrize("cfg", [
    D["llama8b"].with_(B=2, n=9037),                                   # 32/8, ragged tail
    D["llama70b"].with_(n=5000, n_cap=5120),                           # 64/8, n < n_cap
    D["llama8b_long"].with_(B=2, n=12000),                             # heavy-tailed keys
    D["tiny"].with_(Hq=4, Hkv=4, n=3000),                              # Gq = 1
    D["tiny"].with_(Hq=8, Hkv=4, n=2500, budget_permille=300),         # Gq = 2
], ids=["8b-ragged", "70b-ncap", "long-heavy", "gq1", "gq2"])
def test_shrunk_workloads(cfg):
    run_case(cfg)


@pytest.mark.parametrize("bp", synth.BUDGET_SWEEP_PERMILLE)
def test_budget_sweep_heavy_tails(bp):
    run_case(D["llama8b_long"].with_(B=1, n=7000), budget_permille=bp)


@pytest.mark.parametrize("n", [1, 3, 4, 5, 200, 260, 261, 262, 517])
def test_small_contexts(n):
    # n <= sink + local leaves no candidates (K = 0, T = all tokens);
    # n = 261 leaves one candidate.
    cfg = D["tiny"].with_(n=n, n_cap=max(n, 64), needles_per_qhead=0, budget_permille=1000)
    run_case(cfg)


def test_full_budget_is_dense_attention():
    cfg = D["tiny"].with_(n=1500, budget_permille=1000, needles_per_qhead=0)
    r = run_case(cfg)
    x = r["x"]
    q64, K64, V64 = (synth.to_f64(x[k]) for k in ("q", "K", "V"))
    dense, _ = ots.dense_attention(q64, K64[:, :, :1500], V64[:, :, :1500], 1500)
    check_attention(r["out"].cpu().numpy(), dense)


def test_exact_ties_break_to_lower_index():
    cfg = D["tiny"].with_(n=2000, needles_per_qhead=0)
    x_cpu = synth.decode_layer(cfg, 0)
    # duplicate key rows (same index rows, same scores in every head)
    for dst in range(600, 1400, 7):
        x_cpu["K"][:, :, dst] = x_cpu["K"][:, :, 300]
    x = to_dev(x_cpu)
    n, sink, local = cfg.n, cfg.sink, cfg.local
    for K in (1, 50, 113, 400):
        index = gpu_index(x, n, cfg.Hq)
        sel = gpu_select(x, index, n, K, sink, local)
        q64, K64, W64 = (synth.to_f64(x_cpu[k]) for k in ("q", "K", "W"))
        S_ref, _ = ots.select(q64, W64, ots.index_rows(K64[:, :, :n], W64), n, K, sink, local)
        assert np.array_equal(sel.cpu().numpy(), S_ref), K


def test_zero_query_selects_lowest_indices():
    # Every score is zero (of either sign): no head votes for anything, every
    # key ties, and the lowest indices win; theta's range test must treat -0
    # and +0 as one key, as the order-preserving key does.
    cfg = D["tiny"].with_(n=3000)
    x = to_dev(synth.decode_layer(cfg, 0))
    x["q"].zero_()
    x["q"][:, ::2] = -0.0
    n, sink, local = cfg.n, cfg.sink, cfg.local
    index = gpu_index(x, n, cfg.Hq)
    for K in (1, 300, 2000):
        sel = gpu_select(x, index, n, K, sink, local)
        qasc.qasc_device_error()
        want = torch.arange(sink, sink + K, dtype=torch.int32).expand(cfg.B, K)
        assert torch.equal(sel.cpu(), want), K


def test_crowded_threshold_digit():
    """Heads whose threshold digit holds most of C (more keys than the
    per-head shared-memory list): every key row of KV head 0 is the same row
    (its heads score every candidate alike, so theta_h equals that score and
    the head votes for nobody), and half of KV head 1's rows are one row."""
    cfg = D["tiny"].with_(n=20000, needles_per_qhead=0)
    x_cpu = synth.decode_layer(cfg, 0)
    x_cpu["K"][:, 0, :] = x_cpu["K"][:, 0, 123:124]
    x_cpu["K"][:, 1, ::2] = x_cpu["K"][:, 1, 777:778]
    x = to_dev(x_cpu)
    n, sink, local = cfg.n, cfg.sink, cfg.local
    q64, K64, W64 = (synth.to_f64(x_cpu[k]) for k in ("q", "K", "W"))
    idx_ref = ots.index_rows(K64[:, :, :n], W64)
    for bp in (100, 300):
        K = ots.budget_tokens(n, bp, sink, local)
        index = gpu_index(x, n, cfg.Hq)
        sel = gpu_select(x, index, n, K, sink, local)
        qasc.qasc_device_error()
        S_ref, info = ots.select(q64, W64, idx_ref, n, K, sink, local)
        S_gpu = sel.cpu().numpy().astype(np.int64)
        check_selection(S_gpu[0], info["scores"][0], info["theta"][0], info["c0"], K)
        assert np.array_equal(S_gpu, S_ref), bp


def test_random_selected_sets_attention():
    cfg = D["llama8b"].with_(B=2, n=6000)
    x_cpu = synth.decode_layer(cfg, 0)
    x = to_dev(x_cpu)
    q64, K64, V64 = (synth.to_f64(x_cpu[k]) for k in ("q", "K", "V"))
    for K, seed in ((1, 1), (37, 2), (2000, 3), (5740, 4)):
        S = synth.random_selection(cfg.B, cfg.n, K, cfg.sink, cfg.local, seed)
        out, lse = gpu_attn(x, S.cuda(), cfg.n, cfg.sink, cfg.local)
        ref, ref_lse = ots.sparse_attention(q64, K64[:, :, :cfg.n], V64[:, :, :cfg.n], S.numpy(), cfg.n,
                                            cfg.sink, cfg.local)
        check_attention(out.cpu().numpy(), ref)
        check_attention(lse.cpu().numpy(), ref_lse)


def test_decode_append_single_rows():
    cfg = D["tiny"].with_(n=3000, n_cap=3072)
    x_cpu = synth.decode_layer(cfg, 0)
    x = to_dev(x_cpu)
    index = torch.zeros((1, 2, 3072, 32), dtype=torch.bfloat16, device="cuda")
    for t in (0, 1, 777, 2999, 3071):
        qasc.ts_index_append(x["K"], x["W"], index, t, 1, Hq=cfg.Hq)
    ref = ots.index_rows(synth.to_f64(x_cpu["K"]), synth.to_f64(x_cpu["W"]))
    got = synth.to_f64(index)
    for t in (0, 1, 777, 2999, 3071):
        assert np.array_equal(got[:, :, t], ref[:, :, t])
    untouched = [t for t in range(3072) if t not in (0, 1, 777, 2999, 3071)]
    assert np.all(got[:, :, untouched] == 0)


def test_index_append_on_rounding_midpoints():
    """Index values that lie exactly on a bf16 rounding midpoint, or 2^-30
    above or below one (both signs, ties to even and both rounding
    directions), in every column of every token: the fp32 error bound leaves
    each column ambiguous, so the bulk kernel sends all of them through its
    exact recompute queue at full capacity (32 columns of 32 tokens per warp
    pass), and the single-row kernel recomputes them inline.  Both must equal
    the oracle's correctly rounded values bit for bit."""
    n, Hkv, n_cap = 2000, 2, 2048
    rng = np.random.default_rng(5)
    K = np.zeros((1, Hkv, n_cap, 128))
    W = np.zeros((Hkv, 128, 32))
    for g in range(Hkv):
        W[g, 0] = 1 + rng.integers(0, 128, 32) * 2.0 ** -7     # a bf16 value ...
        W[g, 1] = 2.0 ** -8                                     # ... plus half its ulp ...
        W[g, 2] = rng.choice([0.0, 2.0 ** -30, -2.0 ** -30], 32)  # ... plus a nudge
    scale = rng.choice([-1.0, 1.0], n) * 2.0 ** rng.integers(-20, 20, n)
    for g in range(Hkv):
        K[0, g, :n, :3] = scale[:, None]
    K[0, :, np.nonzero(rng.random(n) < 0.05)[0], :3] = 0.0
    Kd = torch.from_numpy(K).to(torch.bfloat16).cuda()
    Wd = torch.from_numpy(W).to(torch.bfloat16).cuda()
    assert np.array_equal(synth.to_f64(Kd), K) and np.array_equal(synth.to_f64(Wd), W)
    ref = ots.index_rows(K[:, :, :n], W)
    index = torch.zeros((1, Hkv, n_cap, 32), dtype=torch.bfloat16, device="cuda")
    qasc.ts_index_append(Kd, Wd, index, 0, n, Hq=2 * Hkv, n=n)
    qasc.qasc_device_error()
    assert np.array_equal(synth.to_f64(index)[:, :, :n], ref)
    rows = torch.zeros_like(index)
    for t in (0, 1, 1000, n - 1):
        qasc.ts_index_append(Kd, Wd, rows, t, 1, Hq=2 * Hkv)
    got = synth.to_f64(rows)
    for t in (0, 1, 1000, n - 1):
        assert np.array_equal(got[:, :, t], ref[:, :, t])


def test_deterministic_repeat():
    cfg = D["llama8b"].with_(B=2, n=8000)
    x = to_dev(synth.decode_layer(cfg, 0))
    K = ots.budget_tokens(cfg.n, cfg.budget_permille, cfg.sink, cfg.local)
    index = gpu_index(x, cfg.n, cfg.Hq)
    s1 = gpu_select(x, index, cfg.n, K, cfg.sink, cfg.local)
    o1, l1 = gpu_attn(x, s1, cfg.n, cfg.sink, cfg.local)
    s2 = gpu_select(x, index, cfg.n, K, cfg.sink, cfg.local)
    o2, l2 = gpu_attn(x, s2, cfg.n, cfg.sink, cfg.local)
    assert torch.equal(s1, s2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ----------------------------------------------------------- full size
def _full_layer(cfg):
    return to_dev(synth.decode_layer(cfg, 0, device="cpu")) if cfg.n * cfg.B <= 140000 else \
        synth.decode_layer(cfg, 0, device="cuda")


def _full_size(cfg, bsample, budget_permille=None, x=None, index=None):
    """Whole layer on the GPU at full size; the oracle checks sequence bsample:
    the index rows bit for bit, the selection by the band rule, and the
    attention output and LSE against the oracle on the GPU's own set and on
    the oracle's set."""
    x = _full_layer(cfg) if x is None else x
    n, sink, local = cfg.n, cfg.sink, cfg.local
    bp = cfg.budget_permille if budget_permille is None else budget_permille
    K = ots.budget_tokens(n, bp, sink, local)
    if index is None:
        index = gpu_index(x, n, cfg.Hq)
    sel = gpu_select(x, index, n, K, sink, local)
    out, lse = gpu_attn(x, sel, n, sink, local)
    qasc.qasc_device_error()
    b = bsample
    q64 = synth.to_f64(x["q"][b:b + 1])
    K64 = synth.to_f64(x["K"][b:b + 1, :, :n])
    V64 = synth.to_f64(x["V"][b:b + 1, :, :n])
    W64 = synth.to_f64(x["W"])
    idx_ref = ots.index_rows(K64, W64)
    got = synth.to_f64(index[b:b + 1, :, :n])
    assert np.array_equal(got, idx_ref)
    S_ref, info = ots.select(q64, W64, idx_ref, n, K, sink, local)
    S_gpu = sel[b].cpu().numpy().astype(np.int64)
    stats = {}
    ndiff = check_selection(S_gpu, info["scores"][0], info["theta"][0], info["c0"], K, stats=stats)
    own, own_lse = ots.sparse_attention(q64, K64, V64, S_gpu[None], n, sink, local)
    check_attention(out[b:b + 1].cpu().numpy(), own)
    check_attention(lse[b:b + 1].cpu().numpy(), own_lse)
    sel_ref = torch.from_numpy(S_ref.astype(np.int32)).cuda()
    xb = {k: x[k][b:b + 1].contiguous() for k in ("q", "K", "V")}
    out_o, lse_o = gpu_attn(xb, sel_ref, n, sink, local)
    ref, ref_lse = ots.sparse_attention(q64, K64, V64, S_ref, n, sink, local)
    check_attention(out_o.cpu().numpy(), ref)
    check_attention(lse_o.cpu().numpy(), ref_lse)
    return dict(ndiff=ndiff, band=stats["band"], K=K, index=index, x=x)


@pytest.mark.slow
def test_full_size_llama8b_32k():
    _full_size(D["llama8b"], 0)


@pytest.mark.slow
def test_full_size_llama8b_128k_b4():
    _full_size(D["llama8b_long"], 3)


@pytest.fixture(scope="module")
def long_layer():
    """The 128K x B4 heavy-tailed layer and its GPU-built index, shared by the
    budget sweep."""
    cfg = D["llama8b_long"]
    x = _full_layer(cfg)
    index = gpu_index(x, cfg.n, cfg.Hq)
    yield cfg, x, index
    del x, index
    torch.cuda.empty_cache()


@pytest.mark.slow
@pytest.mark.parametrize("bp,b", [(50, 0), (100, 1), (150, 2), (300, 3)])
def test_full_size_llama8b_128k_budget_sweep(long_layer, bp, b):
    # the other budgets of the 128K sweep (20 % is the case above), one
    # sampled sequence each
    cfg, x, index = long_layer
    r = _full_size(cfg, b, budget_permille=bp, x=x, index=index)
    assert r["ndiff"] <= r["band"]


@pytest.mark.slow
def test_full_size_llama70b_64k():
    _full_size(D["llama70b"], 1)
