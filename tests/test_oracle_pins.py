"""Pins for the fp64 oracle: what fixes it other than itself.

Each test checks the oracle against a hand-worked example from the pages'
definitions, a closed form, an invariant, a library routine in a special case
it reduces to, or brute-force enumeration on tiny inputs.  CPU only.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import bf16 as obf
from oracle import snapkv as osnap
from oracle import tokenselect as ots

D, DI = 128, 32


# ----------------------------------------------------------------- bf16 RNE
def test_bf16_hand_values():
    # bf16 keeps 8 significant bits: spacing 2^-7 on [1, 2).
    cases = {
        1.0: 0x3F80,
        1.0 + 2.0 ** -8: 0x3F80,                   # exact tie -> even (down)
        1.0 + 3 * 2.0 ** -8: 0x3F82,               # exact tie -> even (up)
        1.0 + 2.0 ** -8 + 2.0 ** -30: 0x3F81,      # just above the tie -> up
        -2.5: 0xC020,
        2.0 ** -126: 0x0080,                       # smallest normal
        2.0 ** -133: 0x0001,                       # smallest subnormal
        2.0 ** -134: 0x0000,                       # tie between 0 and 2^-133 -> even (0)
        3 * 2.0 ** -134: 0x0002,                   # tie between 1 and 2 quanta -> even
        (2 - 2.0 ** -7) * 2.0 ** 127: 0x7F7F,      # largest finite
        (2 - 2.0 ** -9) * 2.0 ** 127: 0x7F80,      # rounds past it -> inf
    }
    for x, bits in cases.items():
        got = obf.bf16_bits(obf.round_bf16(np.array([x])))[0]
        assert got == bits, (x, hex(got), hex(bits))


def test_bf16_matches_torch_cast_on_fp32_inputs():
    rng = np.random.default_rng(7)
    raw = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    f32 = raw.view(np.float32)
    f32 = f32[np.isfinite(f32)]
    ours = obf.bf16_bits(obf.round_bf16(f32.astype(np.float64)))
    theirs = torch.from_numpy(f32.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    # torch maps overflow to inf as well; compare encodings directly
    assert np.array_equal(ours, theirs)


# ----------------------------------------------------------------- index
def _selector(offset, Hkv=1, scale=1.0):
    W = np.zeros((Hkv, D, DI))
    for g in range(Hkv):
        for j in range(DI):
            W[g, (j * 4 + offset + g) % D, j] = scale
    return W


def test_index_selector_projection_is_a_column_gather():
    rng = np.random.default_rng(1)
    K = obf.round_bf16(rng.standard_normal((2, 3, 50, D)))
    W = _selector(1, Hkv=3)
    idx = ots.index_rows(K, W)
    for g in range(3):
        cols = [(j * 4 + 1 + g) % D for j in range(DI)]
        assert np.array_equal(idx[:, g], K[:, g][..., cols])


def test_index_power_of_two_scaling_is_exact():
    rng = np.random.default_rng(2)
    K = obf.round_bf16(rng.standard_normal((1, 1, 40, D)))
    W = _selector(0, scale=0.125)
    assert np.array_equal(ots.index_rows(K, W)[0, 0], K[0, 0][:, 0:D:4] / 8)


def test_index_small_integer_dot_products():
    # K row = (1, 2, ..., 128) / 64 scaled, W column j = e_{j} + e_{j+64}:
    # the dot product is (j+1 + j+65)/64, exactly representable.
    K = (np.arange(1, D + 1) / 64.0)[None, None, None, :]
    W = np.zeros((1, D, DI))
    for j in range(DI):
        W[0, j, j] = 1.0
        W[0, j + 64, j] = 1.0
    want = np.array([(2 * j + 66) / 64.0 for j in range(DI)])
    assert np.array_equal(ots.index_rows(K, W)[0, 0, 0], want)


# ----------------------------------------------------------------- selection
def _hand_case(golden_dir, zero_query=False):
    with open(os.path.join(golden_dir, "tokenselect_hand.json")) as f:
        g = json.load(f)
    n = 8
    K = np.zeros((1, 1, n, D))
    K[0, 0, :, 0] = g["a"]
    K[0, 0, :, 1] = g["b"]
    W = np.zeros((1, D, DI))
    for j in range(DI):
        W[0, j, j] = 1.0
    q = np.zeros((1, 2, D))
    if not zero_query:
        q[0, 0, 0] = 1.0
        q[0, 1, 1] = 1.0
    idx = ots.index_rows(K, W)
    return g, q, K, W, idx


def test_selection_hand_worked_example(golden_dir):
    g, q, K, W, idx = _hand_case(golden_dir)
    S, info = ots.select(q, W, idx, n=8, K=3, sink=1, local=1)
    assert np.allclose(info["scores"][0] * math.sqrt(DI), g["scores_times_sqrt32"])
    assert np.allclose(info["theta"][0] * math.sqrt(DI), g["theta_times_sqrt32"])
    assert info["vote"][0].tolist() == g["vote"]
    assert S[0].tolist() == g["S"]
    assert ots.attended_tokens(S[0], 8, 1, 1).tolist() == g["T"]


def test_zero_query_selection_and_uniform_attention(golden_dir):
    g, q, K, W, idx = _hand_case(golden_dir, zero_query=True)
    zc = g["zero_query_case"]
    S, _ = ots.select(q, W, idx, n=8, K=3, sink=1, local=1)
    assert S[0].tolist() == zc["S"]
    rng = np.random.default_rng(3)
    V = np.zeros((1, 1, 8, D))
    V[0, 0] = rng.integers(-8, 8, size=(8, D))
    out, lse = ots.sparse_attention(q, K, V, S, 8, 1, 1)
    mean = V[0, 0, zc["T"]].mean(axis=0)
    assert np.allclose(out[0, 0], mean) and np.allclose(out[0, 1], mean)
    assert np.allclose(lse, math.log(len(zc["T"])))


def _outranks(a, b):
    """Key tuple (vote, sum, token): a is ranked ahead of b."""
    return (a[0], a[1], -a[2]) > (b[0], b[1], -b[2])


@pytest.mark.parametrize("seed", range(12))
def test_selection_equals_unique_dominating_subset(seed):
    rng = np.random.default_rng(100 + seed)
    n, sink, local = int(rng.integers(8, 17)), 1, 2
    Hkv, group = 2, 2
    Hq = Hkv * group
    q = obf.round_bf16(rng.standard_normal((1, Hq, D)))
    Kc = obf.round_bf16(rng.standard_normal((1, Hkv, n, D)))
    if seed % 3 == 0:               # plant exact duplicates to force ties
        Kc[0, :, 5] = Kc[0, :, 3]
        Kc[0, :, 6] = Kc[0, :, 3]
    W = obf.round_bf16(rng.standard_normal((Hkv, D, DI)) / math.sqrt(D))
    idx = ots.index_rows(Kc, W)
    _, c0, c1, _ = ots.regions(n, sink, local)
    cand = list(range(c0, c1))
    for K in range(0, len(cand) + 1):
        S, info = ots.select(q, W, idx, n, K, sink, local)
        if K == 0:
            assert S.shape == (1, 0)
            continue
        key = {i: (int(info["vote"][0][i - c0]), float(info["ssum"][0][i - c0]), i) for i in cand}
        winners = []
        for sub in itertools.combinations(cand, K):
            inside = set(sub)
            if all(_outranks(key[a], key[b]) for a in inside for b in cand if b not in inside):
                winners.append(sorted(sub))
        assert len(winners) == 1
        assert S[0].tolist() == winners[0]
        # second restatement: pairwise rank counting
        rc = ots.select_by_rank_count(info["vote"][0], info["ssum"][0], c0, K)
        assert sorted(rc.tolist()) == winners[0]


@pytest.mark.parametrize("seed", range(5))
def test_single_head_reduces_to_plain_topk(seed):
    rng = np.random.default_rng(200 + seed)
    n, sink, local = 300, 4, 16
    q = obf.round_bf16(rng.standard_normal((1, 1, D)))
    Kc = obf.round_bf16(rng.standard_normal((1, 1, n, D)))
    Kc[0, 0, 100] = Kc[0, 0, 50]          # an exact tie
    W = obf.round_bf16(rng.standard_normal((1, D, DI)) / math.sqrt(D))
    idx = ots.index_rows(Kc, W)
    _, c0, c1, _ = ots.regions(n, sink, local)
    sc = ots.scores(q, W, idx, n, sink, local)[0, 0]
    for K in (1, 7, 60, c1 - c0):
        S, _ = ots.select(q, W, idx, n, K, sink, local)
        want = np.sort(np.argsort(-sc, kind="stable")[:K] + c0)
        assert np.array_equal(S[0], want)


def test_identical_heads_reduce_to_plain_topk():
    rng = np.random.default_rng(5)
    n, sink, local, Hq = 400, 4, 32, 4
    q1 = obf.round_bf16(rng.standard_normal((1, 1, D)))
    q = np.repeat(q1, Hq, axis=1)
    Kc = obf.round_bf16(rng.standard_normal((1, 1, n, D)))
    W = obf.round_bf16(rng.standard_normal((1, D, DI)) / math.sqrt(D))
    idx = ots.index_rows(Kc, W)
    sc = ots.scores(q, W, idx, n, sink, local)[0, 0]
    for K in (1, 10, 100):
        S, info = ots.select(q, W, idx, n, K, sink, local)
        assert set(np.unique(info["vote"])) <= {0, Hq}
        assert (info["vote"] == Hq).sum() == K - 1
        want = np.sort(np.argsort(-sc, kind="stable")[:K] + sink)
        assert np.array_equal(S[0], want)


@pytest.mark.parametrize("seed", range(4))
def test_threshold_is_kth_order_statistic_and_vmin_property(seed):
    rng = np.random.default_rng(300 + seed)
    n, sink, local, Hkv, group = 700, 4, 64, 2, 4
    Hq = Hkv * group
    q = obf.round_bf16(rng.standard_normal((2, Hq, D)))
    Kc = obf.round_bf16(rng.standard_normal((2, Hkv, n, D)))
    W = obf.round_bf16(rng.standard_normal((Hkv, D, DI)) / math.sqrt(D))
    idx = ots.index_rows(Kc, W)
    for K in (1, 5, 60, 400):
        S, info = ots.select(q, W, idx, n, K, sink, local)
        sc, th = info["scores"], info["theta"]
        assert np.all((sc > th[..., None]).sum(-1) <= K - 1)
        assert np.all((sc >= th[..., None]).sum(-1) >= K)
        assert np.all(np.any(sc == th[..., None], axis=-1))
        _, c0, c1, _ = ots.regions(n, sink, local)
        for b in range(2):
            s = S[b]
            assert len(s) == K and np.all(np.diff(s) > 0)
            assert s.min() >= c0 and s.max() < c1
            nominated = c0 + np.nonzero(info["vote"][b] >= 1)[0]
            if len(nominated) <= K:
                assert set(nominated.tolist()) <= set(s.tolist())
            else:
                assert set(s.tolist()) <= set(nominated.tolist())


def test_gqa_head_to_group_mapping():
    # Only KV group 1 has a non-zero index, only head 6 (group 1 at Gq=4) asks.
    n, sink, local = 64, 4, 8
    Hq, Hkv = 8, 2
    Kc = np.zeros((1, Hkv, n, D))
    Kc[0, 1, :, 0] = np.arange(n) / 8.0
    W = _selector(0, Hkv=Hkv)  # group g reads column 4j + g
    W[1] = 0.0
    W[1, 0, 3] = 1.0           # group 1: index column 3 = K[:, 0]
    q = np.zeros((1, Hq, D))
    q[0, 6, 0] = 2.0           # q'_6 = W_1^T q_6 -> component 3 equals 2
    idx = ots.index_rows(Kc, W)
    sc = ots.scores(q, W, idx, n, sink, local)
    _, c0, c1, _ = ots.regions(n, sink, local)
    want = 2.0 * (np.arange(c0, c1) / 8.0) / math.sqrt(DI)
    assert np.allclose(sc[0, 6], want)
    others = np.delete(sc[0], 6, axis=0)
    assert np.all(others == 0.0)


def test_region_edge_cases():
    assert ots.regions(0, 4, 256) == (0, 4, 4, 0)
    assert ots.regions(3, 4, 256) == (3, 4, 4, 3)
    assert ots.regions(100, 4, 256) == (4, 4, 4, 4)
    assert ots.regions(260, 4, 256) == (4, 4, 4, 4)
    assert ots.regions(261, 4, 256) == (4, 4, 5, 5)
    assert ots.budget_tokens(131072, 200, 4, 256) == 26214
    assert ots.budget_tokens(32768, 200, 4, 256) == 6553
    assert ots.budget_tokens(4096, 100, 4, 256) == 409
    assert ots.budget_tokens(300, 1000, 4, 256) == 40


# ----------------------------------------------------------------- attention
@pytest.mark.parametrize("n", [5, 260, 777])
def test_full_budget_equals_dense_sdpa(n):
    rng = np.random.default_rng(400 + n)
    sink, local, Hkv, group = 4, 256, 2, 4
    Hq = Hkv * group
    q = obf.round_bf16(rng.standard_normal((2, Hq, D)))
    Kc = obf.round_bf16(rng.standard_normal((2, Hkv, n, D)))
    Vc = obf.round_bf16(rng.standard_normal((2, Hkv, n, D)))
    W = obf.round_bf16(rng.standard_normal((Hkv, D, DI)) / math.sqrt(D))
    idx = ots.index_rows(Kc, W)
    _, c0, c1, _ = ots.regions(n, sink, local)
    S, _ = ots.select(q, W, idx, n, c1 - c0, sink, local)
    out, lse = ots.sparse_attention(q, Kc, Vc, S, n, sink, local)
    tq = torch.from_numpy(q).unsqueeze(2)                               # [B,Hq,1,d]
    tk = torch.from_numpy(Kc).repeat_interleave(group, dim=1)
    tv = torch.from_numpy(Vc).repeat_interleave(group, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv)[:, :, 0]
    assert np.allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    logits = (tq @ tk.transpose(-1, -2))[:, :, 0] / math.sqrt(D)
    assert np.allclose(lse, torch.logsumexp(logits, dim=-1).numpy(), rtol=1e-12)


def test_dominant_key_attention_returns_its_value():
    rng = np.random.default_rng(9)
    n = 600
    q = np.zeros((1, 1, D))
    q[0, 0, :] = 1.0
    Kc = obf.round_bf16(rng.standard_normal((1, 1, n, D)) * 0.01)
    Kc[0, 0, 123] = 8.0              # logit 8 * 128 / sqrt(128) ~ 90
    Vc = rng.standard_normal((1, 1, n, D))
    S = np.array([[10, 123, 200]])
    out, _ = ots.sparse_attention(q, Kc, Vc, S, n, 4, 256)
    assert np.allclose(out[0, 0], Vc[0, 0, 123], atol=1e-12)


def test_attention_weights_uniform_when_keys_identical():
    rng = np.random.default_rng(10)
    n = 300
    q = rng.standard_normal((1, 2, D))
    Kc = np.tile(rng.standard_normal((1, 1, 1, D)), (1, 1, n, 1))
    Vc = rng.standard_normal((1, 1, n, D))
    S = np.array([[4, 9, 20, 43]])     # C = [4, 44) for sink 4, local 256
    out, lse = ots.sparse_attention(q, Kc, Vc, S, n, 4, 256)
    T = list(range(4)) + [4, 9, 20, 43] + list(range(44, 300))
    assert np.allclose(out[0, 0], Vc[0, 0, T].mean(0))
    z = Kc[0, 0, 0] @ q[0, 1] / math.sqrt(D)
    assert np.isclose(lse[0, 1], z + math.log(len(T)))


# ----------------------------------------------------------------- SnapKV
def test_snapkv_uniform_case(golden_dir):
    with open(os.path.join(golden_dir, "snapkv_hand.json")) as f:
        g = json.load(f)["uniform_case"]
    q = np.zeros((1, 1, 4, D))
    rng = np.random.default_rng(11)
    Kc = rng.standard_normal((1, 1, 6, D))
    Vc = rng.standard_normal((1, 1, 6, D))
    idx, Kk, Vk, a, p = osnap.compress(q, Kc, Vc, 6, 3, 3)
    assert np.allclose(a[0, 0], g["a"])
    assert np.allclose(p[0, 0] * 18, g["p_times_18"])
    assert idx[0, 0].tolist() == g["S"]
    assert np.array_equal(Kk[0, 0], Kc[0, 0, g["S"]])


def test_snapkv_capacity_over_length_is_identity(golden_dir):
    with open(os.path.join(golden_dir, "snapkv_hand.json")) as f:
        g = json.load(f)["capacity_over_length"]
    rng = np.random.default_rng(12)
    n = g["n"]
    q = rng.standard_normal((2, 4, 3, D))
    Kc = rng.standard_normal((2, 2, n, D))
    Vc = rng.standard_normal((2, 2, n, D))
    idx, Kk, Vk, _, _ = osnap.compress(q, Kc, Vc, n, g["c"], 3)
    assert idx.shape == (2, 2, n)
    assert np.all(idx == np.array(g["S"]))
    assert np.array_equal(Kk, Kc) and np.array_equal(Vk, Vc)


@pytest.mark.parametrize("kernel", [1, 3, 5, 7])
def test_snapkv_pool_matches_library_avg_pool(kernel):
    rng = np.random.default_rng(13)
    a = rng.random((3, 4, 57))
    want = torch.nn.functional.avg_pool1d(torch.from_numpy(a), kernel_size=kernel,
                                          stride=1, padding=kernel // 2).numpy()
    assert np.allclose(osnap.pool(a, kernel), want, rtol=1e-14, atol=0)


def test_snapkv_softmax_rows_and_mean_sum_to_one():
    rng = np.random.default_rng(14)
    q = rng.standard_normal((2, 8, 5, D))
    Kc = rng.standard_normal((2, 2, 90, D))
    A = osnap.window_attention(q, Kc, 90)
    assert np.allclose(A.sum(-1), 1.0)
    a = osnap.window_mean(q, Kc, 90)
    assert np.allclose(a.sum(-1), 1.0)


def test_snapkv_single_row_is_library_softmax():
    rng = np.random.default_rng(15)
    q = rng.standard_normal((1, 1, 1, D))
    Kc = rng.standard_normal((1, 1, 40, D))
    a = osnap.window_mean(q, Kc, 40)[0, 0]
    logits = torch.from_numpy(Kc[0, 0] @ q[0, 0, 0] / math.sqrt(D))
    assert np.allclose(a, torch.softmax(logits, 0).numpy(), rtol=1e-13)


def test_snapkv_group_mean_spans_query_heads():
    # Two query heads share one KV head; head 0 looks at key 1, head 1 at key 4.
    n = 8
    Kc = np.zeros((1, 1, n, D))
    Kc[0, 0, 1, 0] = 1.0
    Kc[0, 0, 4, 1] = 1.0
    q = np.zeros((1, 2, 1, D))
    q[0, 0, 0, 0] = 400.0
    q[0, 1, 0, 1] = 400.0
    a = osnap.window_mean(q, Kc, n)[0, 0]
    assert abs(a[1] - 0.5) < 1e-9 and abs(a[4] - 0.5) < 1e-9
    p = osnap.pool(a[None, None], 3)[0, 0]
    assert np.allclose(p, [1 / 6] * 6 + [0, 0], atol=1e-9)


def test_snapkv_dominant_key_neighbourhood():
    n = 9
    Kc = np.zeros((1, 1, n, D))
    Kc[0, 0, 5, 0] = 1.0
    q = np.zeros((1, 1, 2, D))
    q[0, 0, :, 0] = 500.0
    _, _, _, a, p = osnap.compress(q, Kc, Kc, n, 3, 3)
    idx = osnap.top_c(p, 3)[0, 0]
    assert idx.tolist() == [4, 5, 6]
    assert abs(p[0, 0, 5] - 1 / 3) < 1e-9


# ----------------------------------------------------------------- pin power
# Plant a plausible mistake in the oracle (on the CPU) and check that a pin
# above catches it.

def test_planted_non_strict_vote_is_caught(golden_dir, monkeypatch):
    monkeypatch.setattr(ots, "votes", lambda sc, th: (sc >= th[..., None]).sum(axis=1))
    g, q, K, W, idx = _hand_case(golden_dir)
    S, _ = ots.select(q, W, idx, n=8, K=3, sink=1, local=1)
    assert S[0].tolist() != g["S"]


def test_planted_index_descending_tiebreak_is_caught(golden_dir, monkeypatch):
    def wrong(vote, ssum, c0):
        ids = c0 + np.arange(vote.shape[0])
        return ids[np.lexsort((-ids, -ssum, -vote))]
    monkeypatch.setattr(ots, "rank_order", wrong)
    g, q, K, W, idx = _hand_case(golden_dir)
    S, _ = ots.select(q, W, idx, n=8, K=3, sink=1, local=1)
    assert S[0].tolist() != g["S"]


def test_planted_sum_before_vote_is_caught(golden_dir, monkeypatch):
    def wrong(vote, ssum, c0):
        ids = c0 + np.arange(vote.shape[0])
        return ids[np.lexsort((ids, -vote, -ssum))]
    monkeypatch.setattr(ots, "rank_order", wrong)
    g, q, K, W, idx = _hand_case(golden_dir)
    S, _ = ots.select(q, W, idx, n=8, K=3, sink=1, local=1)
    assert S[0].tolist() != g["S"]


def test_planted_pool_divisor_is_caught(golden_dir, monkeypatch):
    def wrong(a, kernel=3):
        a = np.asarray(a, dtype=np.float64)
        n = a.shape[-1]
        s = np.zeros_like(a)
        c = np.zeros(n)
        for t in range(-(kernel // 2), kernel // 2 + 1):
            lo, hi = max(0, -t), min(n, n - t)
            s[..., lo:hi] += a[..., lo + t:hi + t]
            c[lo:hi] += 1
        return s / c
    monkeypatch.setattr(osnap, "pool", wrong)
    with open(os.path.join(golden_dir, "snapkv_hand.json")) as f:
        g = json.load(f)["uniform_case"]
    q = np.zeros((1, 1, 4, D))
    Kc = np.random.default_rng(11).standard_normal((1, 1, 6, D))
    _, _, _, _, p = osnap.compress(q, Kc, Kc, 6, 3, 3)
    assert not np.allclose(p[0, 0] * 18, g["p_times_18"])


def test_planted_transposed_projection_is_caught(monkeypatch):
    real = ots.query_index

    def wrong(q, W, Hkv):
        Wt = np.ascontiguousarray(np.swapaxes(np.asarray(W)[:, :DI, :], 1, 2))
        Wfull = np.zeros_like(np.asarray(W, dtype=np.float64))
        Wfull[:, :DI, :] = Wt
        return real(q, Wfull, Hkv)
    monkeypatch.setattr(ots, "query_index", wrong)
    with pytest.raises(AssertionError):
        test_gqa_head_to_group_mapping()


def test_planted_wrong_group_mapping_is_caught(monkeypatch):
    real = ots.query_index

    def wrong(q, W, Hkv):
        q = np.asarray(q, dtype=np.float64)
        Hq = q.shape[1]
        W = np.asarray(W, dtype=np.float64)
        g_of_h = np.arange(Hq) % Hkv            # interleaved instead of blocked
        return np.einsum("bhe,hej->bhj", q, W[g_of_h])
    monkeypatch.setattr(ots, "query_index", wrong)
    with pytest.raises(AssertionError):
        test_gqa_head_to_group_mapping()


def test_planted_dropped_sink_is_caught(monkeypatch):
    real = ots.attended_tokens

    def wrong(S_row, n, sink, local):
        return real(S_row, n, sink, local)[min(sink, n):]
    monkeypatch.setattr(ots, "attended_tokens", wrong)
    with pytest.raises(AssertionError):
        test_full_budget_equals_dense_sdpa(777)


def test_planted_unscaled_attention_logits_are_caught(monkeypatch):
    def wrong(q, K, V, S, n, sink, local):
        q, K, V = (np.asarray(t, dtype=np.float64) for t in (q, K, V))
        B, Hq, d = q.shape
        group = Hq // K.shape[1]
        out, lse = np.zeros((B, Hq, d)), np.zeros((B, Hq))
        for b in range(B):
            T = ots.attended_tokens(S[b], n, sink, local)
            for h in range(Hq):
                z = K[b, h // group, T, :] @ q[b, h]            # 1/sqrt(d) dropped
                p = np.exp(z - z.max())
                out[b, h] = p @ V[b, h // group, T, :] / p.sum()
                lse[b, h] = z.max() + np.log(p.sum())
        return out, lse
    monkeypatch.setattr(ots, "sparse_attention", wrong)
    with pytest.raises(AssertionError):
        test_full_budget_equals_dense_sdpa(260)


def _snap_window_attention(q_obs, K, n, scale=True, axis=-1):
    q = np.asarray(q_obs, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)[:, :, :n, :]
    Hq, d = q.shape[1], q.shape[3]
    g_of_h = np.arange(Hq) // (Hq // K.shape[1])
    x = np.einsum("bhrd,bhjd->bhrj", q, K[:, g_of_h]) / (np.sqrt(d) if scale else 1.0)
    e = np.exp(x - x.max(axis=axis, keepdims=True))
    return e / e.sum(axis=axis, keepdims=True)


def test_planted_unscaled_snapkv_logits_are_caught(monkeypatch):
    monkeypatch.setattr(osnap, "window_attention", lambda q, K, n: _snap_window_attention(q, K, n, scale=False))
    with pytest.raises(AssertionError):
        test_snapkv_single_row_is_library_softmax()


def test_planted_snapkv_softmax_over_window_rows_is_caught(monkeypatch):
    monkeypatch.setattr(osnap, "window_attention", lambda q, K, n: _snap_window_attention(q, K, n, axis=2))
    with pytest.raises(AssertionError):
        test_snapkv_softmax_rows_and_mean_sum_to_one()


def test_planted_snapkv_mean_over_one_head_is_caught(monkeypatch):
    def wrong(q_obs, K, n):
        A = osnap.window_attention(q_obs, K, n)
        B, Hq, w, _ = A.shape
        Hkv = np.asarray(K).shape[1]
        return A.reshape(B, Hkv, Hq // Hkv, w, n)[:, :, 0].mean(axis=2)   # first head of the group only
    monkeypatch.setattr(osnap, "window_mean", wrong)
    with pytest.raises(AssertionError):
        test_snapkv_group_mean_spans_query_heads()


def test_planted_snapkv_ties_to_higher_index_are_caught(golden_dir, monkeypatch):
    def wrong(p, c):
        p = np.asarray(p, dtype=np.float64)
        n = p.shape[-1]
        flat = p.reshape(-1, n)
        ids = np.arange(n)
        out = np.stack([np.sort(np.lexsort((-ids, -row))[:min(c, n)]) for row in flat])
        return out.reshape(p.shape[:-1] + (min(c, n),))
    monkeypatch.setattr(osnap, "top_c", wrong)
    with pytest.raises(AssertionError):
        test_snapkv_uniform_case(golden_dir)


def test_planted_snapkv_values_gathered_from_keys_are_caught(golden_dir, monkeypatch):
    real = osnap.compress

    def wrong(q_obs, K, V, n, c, kernel=3):
        return real(q_obs, K, K, n, c, kernel)
    monkeypatch.setattr(osnap, "compress", wrong)
    with pytest.raises(AssertionError):
        test_snapkv_capacity_over_length_is_identity(golden_dir)


def test_planted_threshold_off_by_one_is_caught(golden_dir, monkeypatch):
    monkeypatch.setattr(ots, "thresholds", lambda sc, K: -np.sort(-sc, axis=-1)[..., min(K, sc.shape[-1] - 1)])
    with pytest.raises(AssertionError):
        test_selection_hand_worked_example(golden_dir)


def test_planted_local_window_one_short_is_caught(monkeypatch):
    real = ots.regions

    def wrong(n, sink, local):
        sink_end, c0, c1, local_start = real(n, sink, local)
        return sink_end, c0, c1, min(local_start + 1, n)
    monkeypatch.setattr(ots, "regions", wrong)
    with pytest.raises(AssertionError):
        test_region_edge_cases()


def test_planted_interleaved_attention_groups_are_caught(monkeypatch):
    def wrong(q, K, V, S, n, sink, local):
        q, K, V = (np.asarray(t, dtype=np.float64) for t in (q, K, V))
        B, Hq, d = q.shape
        Hkv = K.shape[1]
        out, lse = np.zeros((B, Hq, d)), np.zeros((B, Hq))
        for b in range(B):
            T = ots.attended_tokens(S[b], n, sink, local)
            for h in range(Hq):
                g = h % Hkv                                      # interleaved instead of blocked
                z = K[b, g, T, :] @ q[b, h] / np.sqrt(d)
                p = np.exp(z - z.max())
                out[b, h] = p @ V[b, g, T, :] / p.sum()
                lse[b, h] = z.max() + np.log(p.sum())
        return out, lse
    monkeypatch.setattr(ots, "sparse_attention", wrong)
    with pytest.raises(AssertionError):
        test_full_budget_equals_dense_sdpa(777)
