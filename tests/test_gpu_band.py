"""The per-head thresholds of the voting select on the GPU.

ts_score_vote_select_ex exposes theta_h and which route found it: the band
list (the band held theta_h) or the exact recount from the index.  Checked:
  - theta_h against the oracle's K-th largest score (fp32 scores on the GPU:
    within 1e-5 * max|score|);
  - the sampled band holds theta_h on the seeded workloads (no recount);
  - a band given by the caller: tight around theta_h gives the same S as the
    sampled band bit for bit; a band wholly above or below theta_h, or one
    whose list overflows, takes the recount and still gives an S that passes
    the oracle's band rule, with theta_h still within 1e-5 * max|score|.
"""

import numpy as np
import pytest
import torch

import synth
from oracle import tokenselect as ots
from tests.parity_rules import check_selection

pytestmark = pytest.mark.gpu

qasc = pytest.importorskip("query_aware_sparse_compressed_gb300")

D = synth.DECODE_CONFIGS
THETA_REL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qasc._lib.load()


def _setup(cfg, bp=None):
    x_cpu = synth.decode_layer(cfg, 0)
    x = {k: v.cuda() for k, v in x_cpu.items()}
    n, sink, local = cfg.n, cfg.sink, cfg.local
    K = ots.budget_tokens(n, cfg.budget_permille if bp is None else bp, sink, local)
    B, Hkv, n_cap = cfg.B, cfg.Hkv, cfg.cap
    index = torch.zeros((B, Hkv, n_cap, 32), dtype=torch.bfloat16, device="cuda")
    qasc.ts_index_append(x["K"], x["W"], index, 0, n, Hq=cfg.Hq, n=n)
    q64, K64, W64 = (synth.to_f64(x_cpu[k]) for k in ("q", "K", "W"))
    S_ref, info = ots.select(q64, W64, ots.index_rows(K64[:, :, :n], W64), n, K, sink, local)
    return x, index, K, S_ref, info


def _select_ex(cfg, x, index, K, band=None):
    B, Hq = cfg.B, cfg.Hq
    sel = torch.full((B, K), -1, dtype=torch.int32, device="cuda")
    theta = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
    flag = torch.full((B, Hq), -1, dtype=torch.int32, device="cuda")
    ws = qasc.alloc_workspace(qasc.ts_select_workspace_bytes(B, Hq, cfg.Hkv, cfg.n, cfg.cap, K, cfg.sink,
                                                             cfg.local))
    qasc.ts_score_vote_select_ex(x["q"], x["W"], index, sel, ws, n=cfg.n, K=K, sink=cfg.sink, local=cfg.local,
                                 theta=theta, band=band, fallback=flag)
    qasc.qasc_device_error()
    torch.cuda.synchronize()
    return sel.cpu().numpy().astype(np.int64), theta.cpu().numpy().astype(np.float64), flag.cpu().numpy()


def _check(cfg, sel, theta, info, K):
    for b in range(cfg.B):
        sc = info["scores"][b]
        tol = THETA_REL * np.abs(sc).max()
        err = np.abs(theta[b] - info["theta"][b]).max()
        assert err <= tol, "theta off by %.3g (> %.3g)" % (err, tol)
        check_selection(sel[b], sc, info["theta"][b], info["c0"], K)


CASES = [
    D["tiny"],
    D["llama8b"].with_(B=2, n=9037),
    D["llama70b"].with_(n=5000, n_cap=5120),
    D["llama8b_long"].with_(B=2, n=12000),
    D["tiny"].with_(Hq=4, Hkv=4, n=3000),
    D["tiny"].with_(Hq=8, Hkv=4, n=2500, budget_permille=300),
]
IDS = ["tiny", "8b-ragged", "70b-ncap", "long-heavy", "gq1", "gq2"]


@pytest.mark.parametrize("cfg", CASES, ids=IDS)
def test_sampled_band_holds_theta(cfg):
    x, index, K, S_ref, info = _setup(cfg)
    sel, theta, flag = _select_ex(cfg, x, index, K)
    assert (flag == 0).all(), "heads that needed the recount: %s" % np.argwhere(flag != 0).tolist()
    _check(cfg, sel, theta, info, K)
    # the plain call gives the same set
    sel2 = torch.empty((cfg.B, K), dtype=torch.int32, device="cuda")
    ws = qasc.alloc_workspace(qasc.ts_select_workspace_bytes(cfg.B, cfg.Hq, cfg.Hkv, cfg.n, cfg.cap, K, cfg.sink,
                                                             cfg.local))
    qasc.ts_score_vote_select(x["q"], x["W"], index, sel2, ws, n=cfg.n, K=K, sink=cfg.sink, local=cfg.local)
    torch.cuda.synchronize()
    assert np.array_equal(sel2.cpu().numpy(), sel)


@pytest.mark.parametrize("bp", synth.BUDGET_SWEEP_PERMILLE)
def test_sampled_band_budget_sweep(bp):
    cfg = D["llama8b_long"].with_(B=1, n=7000)
    x, index, K, S_ref, info = _setup(cfg, bp)
    sel, theta, flag = _select_ex(cfg, x, index, K)
    assert (flag == 0).all()
    _check(cfg, sel, theta, info, K)


@pytest.mark.parametrize("cfg", [CASES[0], CASES[1], CASES[4]], ids=["tiny", "8b-ragged", "gq1"])
def test_given_bands_every_route(cfg):
    x, index, K, S_ref, info = _setup(cfg)
    sel0, theta0, flag0 = _select_ex(cfg, x, index, K)
    B, Hq = cfg.B, cfg.Hq
    th = torch.from_numpy(theta0).float()
    # tight band around theta: the list route, the same set bit for bit
    tight = torch.stack([th - 1e-3, th + 1e-3], dim=-1).cuda()
    sel, theta, flag = _select_ex(cfg, x, index, K, band=tight)
    assert (flag == 0).all() and np.array_equal(sel, sel0) and np.array_equal(theta, theta0)
    # a band wholly above theta (nothing above it, nothing in it) and one
    # wholly below (every score above it): the recount
    for lo, hi in ((1e30, 2e30), (-2e30, -1e30)):
        band = torch.tensor([lo, hi], dtype=torch.float32).expand(B, Hq, 2).contiguous().cuda()
        sel, theta, flag = _select_ex(cfg, x, index, K, band=band)
        assert (flag == 1).all()
        _check(cfg, sel, theta, info, K)
    # half the heads with a useless band, half with a tight one
    mixed = tight.clone()
    mixed[:, ::2, 0] = 1e30
    mixed[:, ::2, 1] = 2e30
    sel, theta, flag = _select_ex(cfg, x, index, K, band=mixed)
    assert (flag[:, ::2] == 1).all() and (flag[:, 1::2] == 0).all()
    _check(cfg, sel, theta, info, K)


def test_unbounded_band_overflows_into_the_recount():
    # every candidate in the band: more than the list holds at this size
    cfg = D["llama8b"].with_(B=1, n=30000)
    x, index, K, S_ref, info = _setup(cfg)
    band = torch.tensor([-float("inf"), float("inf")]).expand(1, cfg.Hq, 2).contiguous().cuda()
    sel, theta, flag = _select_ex(cfg, x, index, K, band=band)
    assert (flag == 1).all()
    _check(cfg, sel, theta, info, K)


def test_unbounded_band_fits_when_small():
    # at this size the list holds every candidate: the list route
    cfg = D["tiny"].with_(n=1500, needles_per_qhead=0)
    x, index, K, S_ref, info = _setup(cfg)
    band = torch.tensor([-float("inf"), float("inf")]).expand(1, cfg.Hq, 2).contiguous().cuda()
    sel, theta, flag = _select_ex(cfg, x, index, K, band=band)
    assert (flag == 0).all()
    _check(cfg, sel, theta, info, K)


@pytest.mark.slow
def test_full_size_128k_sampled_band():
    cfg = D["llama8b_long"]
    x = synth.decode_layer(cfg, 0, device="cuda")
    n, sink, local = cfg.n, cfg.sink, cfg.local
    index = torch.zeros((cfg.B, cfg.Hkv, n, 32), dtype=torch.bfloat16, device="cuda")
    qasc.ts_index_append(x["K"], x["W"], index, 0, n, Hq=cfg.Hq, n=n)
    for bp in synth.BUDGET_SWEEP_PERMILLE:
        K = ots.budget_tokens(n, bp, sink, local)
        sel, theta, flag = _select_ex(cfg, x, index, K)
        assert (flag == 0).all(), (bp, np.argwhere(flag != 0).tolist())
    # theta of one sequence against the oracle at 20 %
    K = ots.budget_tokens(n, 200, sink, local)
    sel, theta, flag = _select_ex(cfg, x, index, K)
    b = 2
    q64 = synth.to_f64(x["q"][b:b + 1])
    W64 = synth.to_f64(x["W"])
    idx64 = synth.to_f64(index[b:b + 1, :, :n])
    sc = ots.scores(q64, W64, idx64, n, sink, local)[0]
    th = ots.thresholds(sc[None], K)[0]
    assert np.abs(theta[b] - th).max() <= THETA_REL * np.abs(sc).max()
