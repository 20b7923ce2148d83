"""GPU parity of snapkv_compress against the fp64 oracle.

The kept indices must pass the band rule on the oracle's pooled scores
(exact except within 1e-4 * max p of the cutoff), and the compacted K and V
rows must be bit copies of the input rows at the GPU's own indices."""

import numpy as np
import pytest
import torch

import synth
from oracle import snapkv as osnap
from tests.parity_rules import check_topc

pytestmark = pytest.mark.gpu

qasc = pytest.importorskip("query_aware_sparse_compressed_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qasc._lib.load()


def run_snap(cfg, layer=0, device="cpu", check_b=None, mutate=None):
    x_cpu = synth.snap_layer(cfg, layer, device=device)
    if mutate is not None:
        mutate(x_cpu)
    x = {k: v.cuda() for k, v in x_cpu.items()}
    B, Hq, Hkv, n, cap, w = cfg.B, cfg.Hq, cfg.Hkv, cfg.n, cfg.cap, cfg.window
    cc = min(cfg.c, n)
    # outputs inside canary-filled buffers: nothing may be written around them
    G = 128
    idx_buf = torch.full((B * Hkv * cc + 2 * G,), -7, dtype=torch.int32, device="cuda")
    idx = idx_buf[G:G + B * Hkv * cc].view(B, Hkv, cc)
    ko_buf = torch.full((B * Hkv * cc * 128 + 2 * G,), -3.0, dtype=torch.bfloat16, device="cuda")
    vo_buf = torch.full_like(ko_buf, -5.0)
    Ko = ko_buf[G:G + B * Hkv * cc * 128].view(B, Hkv, cc, 128)
    Vo = vo_buf[G:G + B * Hkv * cc * 128].view(B, Hkv, cc, 128)
    ws = qasc.alloc_workspace(qasc.snapkv_workspace_bytes(B, Hq, Hkv, n, cap, cfg.c, w, cfg.pool_k))
    qasc.snapkv_compress(x["q_obs"], x["K"], x["V"], idx, Ko, Vo, ws, n=n, c=cfg.c, pool_k=cfg.pool_k)
    qasc.qasc_device_error()
    torch.cuda.synchronize()
    for buf, fill, nm in ((idx_buf, -7, "idx"), (ko_buf, -3.0, "K_out"), (vo_buf, -5.0, "V_out")):
        assert bool((buf[:G] == fill).all()) and bool((buf[-G:] == fill).all()), "%s: write outside the output" % nm
    idx_c = idx.cpu().numpy().astype(np.int64)
    # compacted rows are bit copies of the rows the GPU chose
    Kc = x["K"].cpu()
    Vc = x["V"].cpu()
    for b in range(B):
        for g in range(Hkv):
            assert torch.equal(Ko[b, g].cpu(), Kc[b, g, idx_c[b, g]])
            assert torch.equal(Vo[b, g].cpu(), Vc[b, g, idx_c[b, g]])
    bs = range(B) if check_b is None else [check_b]
    for b in bs:
        q64 = synth.to_f64(x["q_obs"][b:b + 1])
        K64 = synth.to_f64(x["K"][b:b + 1, :, :n])
        a = osnap.window_mean(q64, K64, n)
        p = osnap.pool(a, cfg.pool_k)
        for g in range(Hkv):
            check_topc(idx_c[b, g], p[0, g], cfg.c)
    return idx_c


S = synth.SNAP_CONFIGS["snapkv"]


@pytest.mark.parametrize("n,c", [(1, 4), (5, 3), (100, 40), (129, 128), (1000, 64), (4097, 4096), (3000, 5000)])
def test_single_group_lengths(n, c):
    run_snap(S.with_(B=1, Hq=4, Hkv=1, n=n, c=c))


def test_shrunk_llama8b_shape():
    run_snap(S.with_(n=3000, c=256))


def test_group_smaller_than_tile_and_ncap():
    # Gq = 2 heads x w = 32 rows = 64 of the 128 tile rows; n < n_cap
    run_snap(S.with_(B=2, Hq=4, Hkv=2, n=2500, n_cap=2600, c=300))


def test_single_row_window_and_wide_pool():
    run_snap(S.with_(B=1, Hq=2, Hkv=2, n=700, c=50, window=1))
    run_snap(S.with_(B=1, Hq=4, Hkv=1, n=700, c=50, pool_k=5))


def test_capacity_over_length_is_identity():
    cfg = S.with_(B=1, Hq=8, Hkv=2, n=300, c=4096)
    idx = run_snap(cfg)
    assert np.array_equal(idx, np.broadcast_to(np.arange(300), idx.shape))


def test_deterministic_repeat():
    cfg = S.with_(B=1, Hq=8, Hkv=2, n=5000, c=500)
    a = run_snap(cfg)
    b = run_snap(cfg)
    assert np.array_equal(a, b)


def test_zero_window_ties_go_to_lower_indices():
    """A zero observation window makes every logit 0: every key's window mean
    is the same value (1/n in each row), so the pooled scores of the interior
    keys tie exactly and the two end keys (padded with one zero) are lower.
    The top c are then keys 1..c (ties to the lower index), which exercises
    the top-c with one digit holding more keys than rank 0 can gather."""
    cfg = S.with_(B=1, Hq=4, Hkv=1, n=20000, c=3000)

    def zero_q(x):
        x["q_obs"].zero_()

    idx = run_snap(cfg, mutate=zero_q)
    assert np.array_equal(idx[0, 0], np.arange(1, 3001))


@pytest.mark.slow
def test_full_size_layer():
    # every sequence of the layer against the oracle (each KV head's top-c)
    run_snap(S, device="cuda")
