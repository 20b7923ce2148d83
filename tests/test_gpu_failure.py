"""The failure path every kernel shares, exercised on the GPU without a
fault: a bounded wait on a barrier that nothing arrives on gives up, the
kernel records a timeout and returns, qasc_device_error() reports it once,
and the context keeps working."""

import time

import pytest
import torch

import synth
from oracle import tokenselect as ots

pytestmark = pytest.mark.gpu

qasc = pytest.importorskip("query_aware_sparse_compressed_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qasc._lib.load()


def test_bounded_wait_times_out_and_is_reported_once():
    qasc.qasc_device_error()                       # start from a clear error word
    t0 = time.perf_counter()
    qasc.qasc_selftest_bounded_wait(20000)         # 20 ms
    with pytest.raises(qasc.QascError) as e:
        qasc.qasc_device_error()
    elapsed = time.perf_counter() - t0
    assert e.value.status == 5                     # QASC_ERR_TIMEOUT
    assert 0.015 < elapsed < 5.0
    qasc.qasc_device_error()                       # reported once, then cleared


def test_context_usable_after_a_timeout():
    qasc.qasc_selftest_bounded_wait(1000)
    with pytest.raises(qasc.QascError):
        qasc.qasc_device_error()
    cfg = synth.DECODE_CONFIGS["tiny"]
    x = {k: v.cuda() for k, v in synth.decode_layer(cfg, 0).items()}
    n, sink, local = cfg.n, cfg.sink, cfg.local
    K = ots.budget_tokens(n, cfg.budget_permille, sink, local)
    index = torch.zeros((cfg.B, cfg.Hkv, x["K"].shape[2], 32), dtype=torch.bfloat16, device="cuda")
    qasc.ts_index_append(x["K"], x["W"], index, 0, n, Hq=cfg.Hq, n=n)
    sel = torch.empty((cfg.B, K), dtype=torch.int32, device="cuda")
    ws = qasc.alloc_workspace(qasc.ts_select_workspace_bytes(cfg.B, cfg.Hq, cfg.Hkv, n, x["K"].shape[2], K, sink,
                                                             local))
    qasc.ts_score_vote_select(x["q"], x["W"], index, sel, ws, n=n, K=K, sink=sink, local=local)
    qasc.qasc_device_error()
    s = sel.cpu()
    assert s.shape == (cfg.B, K) and bool((s[:, 1:] > s[:, :-1]).all())
