"""ts_sparse_attn_noalloc: attention for callers that cannot allocate device
memory (its split-K scratch is a fixed area inside the library instead of a
caller workspace).  Checked through the C ABI against ts_sparse_attn on the
same inputs, on consecutive calls, against the oracle directly, and for its
size limit (a refused call writes nothing and the next call is still right).
Collected last so that a failure here cannot hide failures elsewhere."""

import numpy as np
import pytest
import torch

import synth
from oracle import tokenselect as ots
from tests.parity_rules import check_attention

pytestmark = pytest.mark.gpu

qasc = pytest.importorskip("query_aware_sparse_compressed_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qasc._lib.load()


def _inputs(cfg, K, seed):
    x = {k: v.cuda() for k, v in synth.decode_layer(cfg, 0).items()}
    sel = synth.random_selection(cfg.B, cfg.n, K, cfg.sink, cfg.local, seed).cuda()
    return x, sel


def _with_workspace(x, sel, cfg):
    B, Hq, Hkv = cfg.B, cfg.Hq, cfg.Hkv
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    ws = qasc.alloc_workspace(qasc.ts_attn_workspace_bytes(B, Hq, Hkv, cfg.n, cfg.cap, sel.shape[1],
                                                           cfg.sink, cfg.local))
    qasc.ts_sparse_attn(x["q"], x["K"], x["V"], sel, out, ws, n=cfg.n, sink=cfg.sink, local=cfg.local, lse=lse)
    return out, lse


def _no_alloc(x, sel, cfg):
    out = torch.full((cfg.B, cfg.Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((cfg.B, cfg.Hq), float("nan"), dtype=torch.float32, device="cuda")
    qasc.ts_sparse_attn_noalloc(x["q"], x["K"], x["V"], sel, out, n=cfg.n, sink=cfg.sink, local=cfg.local,
                                lse=lse)
    return out, lse


def test_no_alloc_matches_workspace_call_on_consecutive_calls():
    D = synth.DECODE_CONFIGS
    cases = [(D["llama8b"].with_(B=2, n=9000), 1700, 11), (D["tiny"], 409, 12)]
    for cfg, K, seed in cases:
        x, sel = _inputs(cfg, K, seed)
        ref_out, ref_lse = _with_workspace(x, sel, cfg)
        for _ in range(2):    # the shared area keeps the previous call's contents
            out, lse = _no_alloc(x, sel, cfg)
            torch.cuda.synchronize()
            check_attention(out.cpu().numpy(), ref_out.cpu().numpy())
            check_attention(lse.cpu().numpy(), ref_lse.cpu().numpy())
        # and against the oracle itself on the same selected sets
        q64, K64, V64 = (synth.to_f64(x[k]) for k in ("q", "K", "V"))
        want, want_lse = ots.sparse_attention(q64, K64[:, :, :cfg.n], V64[:, :, :cfg.n],
                                              sel.cpu().numpy().astype(np.int64), cfg.n, cfg.sink, cfg.local)
        check_attention(out.cpu().numpy(), want)
        check_attention(lse.cpu().numpy(), want_lse)
    qasc.qasc_device_error()


def test_no_alloc_rejects_scratch_beyond_its_area():
    # 512 sequences x 8 KV heads x 8 query heads per group: the split-K
    # partials (at least two covering CTAs x 8 groups x 8 heads x 132 floats
    # per (b, g)) far exceed the 16 MiB area, so the call must refuse up front.
    cfg = synth.DECODE_CONFIGS["tiny"].with_(B=512, Hq=64, Hkv=8, n=300, needles_per_qhead=0)
    x = synth.decode_layer(cfg, 0, device="cuda")
    out = torch.full((cfg.B, cfg.Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    with pytest.raises(qasc.QascError) as e:
        qasc.ts_sparse_attn_noalloc(x["q"], x["K"], x["V"], None, out, n=cfg.n, sink=cfg.sink, local=cfg.local)
    assert e.value.status == 3 and "built-in area" in str(e.value)
    torch.cuda.synchronize()
    assert torch.isnan(out).all(), "the refused call wrote its output"
    # a call within the limit right after the refusal is still correct
    small = synth.DECODE_CONFIGS["tiny"]
    xs, sel = _inputs(small, 409, 13)
    ref_out, ref_lse = _with_workspace(xs, sel, small)
    got, got_lse = _no_alloc(xs, sel, small)
    torch.cuda.synchronize()
    check_attention(got.cpu().numpy(), ref_out.cpu().numpy())
    check_attention(got_lse.cpu().numpy(), ref_lse.cpu().numpy())
    qasc.qasc_device_error()
