"""GPU parity of the dense (full) attention baseline against the fp64 oracle.

ts_dense_attn attends every cached token; the oracle is the same plain
softmax attention over [0, n) in fp64 (oracle.tokenselect.dense_attention).
Bar: max-abs <= 1e-3 and relative L2 <= 1e-3 on out and lse.
"""

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


def gpu_dense(x, n):
    q, K, V = x["q"], x["K"], x["V"]
    B, Hq, _ = q.shape
    _, Hkv, n_cap, _ = K.shape
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    ws = qasc.alloc_workspace(qasc.ts_dense_attn_workspace_bytes(B, Hq, Hkv, n, n_cap))
    qasc.ts_dense_attn(q, K, V, out, ws, n=n, lse=lse)
    qasc.qasc_device_error()
    return out, lse


def check_against_oracle(x, n, bs=None, hs=None):
    out, lse = gpu_dense(x, n)
    q64 = synth.to_f64(x["q"])
    K64 = synth.to_f64(x["K"][:, :, :n])
    V64 = synth.to_f64(x["V"][:, :, :n])
    if bs is not None:   # a sample of (b, h): the oracle evaluates those heads only
        Hq, Hkv = q64.shape[1], K64.shape[1]
        for b in bs:
            for h in hs:
                g = h // (Hq // Hkv)
                ref, ref_lse = ots.dense_attention(q64[b:b + 1, h:h + 1], K64[b:b + 1, g:g + 1],
                                                   V64[b:b + 1, g:g + 1], n)
                check_attention(out[b:b + 1, h:h + 1].cpu().numpy(), ref)
                check_attention(lse[b:b + 1, h:h + 1].cpu().numpy(), ref_lse)
        return
    ref, ref_lse = ots.dense_attention(q64, K64, V64, n)
    check_attention(out.cpu().numpy(), ref)
    check_attention(lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("n", [1, 7, 127, 128, 129, 1000, 4097])
def test_dense_ragged_lengths(n):
    cfg = D["tiny"].with_(B=2, n=n, n_cap=n + 3, needles_per_qhead=0)
    x = {k: v.cuda() for k, v in synth.decode_layer(cfg, 0).items()}
    check_against_oracle(x, n)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 4), (8, 2), (16, 2)])
def test_dense_group_sizes(Hq, Hkv):
    cfg = D["tiny"].with_(Hq=Hq, Hkv=Hkv, n=3000, needles_per_qhead=4)
    x = {k: v.cuda() for k, v in synth.decode_layer(cfg, 0).items()}
    check_against_oracle(x, cfg.n)


def test_dense_equals_sparse_with_every_token_selected():
    # TokenSelect with the whole candidate range selected attends every token.
    cfg = D["tiny"].with_(n=2048, needles_per_qhead=0)
    x = {k: v.cuda() for k, v in synth.decode_layer(cfg, 0).items()}
    n, sink, local = cfg.n, cfg.sink, cfg.local
    B, Hq = cfg.B, cfg.Hq
    K = ots.budget_tokens(n, 1000, sink, local)
    sel = torch.arange(sink, sink + K, dtype=torch.int32, device="cuda").repeat(B, 1).contiguous()
    out_s = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    ws = qasc.alloc_workspace(qasc.ts_attn_workspace_bytes(B, Hq, cfg.Hkv, n, n, K, sink, local))
    qasc.ts_sparse_attn(x["q"], x["K"], x["V"], sel, out_s, ws, n=n, sink=sink, local=local)
    out_d, _ = gpu_dense(x, n)
    check_attention(out_s.cpu().numpy(), out_d.double().cpu().numpy(), max_abs=1e-5, rel_l2=1e-5)


@pytest.mark.slow
def test_dense_full_size_llama8b_32k():
    cfg = D["llama8b"].with_(layers=1)
    x = synth.decode_layer(cfg, 0, device="cuda")
    check_against_oracle(x, cfg.n, bs=[0], hs=[0, 5, 17, 31])


@pytest.mark.slow
def test_dense_full_size_llama8b_128k_b4():
    cfg = D["llama8b_long"].with_(layers=1)
    x = synth.decode_layer(cfg, 0, device="cuda")
    check_against_oracle(x, cfg.n, bs=[0, 3], hs=[2, 30])
