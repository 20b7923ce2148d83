"""Seeded synthetic inputs shaped like the pages' workloads.

This module is shared by the tests, the bench and the oracle checks.  It only
draws and shapes random tensors; it contains none of the method's arithmetic
(no scoring, thresholds, voting, selection, softmax or pooling).

Workloads (LLaMA-3-8B / 70B grouped-query shapes at 4K-128K context, the
TokenSelect budget sweep, and SnapKV's window 32 / kernel 3 / capacity 4096):

  tiny      1 layer,  B1, 8 q / 2 KV heads,  n=4096,   budget 10 %, 16 needles per q head
  llama8b   32 layers, B1, 32 / 8,           n=32768,  budget 20 %, 16 needles per q head
  llama8b_long 32 layers, B4, 32 / 8,        n=131072, budgets 5/10/15/20/30 %,
                                             1 % of key rows heavy-tailed (Student t, nu=3, / sqrt 3)
  llama70b  80 layers, B2, 64 / 8,           n=65536,  budget 15 %, 16 needles per q head
  snapkv    32 layers, B2, 32 / 8,           n=65536,  w=32, c=4096, pool kernel 3

Every tensor has its own seed: 1000 * config_id + 10 * layer + tensor_id.
A "needle" for query head h is a key row 3 * q_h / |q_h| * sqrt(d) plus
N(0, 0.3^2) noise per element, planted in its KV head at a uniformly drawn
candidate position (positions distinct within a KV head).
"""

from dataclasses import dataclass, replace
import math

import torch

D = 128
D_IDX = 32

# tensor ids inside one (config, layer)
_T_Q, _T_K, _T_V, _T_W, _T_NPOS, _T_NNOISE, _T_HROWS, _T_HVAL, _T_QOBS, _T_SEL = range(1, 11)


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    config_id: int
    layers: int
    B: int
    Hq: int
    Hkv: int
    n: int
    budget_permille: int
    needles_per_qhead: int = 0
    heavy_frac_permille: int = 0
    sink: int = 4
    local: int = 256
    vmin: int = 1
    n_cap: int = 0          # 0 -> n

    @property
    def cap(self):
        return self.n_cap or self.n

    def with_(self, **kw):
        return replace(self, **kw)


@dataclass(frozen=True)
class SnapConfig:
    name: str
    config_id: int
    layers: int
    B: int
    Hq: int
    Hkv: int
    n: int
    window: int = 32
    c: int = 4096
    pool_k: int = 3
    n_cap: int = 0

    @property
    def cap(self):
        return self.n_cap or self.n

    def with_(self, **kw):
        return replace(self, **kw)


DECODE_CONFIGS = {
    "tiny": DecodeConfig("tiny", 1, 1, 1, 8, 2, 4096, 100, needles_per_qhead=16),
    "llama8b": DecodeConfig("llama8b", 2, 32, 1, 32, 8, 32768, 200, needles_per_qhead=16),
    "llama8b_long": DecodeConfig("llama8b_long", 3, 32, 4, 32, 8, 131072, 200,
                                 heavy_frac_permille=10),
    "llama70b": DecodeConfig("llama70b", 4, 80, 2, 64, 8, 65536, 150, needles_per_qhead=16),
}
BUDGET_SWEEP_PERMILLE = (50, 100, 150, 200, 300)

SNAP_CONFIGS = {
    "snapkv": SnapConfig("snapkv", 5, 32, 2, 32, 8, 65536),
}


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _seed(config_id, layer, tensor_id):
    return 1000 * config_id + 10 * layer + tensor_id


def _randn_bf16(shape, seed, device, std=1.0):
    x = torch.randn(shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(torch.bfloat16)


def projection(config_id, layer, Hkv, device="cpu"):
    """Per-KV-head projection W [Hkv, d, d_idx], N(0, 1/d) drawn in fp32 and
    rounded once to bf16."""
    return _randn_bf16((Hkv, D, D_IDX), _seed(config_id, layer, _T_W), device,
                       std=1.0 / math.sqrt(D))


def decode_layer(cfg: DecodeConfig, layer: int = 0, device="cpu"):
    """Inputs of one decode layer-step: dict(q, K, V, W, needles).

    q [B,Hq,d], K/V [B,Hkv,n_cap,d], W [Hkv,d,d_idx], all bf16 on `device`;
    rows n..n_cap-1 of K/V are zero.  `needles` is an int64 tensor
    [B, Hq, P] of planted positions (P may be 0).
    """
    B, Hq, Hkv, n, cap = cfg.B, cfg.Hq, cfg.Hkv, cfg.n, cfg.cap
    cid = cfg.config_id
    q = _randn_bf16((B, Hq, D), _seed(cid, layer, _T_Q), device)
    K = torch.zeros((B, Hkv, cap, D), dtype=torch.bfloat16, device=device)
    V = torch.zeros((B, Hkv, cap, D), dtype=torch.bfloat16, device=device)
    K[:, :, :n] = _randn_bf16((B, Hkv, n, D), _seed(cid, layer, _T_K), device)
    V[:, :, :n] = _randn_bf16((B, Hkv, n, D), _seed(cid, layer, _T_V), device)
    W = projection(cid, layer, Hkv, device)

    c0 = cfg.sink
    c1 = max(n - cfg.local, c0)
    nc = c1 - c0
    group = Hq // Hkv

    if cfg.heavy_frac_permille and nc > 0:
        rows = max(1, (nc * cfg.heavy_frac_permille) // 1000)
        gsel = _gen(_seed(cid, layer, _T_HROWS), device)
        pos = torch.rand((B, Hkv, nc), generator=gsel, device=device).argsort(dim=-1)[..., :rows] + c0
        gval = _gen(_seed(cid, layer, _T_HVAL), device)
        z = torch.randn((B, Hkv, rows, D), generator=gval, device=device)
        chi = torch.randn((B, Hkv, rows, D, 3), generator=gval, device=device).pow(2).sum(-1)
        t3 = z / torch.sqrt(chi / 3.0) / math.sqrt(3.0)
        idx = pos.unsqueeze(-1).expand(-1, -1, -1, D)
        K.scatter_(2, idx, t3.to(torch.bfloat16))

    P = cfg.needles_per_qhead
    needles = torch.zeros((B, Hq, 0), dtype=torch.int64, device=device)
    if P > 0 and nc >= group * P:
        gpos = _gen(_seed(cid, layer, _T_NPOS), device)
        perm = torch.rand((B, Hkv, nc), generator=gpos, device=device).argsort(dim=-1)
        pos = perm[..., :group * P].reshape(B, Hkv, group, P) + c0      # [B,Hkv,G,P]
        gno = _gen(_seed(cid, layer, _T_NNOISE), device)
        noise = 0.3 * torch.randn((B, Hkv, group, P, D), generator=gno, device=device)
        qf = q.float().reshape(B, Hkv, group, D)
        unit = qf / qf.norm(dim=-1, keepdim=True).clamp_min(1e-30)
        rows = 3.0 * unit.unsqueeze(3) * math.sqrt(D) + noise        # [B,Hkv,G,P,D]
        idx = pos.reshape(B, Hkv, group * P, 1).expand(-1, -1, -1, D)
        K.scatter_(2, idx, rows.reshape(B, Hkv, group * P, D).to(torch.bfloat16))
        needles = pos.reshape(B, Hq, P)
    return dict(q=q, K=K, V=V, W=W, needles=needles)


def random_selection(B, n, K, sink, local, seed, device="cpu"):
    """A seeded, sorted, duplicate-free candidate set [B, K] int32 drawn
    uniformly from C, for exercising the attention path on its own."""
    c0 = sink
    c1 = max(n - local, c0)
    g = _gen(seed, device)
    perm = torch.rand((B, c1 - c0), generator=g, device=device).argsort(dim=-1)[:, :K]
    return (perm + c0).sort(dim=-1).values.to(torch.int32)


def snap_layer(cfg: SnapConfig, layer: int = 0, device="cpu"):
    """Inputs of one SnapKV compaction: dict(q_obs [B,Hq,w,d], K, V)."""
    B, Hq, Hkv, n, cap, w = cfg.B, cfg.Hq, cfg.Hkv, cfg.n, cfg.cap, cfg.window
    cid = cfg.config_id
    q_obs = _randn_bf16((B, Hq, w, D), _seed(cid, layer, _T_QOBS), device)
    K = torch.zeros((B, Hkv, cap, D), dtype=torch.bfloat16, device=device)
    V = torch.zeros((B, Hkv, cap, D), dtype=torch.bfloat16, device=device)
    K[:, :, :n] = _randn_bf16((B, Hkv, n, D), _seed(cid, layer, _T_K), device)
    V[:, :, :n] = _randn_bf16((B, Hkv, n, D), _seed(cid, layer, _T_V), device)
    return dict(q_obs=q_obs, K=K, V=V)


def to_f64(t):
    """Exact widening of a (bf16) torch tensor to a NumPy fp64 array."""
    return t.detach().to("cpu").to(torch.float64).numpy()
