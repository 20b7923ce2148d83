"""Host logic of bench.py: argument defaults, byte accounting, rank
aggregation (max time over ranks, sum of units) over a 2-rank gloo group."""

import os

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import synth


def test_defaults_and_workload():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.steps >= 10
    assert a.workload == "llama8b_long" and a.budget == 200


def test_algorithmic_bytes_128k_budget20():
    cfg = synth.DECODE_CONFIGS["llama8b_long"]
    from oracle.tokenselect import budget_tokens
    K = budget_tokens(cfg.n, 200, cfg.sink, cfg.local)
    assert K == 26214
    ab = bench.algorithmic_bytes(cfg, K)
    assert ab["index"] == 4 * 8 * (131072 - 260) * 64
    assert ab["gather"] == 4 * 8 * (26214 + 260) * 512
    assert abs(ab["total"] / 1e6 - 701.8) < 0.5


def test_aggregate_takes_slowest_rank():
    v, t = bench.aggregate([2.0, 2.5], [100, 100], 2)
    assert t == 2.5 and v == 80.0


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = torch.tensor([1.0 + rank, 3.0 - rank])
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    q.put((rank, t.tolist()))
    dist.destroy_process_group()


def test_two_rank_max_reduce_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(60)
    got = dict(q.get(timeout=5) for _ in range(2))
    assert got[0] == got[1] == [2.0, 3.0]


def test_peaks_reads_measured_file():
    peak, kind = bench.peaks()
    assert peak > 1000 and kind in ("measured", "fallback")
