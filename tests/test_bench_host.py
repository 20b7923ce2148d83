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


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CONTRACT_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                 "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e",
                 "gpu_launches"}


def _json_lines(out):
    import json
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def _check_reference_line(line, n_gpus):
    assert CONTRACT_KEYS <= set(line), CONTRACT_KEYS - set(line)
    assert line["impl"] == "reference" and line["n_gpus"] == n_gpus and line["steps"] == 1
    assert line["value"] > 0 and line["vs_baseline"] is None and line["higher_is_better"] is True
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    assert 0 < cb["effective_threads"] <= 2 * cb["cores"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_prints_one_contract_line():
    import subprocess
    import sys
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_reference_line(lines[0], 1)


def test_reference_arm_under_torchrun_prints_only_on_rank0():
    import subprocess
    import sys
    port = 29600 + os.getpid() % 1000
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
                        "reference", "--gpus", "2", "--steps", "1", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_reference_line(lines[0], 2)


def test_cpu_baseline_entry_on_a_small_workload():
    # The helper the GPU arm calls for its cpu_baseline object, run here on
    # the small decode workload with a short sample.
    from oracle.tokenselect import budget_tokens
    cfg = synth.DECODE_CONFIGS["tiny"]
    K = budget_tokens(cfg.n, cfg.budget_permille, cfg.sink, cfg.local)
    e = bench.cpu_baseline_entry(cfg, K, 0.5, "cpu", "tiny", cfg.budget_permille)
    assert set(e) == {"value", "unit", "cores", "kind", "sample", "seconds", "effective_threads", "single_thread"}
    assert e["single_thread"]["cores"] == 1 and e["single_thread"]["value"] > 0
    assert e["kind"] == "oracle" and e["unit"] == bench.UNIT and e["value"] > 0
    assert e["cores"] == len(os.sched_getaffinity(0))
    # CPU time over a sub-second sample is coarse: only a loose sanity bound.
    assert 0 < e["effective_threads"] <= 2 * e["cores"]


def test_single_thread_oracle_child():
    """The hidden oracle-only mode, run as the child the bench line's
    cpu_baseline.single_thread comes from (tiny workload, CPU inputs)."""
    r = bench.single_thread_oracle("tiny", 100, 0.2)
    assert "unavailable" not in r, r
    assert r["cores"] == 1 and r["kind"] == "oracle" and r["value"] > 0 and r["sample"]
    assert set(r["threads_env"]) == set(bench.ONE_THREAD_ENV)


def test_point_entry_fields():
    cfg = synth.DECODE_CONFIGS["llama8b"].with_(layers=8)
    from oracle.tokenselect import budget_tokens
    K = budget_tokens(cfg.n, cfg.budget_permille, cfg.sink, cfg.local)
    ab = bench.algorithmic_bytes(cfg, K)
    e = bench.point_entry(cfg, K, 200, dict(layer_s=1e-4, sel_s=4e-5, attn_s=5e-5, bytes=ab), 6000.0, "8 layers")
    assert e["layer_steps_per_s"] == 10000.0 and e["ms_per_layer"] == 0.1
    assert e["hbm_gbs"] == round(ab["total"] / 1e-4 / 1e9, 1)
    assert abs(e["frac_of_peak"] - e["hbm_gbs"] / 6000.0) < 1e-3
    assert "K=%d" % K in e["workload"] and "budget 20%" in e["workload"]
