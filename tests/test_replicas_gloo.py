"""The bench's multi-process path on CPU: two gloo ranks.

The layer does not shard (one replica per GPU), so the host logic is all
there is to test without GPUs: rank set-up from the environment, the
barrier, the max-over-ranks time with the summed tokens, and the reference
arm that runs on rank 0 only while the other ranks exit without work.
"""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(ws),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import argparse
    import bench
    try:
        got_ws, got_rank, _ = bench.dist_env()
        dist = bench.init_dist(got_ws, "gloo")
        bench.barrier(dist)
        # rank r took 1 + r seconds for 10 (r + 1) tokens
        t, u = bench.aggregate_over_ranks(dist, 1.0 + rank, 10.0 * (rank + 1))
        args = argparse.Namespace(config=0, steps=2, warmup=1, tokens=0)
        ref = bench.run_reference(args)
        bench.barrier(dist)
        q.put((rank, got_ws, got_rank, t, u, ref))
        dist.destroy_process_group()
    except Exception as e:  # reported to the parent
        q.put((rank, "error", repr(e)))


def test_two_gloo_ranks():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        item = q.get(timeout=120)
        res[item[0]] = item
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        assert res[r][1] != "error", res[r]
        _, ws, rank, t, u, ref = res[r]
        assert (ws, rank) == (2, r)
        assert (t, u) == (2.0, 30.0)  # max of the times, sum of the tokens
    ref0, ref1 = res[0][5], res[1][5]
    assert ref1 is None
    assert ref0["impl"] == "reference" and ref0["n_gpus"] == 2
    assert ref0["config"]["parallelism"] == "replicas"
    assert ref0["cpu_baseline"]["kind"] == "oracle" and ref0["value"] > 0
    assert ref0["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_line_keys(monkeypatch):
    """The reference arm's JSON line carries every key of the bench contract
    (single process: rank 0 runs it)."""
    import argparse
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    ref = bench.run_reference(argparse.Namespace(config=0, steps=3, warmup=1, tokens=0))
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "impl", "cpu_baseline", "e2e"):
        assert key in ref, key
    assert ref["impl"] == "reference" and ref["n_gpus"] == 1 and ref["steps"] == 3
    assert ref["metric"] == bench.METRIC and ref["unit"] == bench.UNIT
    assert ref["config"]["workload"] == "tiny-h256-e8-top2"
    assert ref["config"]["parallelism"] == "single-gpu"
    assert ref["e2e"]["unit"] == bench.UNIT and ref["e2e"]["value"] == ref["value"]
    assert "3 tokens" in ref["cpu_baseline"]["sample"]  # every requested step timed
