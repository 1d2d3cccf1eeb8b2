"""The benchmark's multi-GPU path, on the CPU with two gloo ranks.

The path has no exchange step: every rank runs an independent replica (its own seeded
batch), the ranks meet only at the barrier around the timed region and at the max-over-
ranks reduction of the step times, and the job's throughput is world x per-rank units over
the slowest rank's time. These tests exercise exactly that host logic without a GPU.
"""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        assert b.dist_env() == (rank, world, rank)
        # rank r pretends to have taken (1 + r) ms per step and (10 - r) ms per kernel
        got = b.max_over_ranks([1.0 + rank, 10.0 - rank, 0.0], world, "cpu")
        value = b.whole_job_value(3.0, world, got[0])
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"max": got, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_replica(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["max"] == [2.0, 10.0, 0.0]          # max over ranks, element by element
        assert r["value"] == pytest.approx(3.0 * 2 / 2e-3)  # 2 replicas x 3 units / slowest 2 ms


def test_single_rank_needs_no_process_group():
    b = _bench()
    assert b.max_over_ranks([1.5, 2.5], 1, "cpu") == [1.5, 2.5]
    assert b.whole_job_value(4.0, 1, 2.0) == pytest.approx(2000.0)


def test_reference_arm_prints_only_on_rank_zero():
    """Under torchrun the oracle arm runs on rank 0 alone; the other ranks exit 0 silently."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1", MASTER_PORT="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "1",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


@pytest.mark.parametrize("extra", [["--config", "1"], ["--op", "cache_write", "--config", "2"]])
def test_reference_arm_line_keeps_the_contract(extra):
    """Rank 0's oracle arm prints one JSON line with the contract's keys (small workloads)."""
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *extra,
                        "--steps", "1", "--warmup", "0", "--cpu-seconds", "1"], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert "workload" in d["config"]
