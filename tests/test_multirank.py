"""Multi-rank host logic of bench.py on CPU: two gloo ranks (world size 2).

bench.py runs one replica of the decode workload per GPU (weak scaling, no
collective on the data path); the only cross-rank steps are the barrier and
the max over ranks of the timed region.  These tests run that logic with the
gloo backend and check the whole-job aggregate and the reference arm's
rank-0-only output.
"""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench
    import workloads as wl

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # every rank times its own replica; the job's time is the slowest one
        ms = 10.0 + 7.5 * rank
        dist.barrier()
        slow = bench.max_over_ranks(torch, dist, ms, "cpu")
        # each rank builds its replica's inputs from the same seeds
        w = wl.decode_outlier(256)
        k, _ = w.kv(0)
        digest = float(np.abs(k.astype(np.float64)).sum())
        got = [None] * world
        dist.all_gather_object(got, digest)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"slow": slow, "digests": got,
                       "value": bench.whole_job_gbs(world, 4, 1_000_000_000, slow)}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_replica_inputs(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    for r in res:
        assert r["slow"] == 17.5                       # max, not rank 0's own time
        assert r["digests"][0] == r["digests"][1]     # identical replicas
        # 2 ranks x 4 steps x 1 GB in 17.5 ms
        assert r["value"] == pytest.approx(2 * 4 * 1.0 / 17.5e-3)


def test_reference_arm_prints_on_rank0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "1"], env=env, capture_output=True, text=True, timeout=120)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""


def test_reference_arm_line_matches_the_headline_config():
    """Rank 0 of the reference arm times the oracle on the headline's own config,
    metric and unit, and reports its sample as the cpu_baseline."""
    sys.path.insert(0, ROOT)
    import bench
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1"], env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["config"] == bench.headline_config(1, bench.LAYERS)
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and "sample" in d["cpu_baseline"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_whole_job_value_scales_with_ranks():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_gbs(1, 10, 2_000_000_000, 5.0)
    two = bench.whole_job_gbs(2, 10, 2_000_000_000, 5.0)
    assert two == pytest.approx(2 * one)
    assert one == pytest.approx(10 * 2.0 / 5e-3)
