"""The N > 1 host logic of bench.py, run as two gloo ranks on the CPU.

With several GPUs every rank runs its own replica of the layer; the ranks meet
only at the barriers around the timed region and in the max-over-ranks
reduction of the duration.  These tests run exactly those helpers over gloo:
the reduction must give the slowest rank's time on every rank, the job
throughput must count every rank's tokens over that time, the replicas must
draw different batches, and the reference arm must leave ranks other than 0
without work or output.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, ms_of_rank, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    bench.init_ranks(torch, w, backend="gloo")
    bench.barrier(torch, w)
    ms = bench.max_over_ranks(torch, ms_of_rank[r], w, "cpu")
    value = bench.job_tokens_per_s(w, 8192, 10, ms)
    seed = bench.replica_seed(1234, r)
    bench.finish_ranks(torch, w)
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"ms": ms, "value": value, "seed": seed}, f)


def test_two_gloo_ranks_max_and_job_throughput(tmp_path):
    world = 2
    ms_of_rank = [812.5, 1093.75]
    mp.start_processes(_rank_main, args=(world, _free_port(), ms_of_rank, str(tmp_path)),
                       nprocs=world, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    slowest = max(ms_of_rank)
    for r in res:
        assert r["ms"] == slowest
        # 2 ranks x 8192 tokens x 10 steps over the slowest rank's 1.09375 s
        assert r["value"] == pytest.approx(2 * 8192 * 10 / 1.09375, rel=1e-12)
    assert res[0]["seed"] == 1234
    assert res[0]["seed"] != res[1]["seed"]


def test_single_rank_needs_no_process_group():
    assert not torch.distributed.is_initialized()
    bench.init_ranks(torch, 1, backend="gloo")
    assert not torch.distributed.is_initialized()
    assert bench.max_over_ranks(torch, 12.5, 1, "cpu") == 12.5
    assert bench.job_tokens_per_s(1, 4096, 4, 2000.0) == pytest.approx(8192.0)
    bench.finish_ranks(torch, 1)


def test_replica_seeds_distinct_across_eight_ranks():
    seeds = [bench.replica_seed(77, r) for r in range(8)]
    assert len(set(seeds)) == 8 and seeds[0] == 77


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=240)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
