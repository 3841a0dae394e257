"""The multi-rank path of bench.py on CPU: two gloo ranks on 127.0.0.1.

bench.py runs replicas (each rank the full workload on its own GPU, no
collective on the data path); the only cross-rank steps are the barrier, the
max of the ranks' times and the reference arm running on rank 0 alone. Those
are exercised here with world_size 2 and no GPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        got = bench.max_over_ranks(ms, torch.device("cpu"), world)
        value = bench.whole_job_tflops(2.0e12, 4, world, got)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"max_ms": got, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["max_ms"] == 15.0
        # 2 ranks x 4 steps x 2 TFLOP in 15 ms
        assert abs(r["value"] - 2 * 4 * 2.0 / 0.015) < 1e-6


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, "cpu", 1) == 3.5


@pytest.mark.parametrize("rank", [1])
def test_reference_arm_non_zero_rank_exits_without_work(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
