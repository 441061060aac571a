"""The benchmark's multi-rank logic on CPU: two gloo ranks agree on the slowest rank's time and report the
whole job's throughput (weak scaling); the reference arm's non-zero ranks exit at once."""

import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms_local = [3.0, 5.0][rank]
        ms, value = bench.aggregate(dist, world, 2e12, ms_local, torch.device("cpu"))
        out[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for rank in range(world):
        ms, value = out[rank]
        assert ms == 5.0
        assert abs(value - world * 2e12 / 5e-3 / 1e12) < 1e-9


def test_single_process_aggregate_is_the_local_time():
    sys.path.insert(0, ROOT)
    import bench
    ms, value = bench.aggregate(None, 1, 1e12, 4.0, None)
    assert ms == 4.0 and abs(value - 250.0) < 1e-12


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1", MASTER_PORT="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
