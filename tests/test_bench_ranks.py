"""bench.py's multi-rank host logic on CPU: two gloo ranks stand in for two
GPUs (every rank runs the whole workload; the job's time is the slowest
rank's and its throughput counts every rank's bytes), and the reference arm
does no work on ranks other than 0."""
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        sec = 1.0 + 0.5 * rank  # rank 1 is the slower one
        job = bench.max_over_ranks(sec, dist, torch, device="cpu")
        out[rank] = job
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world, port = 2, _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert dict(out) == {0: 1.5, 1: 1.5}
    # two replicas each streaming 1e9 bytes per step, 10 steps, the slower one in 1.5 s
    assert abs(bench.job_gbps(world, 1e9, 10, 1.5) - 2 * 10 / 1.5) < 1e-12


def test_single_rank_time_is_its_own():
    assert bench.max_over_ranks(0.25, None, torch) == 0.25


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_capture_hash_ignores_comments_not_code():
    a = "int f(int x) { return x + 1; }  // one\n/* two */\n"
    b = "// another comment\nint f(int x) {\n  return x + 1;\n}\n"
    c = "int f(int x) { return x + 2; }\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
