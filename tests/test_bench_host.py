"""Host logic of the benchmark, without a GPU: the replicas' step time is the
maximum over ranks (two gloo ranks on the CPU), the whole-job value counts every
replica, and the reference arm prints nothing on ranks other than 0."""
import os
import socket
import subprocess
import sys

import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r's step takes 1 + r ms: every rank must report the slowest one
        q.put((rank, bench.max_over_ranks(1.0 + rank, world, "cpu")))
        torch.distributed.barrier()
    finally:
        torch.distributed.destroy_process_group()


def test_step_time_is_the_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2.0), (1, 2.0)]


def test_single_rank_and_job_value():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    # two replicas of 1e12 flops each in 1 ms: 2000 TFLOP/s for the job
    assert bench.job_tflops(2, 1e12, 1.0) == 2000.0
    assert bench.job_tflops(1, 1e12, 1.0) == 1000.0


def test_reference_arm_is_silent_on_other_ranks():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
