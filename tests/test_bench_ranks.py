"""Host logic of bench.py for N > 1 ranks, run as two gloo processes on the CPU.

The decode block has no cross-GPU exchange, so N GPUs run N independent
replicas; the job's time per step is the maximum over ranks, and rank 0
alone prints the JSON line (the reference arm's other ranks exit without
work).
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank)})
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        ms = bench.max_over_ranks(1.5 + 2.0 * rank, "cpu", w)
        q.put((r, local, w, ms))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1] and [o[1] for o in out] == [0, 1]
    assert all(o[2] == 2 for o in out)
    assert all(o[3] == 3.5 for o in out)  # both ranks report the slower rank's time


def test_single_rank_is_identity():
    assert bench.max_over_ranks(2.25, "cpu", 1) == 2.25


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
