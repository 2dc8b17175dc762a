"""Multi-rank control plane of bench.py on CPU (gloo, world size 2).

The path needs no data exchange between GPUs: under torchrun each rank runs
an independent replica, and ranks only meet at barriers and in the
max-over-ranks reduction of the timed region. These tests run that logic as
two CPU processes.
"""
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


def _rank_main(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    w, r, local = bench.dist_env()
    dist = bench.init_dist(w)
    bench.barrier(dist)
    slowest = bench.max_over_ranks(dist, 10.0 + 5.0 * r)      # rank 1 is slower
    bench.barrier(dist)
    out_q.put((r, w, local, slowest))
    dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2, 0, 15.0), (1, 2, 1, 15.0)]


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.init_dist(1) is None
    assert bench.max_over_ranks(None, 3.5) == 3.5


@pytest.mark.parametrize("rank", [1])
def test_reference_arm_is_silent_on_other_ranks(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
