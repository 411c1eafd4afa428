"""The N-GPU bench path on the host: two gloo ranks run bench.py's rank logic
(process group set-up, barriers, max over ranks of the timed region) and the
reference arm's rank filter. The path itself has no data exchange: each rank
is an independent replica."""
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    r, w, _ = bench.dist_setup()
    assert (r, w) == (rank, world)
    bench.barrier(w)
    # each rank's own "timed region": the reported time is the slowest rank's
    t = bench.max_over_ranks(1.0 + rank, w)
    out.put((rank, t))
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert got == [(0, 2.0), (1, 2.0)]


def test_reference_arm_runs_on_rank_zero_only():
    # rank 1 of a torchrun launch prints nothing and exits 0 without work
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1",
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
