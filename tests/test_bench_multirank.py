"""The benchmark's multi-rank timing path on CPU ranks (gloo, world size 2).

With N GPUs the benchmark runs one replica per rank (the layer has no data
exchange): every rank times its own steps between barriers, the step time
reported is the maximum over ranks, and only rank 0 prints.  These tests run
the same helpers in two CPU processes; no GPU is involved.
"""
import os
import socket
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_ranks(body, world=2, timeout=120):
    """Runs `body` (Python source) in `world` processes with the torchrun
    environment set; returns their stdout."""
    port = _free_port()
    procs = []
    for rank in range(world):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), PYTHONPATH=ROOT)
        procs.append(subprocess.Popen([sys.executable, "-c", textwrap.dedent(body)], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=timeout)
        except subprocess.TimeoutExpired:
            p.kill()
            out, err = p.communicate()
        assert p.returncode == 0, err[-2000:]
        outs.append(out)
    return outs


def test_barrier_and_max_over_ranks():
    outs = _run_ranks("""
        import bench
        ws, rank, local = bench.dist_env()
        dist = bench.init_dist("gloo")
        assert dist is not None and dist.get_world_size() == ws == 2
        bench.barrier(dist)
        # each rank reports its own step time; the job's time is the slowest
        t = bench.max_over_ranks(dist, 1.5 + rank)
        print("rank %d max %.3f" % (rank, t))
        dist.destroy_process_group()
    """)
    assert outs[0].strip() == "rank 0 max 2.500"
    assert outs[1].strip() == "rank 1 max 2.500"


def test_single_rank_needs_no_process_group():
    import bench
    env = {k: os.environ.pop(k) for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK") if k in os.environ}
    try:
        assert bench.dist_env() == (1, 0, 0)
        assert bench.init_dist("gloo") is None
        assert bench.max_over_ranks(None, 3.25) == 3.25
    finally:
        os.environ.update(env)


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun only rank 0 times the oracle and prints; the others exit
    at once (here: rank 1 of 2 returns without output or work)."""
    outs = _run_ranks("""
        import sys
        import bench
        ws, rank, local = bench.dist_env()
        if rank == 1:
            sys.argv = ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"]
            bench.main()
            print("rank 1 done")
    """)
    assert outs[0].strip() == ""
    assert outs[1].strip() == "rank 1 done"
