"""The benchmark's N-rank path on the CPU: world size 2 over gloo.

The path does not shard (every rank is an independent replica of the step), so
the only cross-rank logic is the timing: the job is as slow as its slowest rank,
and its throughput is the per-rank work times the ranks.  The reference arm runs
on rank 0 only.
"""
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.env_rank()
        slow = 2.5 if rank == 1 else 1.0          # rank 1 is the slower replica
        q.put((r, lr, w, bench.max_over_ranks(slow, w), bench.job_value(10.0, w)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_is_the_max_and_value_scales():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29000 + os.getpid() % 2000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=5) for _ in range(2))
    assert [o[:3] for o in out] == [(0, 0, 2), (1, 1, 2)]
    assert all(o[3] == 2.5 for o in out)          # every rank reports the slowest time
    assert all(o[4] == 20.0 for o in out)         # whole-job throughput: two replicas


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25, 1) == 1.25 and bench.job_value(3.0, 1) == 3.0


def test_reference_arm_other_ranks_exit_without_work():
    # rank 1 of 2 under the launcher: the oracle arm prints nothing and exits 0
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3", "--gpus", "2"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
