"""The benchmark's multi-rank host logic on CPU: two gloo ranks.

The path shards across independent requests with no exchange step, so N ranks are replicas
that each own their own requests; the job's time is the slowest rank's and its throughput is
every rank's work over that time. These tests run bench.py's helpers in two spawned
processes over gloo (127.0.0.1): the max-over-ranks reduction, distinct seeded requests per
rank, and the reference arm's rule that only rank 0 works and prints.
"""
import os
import socket
import subprocess
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    from paged_sliding_window_qkv_gb300 import workloads as W
    dist.init_process_group("gloo", rank=rank, world_size=world)
    slowest = bench.max_over_ranks(1.5 + rank, world, "cpu")
    s5, s4 = bench.rank_seeds(rank)
    wl4 = W.make_workload(4, seed=s4)
    fp = int(np.asarray(wl4.families[0].batch.start_pos).sum())  # a fingerprint of the requests
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, slowest, s5, s4, fp))


def test_two_gloo_ranks_reduce_to_the_slowest_and_own_distinct_requests():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, t0, a5, a4, f0), (r1, t1, b5, b4, f1) = got
    assert (r0, r1) == (0, 1)
    assert t0 == t1 == 2.5                       # both ranks see the slowest rank's time
    assert a5 != b5 and a4 != b4 and f0 != f1    # independent requests per rank


def test_job_value_counts_every_rank_over_the_slowest_time():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_value(1, 2e12, 1.0) == 2000.0
    assert bench.job_value(4, 2e12, 2.0) == 4000.0
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25


def test_reference_arm_on_rank_one_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
