"""Host logic of a multi-rank benchmark run, on CPU with the gloo backend and two ranks: the job's time
is the slowest rank's, the throughput counts every rank's batches, each rank scores its own batch of
the same shape with the same model, and only rank 0 runs the oracle arm."""
import os
import socket
import subprocess
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(10.0 + 5.0 * rank)
        wl = bench.workload_for_rank("tiny", rank)
        q.put((rank, t, wl.n_req, wl.n_cand, int(wl.bag_ids.sum()), wl.seed))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_score_distinct_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, t0, R0, B0, s0, seed0), (r1, t1, R1, B1, s1, seed1) = res
    assert t0 == t1 == 15.0
    assert (R0, B0) == (R1, B1)
    assert seed0 != seed1 and s0 != s1


def test_single_process_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25


def test_job_throughput_counts_every_rank():
    import bench
    # 4 ranks x 4096 candidates x 10 steps in 20 ms (slowest rank) -> 8.192e6 candidates/s
    assert np.isclose(bench.job_throughput(4, 4096, 10, 20.0), 4 * 4096 * 10 / 0.020)


def test_rank_zero_scores_the_configurations_own_batch():
    import bench
    import synth
    a, b = bench.workload_for_rank("tiny", 0), synth.make_workload("tiny")
    assert np.array_equal(a.bag_ids, b.bag_ids) and np.array_equal(a.seq_ids, b.seq_ids)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
