"""The benchmark's multi-rank host logic on CPU (gloo, world size 2): every rank runs an
independent replica, the job time is the slowest rank's, the job rate counts all ranks'
work; the reference arm runs on rank 0 only."""
import os
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = [10.0 + rank, 3.0 - rank]  # per-rank step time and e2e time (ms)
    got = bench.reduce_max_over_ranks(local)
    out.put((rank, got, bench.job_throughput(100.0, world, got[0])))
    dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, got, rate in res:
        assert got == [11.0, 3.0]                 # max over ranks, element-wise
        assert abs(rate - 2 * 100.0 / 11e-3) < 1e-6  # both ranks' work over the slowest time


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.reduce_max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert bench.job_throughput(10.0, 1, 5.0) == 2000.0


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
