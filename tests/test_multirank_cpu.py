"""The bench's multi-rank host logic on the CPU: two gloo ranks on 127.0.0.1.

With more GPUs each rank runs its own batch (independent heads, no collective
on the data path); the only cross-rank steps are the barriers around the
timed region and the max over ranks of the measured time, which sets the
whole job's rate.  Those, the per-rank input shards and the reference arm's
rank-0-only run are what these tests cover; no GPU is touched.
"""

import multiprocessing as mp
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench.dist_env()
        elapsed = [3.0, 5.0, 4.0, 1.0][rank]          # each rank's own timed region
        dist.barrier()
        slowest = bench.max_over_ranks(torch, elapsed, torch.device("cpu"), w)
        out.put((r, w, lr, slowest, bench.rank_seed(r)))
    finally:
        dist.destroy_process_group()


def _run_ranks(world):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return res


def test_two_ranks_agree_on_the_slowest_time_and_draw_distinct_shards():
    res = _run_ranks(2)
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] == 2 and r[2] == r[0] for r in res)
    assert all(r[3] == 5.0 for r in res)              # every rank sees the max
    assert res[0][4] != res[1][4]                     # each rank its own batch


def test_whole_job_rate_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_tflops(1, 2.0e12, 1.0)
    assert one == 2000.0
    assert bench.whole_job_tflops(2, 2.0e12, 1.0) == 2 * one
    # alone, max over ranks is the value itself and needs no process group
    assert bench.max_over_ranks(None, 7.5, None, 1) == 7.5


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True,
                       text=True, timeout=120, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""                     # no line, no oracle work
