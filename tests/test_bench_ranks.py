"""The bench's multi-rank host logic on two gloo ranks (no GPU): the job's step
time is the slowest rank's, the whole-job rate counts every rank's sequences,
and the reference arm runs on rank 0 only."""
import argparse
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, loc = bench.dist_env()
    ms = 10.0 + 5.0 * rank                     # rank 1 is the slower one
    slowest = bench.slowest_rank(ms, w, device="cpu")
    rate = bench.whole_job_rate(w, 4, 8, slowest / 2)
    skipped = None
    if rank != 0:                              # the reference arm does no work off rank 0
        args = argparse.Namespace(workload="llama3_8b_tree60", steps=1, warmup=0)
        skipped = bench.run_reference(args) is None
    dist.barrier()
    dist.destroy_process_group()
    q.put((r, w, loc, slowest, rate, skipped))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_ranks_take_the_slowest_time_and_count_every_rank():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    for rank, (r, w, loc, slowest, rate, skipped) in enumerate(res):
        assert (r, w, loc) == (rank, 2, rank)
        assert slowest == 15.0                  # both ranks see the slower rank's time
        assert abs(rate - 2 * 4 * 8 / 7.5e-3) < 1e-6
    assert res[1][5] is True


def test_one_rank_keeps_its_own_time():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank(12.5, 1) == 12.5
    assert bench.whole_job_rate(1, 1, 60, 0.05) == 60 / 5e-5
