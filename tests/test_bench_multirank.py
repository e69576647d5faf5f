"""bench.py's multi-GPU path on the CPU: two gloo ranks stand in for two GPUs.

Each rank runs an independent replica (the channels of a scan are independent, so the work shards
with no collective on the data path); the only communication is the timing reduction after the
timed region.  These tests check that reduction (slowest rank's time, launches summed), the
whole-job rate, and that only rank 0 runs the reference arm.
"""
import os
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import bench
    import synth

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        total, scan, launches = bench.aggregate_ranks(dist, torch.device("cpu"), 10.0 + rank, 1.0 + 2 * rank,
                                                      3 + rank)
        cfg = synth.CONFIGS["tiny"]

        class Args:
            steps, warmup, gpus, workload = 1, 0, world, "tiny"

        ref = bench.run_reference(Args, cfg, rank)
        out.put((rank, total, scan, launches, ref is None))
    except Exception as e:  # report instead of leaving the parent waiting
        out.put((rank, repr(e), None, None, None))
        raise
    finally:
        dist.destroy_process_group()


def test_two_rank_reduction_and_reference_arm():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, total, scan, launches, ref_none in res:
        assert not isinstance(total, str), total
        assert total == 11.0 and scan == 3.0     # slowest rank's times on every rank
        assert launches == 3 + 4                 # launches of both ranks
        assert ref_none == (rank != 0)           # the reference arm runs on rank 0 only


def test_whole_job_rate_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.whole_job_rate(1000, 10, 1, 1.0) == pytest.approx(1e7)
    assert bench.whole_job_rate(1000, 10, 4, 1.0) == pytest.approx(4e7)
