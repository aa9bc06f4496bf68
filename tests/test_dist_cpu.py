"""N > 1 host logic of the benchmark, on CPU with the gloo backend.

The hot path has no exchange step: each rank runs an independent replica and
the job's throughput is (units summed over ranks) / (max elapsed over ranks).
These tests run two gloo ranks on 127.0.0.1 and check that aggregation, and
that the reference arm does its work on rank 0 only.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist_mod = bench.init_group(world, "gloo")
    elapsed, units = bench.aggregate(1.0 + rank, 10.0 * (rank + 1), dist_mod)
    q.put((rank, elapsed, units))
    dist_mod.barrier()
    dist_mod.destroy_process_group()


def _ref_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    if rank != 0:
        q.put((rank, bench.run_reference(bench_args()) is None))
    else:
        q.put((rank, True))


def bench_args():
    import argparse
    return argparse.Namespace(steps=1, warmup=0, reference_rows=8, reference_cols=8)


@pytest.mark.parametrize("world", [2])
def test_aggregate_max_time_sum_units(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, elapsed, units in res:
        assert elapsed == pytest.approx(float(world))
        assert units == pytest.approx(10.0 * world * (world + 1) / 2)


def test_reference_arm_only_rank0_works():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    p = ctx.Process(target=_ref_worker, args=(1, 2, port, q))
    p.start()
    rank, ok = q.get(timeout=120)
    p.join(timeout=60)
    assert rank == 1 and ok and p.exitcode == 0
