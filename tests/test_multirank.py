"""The N > 1 path of bench.py (replicas only: no collective on the data path)
checked with world_size-2 gloo process groups on CPU: the barrier, the
max-over-ranks timing, the whole-job throughput, and the reference arm's
rule that ranks other than 0 exit without work."""
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
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import argparse

    import torch.distributed as dist

    import bench
    args = argparse.Namespace(impl="ours", gpus=world)
    w, r, local = bench.dist_setup(args)
    assert (w, r, local) == (world, rank, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    slowest = bench.max_over_ranks(w, 10.0 + rank)  # rank 1 is the slowest
    value = bench.job_value(w, 85, 100, slowest)
    # the reference arm: rank != 0 returns at once without building anything
    ref = bench.run_reference(argparse.Namespace(weights="bf16", shape="mixtral", zipf=None,
                                                 seed=0, warmup=1, steps=1, gpus=world), w, r) \
        if r != 0 else None
    bench.barrier(w)
    dist.destroy_process_group()
    q.put((rank, slowest, value, ref))


def test_two_rank_replicas_on_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=300) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value, ref in out:
        assert slowest == 11.0
        # 2 replicas x 85 tokens x 100 steps in 11 ms of the slowest rank
        assert value == pytest.approx(2 * 85 * 100 / 0.011)
        assert ref is None


def test_job_value_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_value(1, 85, 600, 900.0) == pytest.approx(85 * 600 / 0.9)
